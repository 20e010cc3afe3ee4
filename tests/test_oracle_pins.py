"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: closed forms,
the exact output law derived in "Speculative Decoding in Large Language
Models", section 2 "Proof of Distributional Invariance", statistical laws
that follow from it, plain argmax decoding, special cases, and the worked
numbers printed on that page.  A plausible slip in the oracle (accept test the
wrong way round, residual q - p instead of p - q, the correction drawn with the
rejected position's own uniform, no bonus token, the scan not stopping at the
first rejection, a transposed GEMM operand) fails at least one of them.
"""
from __future__ import annotations

import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import speedup

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# softmax / argmax
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_softmax_closed_form(T):
    w = np.array([1.0, 2.0, 3.0, 4.0])
    z = (T * np.log(w))[None, :]
    p = oracle.softmax_rows(z, T)[0]
    np.testing.assert_allclose(p, w / w.sum(), rtol=0, atol=1e-15)
    # shift invariance and an impossible token (-inf logit -> p = 0)
    z2 = np.concatenate([z + 300.0, [[-np.inf]]], axis=1)
    p2 = oracle.softmax_rows(z2, T)[0]
    # z / T near 430 carries ~1e-13 of rounding into the exponent
    np.testing.assert_allclose(p2[:4], w / w.sum(), rtol=0, atol=1e-12)
    assert p2[4] == 0.0


def test_softmax_bf16_decodes_exactly():
    z = torch.tensor([[0.0, 1.0, 2.0, -3.5]], dtype=torch.bfloat16)
    p = oracle.softmax_rows(z, 1.0)[0]
    e = np.exp(np.array([0.0, 1.0, 2.0, -3.5]))
    np.testing.assert_allclose(p, e / e.sum(), rtol=1e-15)


def test_argmax_lowest_index_on_ties():
    z = np.array([[1.0, 5.0, 2.0, 5.0, 5.0], [7.0, 7.0, 7.0, 7.0, 7.0]], dtype=np.float32)
    assert list(oracle.argmax_rows(z)) == [1, 0]


# --------------------------------------------------------------------------
# exact output law by enumeration (dyadic probabilities)
# --------------------------------------------------------------------------
def _dyadic_case(rng, V, K):
    """Rows of p and q (numerators over 16) for which every breakpoint of the
    algorithm in u (p/q ratios, residual CDF values) is a multiple of 1/16, so
    that evaluating the oracle at the centres of a 16-cell grid per uniform
    integrates it exactly."""
    def rand_row(allowed=None):
        while True:
            if allowed is None:
                cuts = np.sort(rng.integers(0, 17, size=V - 1))
                row = np.diff(np.concatenate([[0], cuts, [16]]))
            else:
                row = rng.choice(allowed, size=V)
                if row.sum() != 16:
                    continue
            return row.astype(int)

    while True:
        P = [rand_row() for _ in range(K + 1)]
        Q = [rand_row(allowed=[0, 1, 2, 4, 8]) for _ in range(K)]
        ok = True
        for j in range(K):
            Rnum = sum(max(0, P[j][v] - Q[j][v]) for v in range(V))
            if Rnum not in (0, 1, 2, 4, 8, 16):
                ok = False
            if Rnum == 0:
                ok = False  # p == q row: no rejection possible, fine but uninformative
        if ok:
            return P, Q


def _proof_law(P, Q, K, V):
    """Joint law of (AL, emitted tokens) from the invariance proof:
    accept x with probability min(p, q) mass, emit the residual p - min(p, q)
    at the first rejection, and p_K as the bonus."""
    p = [[Fraction(n, 16) for n in row] for row in P]
    q = [[Fraction(n, 16) for n in row] for row in Q]
    law = {}
    for L in range(1, K + 2):  # AL = L: accepted tokens a_0..a_{L-2}, then one more
        for acc in itertools.product(range(V), repeat=L - 1):
            w = Fraction(1)
            for j, a in enumerate(acc):
                w *= min(p[j][a], q[j][a])
            if w == 0:
                continue
            j = L - 1
            for v in range(V):
                if j < K:
                    last = p[j][v] - min(p[j][v], q[j][v])
                else:
                    last = p[K][v]
                if last:
                    law[(L,) + acc + (v,)] = law.get((L,) + acc + (v,), 0) + w * last
    return law


@pytest.mark.parametrize("K,seed", [(1, 0), (1, 1), (2, 2), (2, 3), (2, 4)])
@pytest.mark.parametrize("T", [1.0, 0.5])
def test_exact_output_law_by_enumeration(K, seed, T):
    V = 4
    rng = np.random.default_rng(seed)
    P, Q = _dyadic_case(rng, V, K)
    with np.errstate(divide="ignore"):
        z = np.stack([T * np.log(np.array(row, dtype=np.float64) / 16.0) for row in P])
    q = np.stack([np.array(row, dtype=np.float32) / 16.0 for row in Q])
    grid = (np.arange(16) + 0.5) / 16.0
    reqs = []
    for x in itertools.product(range(V), repeat=K):
        w = Fraction(1)
        for j, a in enumerate(x):
            w *= Fraction(Q[j][a], 16)
        if w == 0:
            continue
        for us in itertools.product(grid, repeat=K + 1):
            reqs.append((x, us, w))
    n = len(reqs)
    logits = np.ascontiguousarray(np.broadcast_to(z, (n, K + 1, V)).reshape(n * (K + 1), V))
    qq = np.ascontiguousarray(np.broadcast_to(q, (n, K, V)).reshape(n * K, V)).astype(np.float32)
    draft = np.array([r[0] for r in reqs], dtype=np.int32).reshape(-1)
    uni = np.array([r[1] for r in reqs], dtype=np.float32).reshape(-1)
    res = oracle.verify_fixed(logits, qq, draft, uni, n, K, T)
    out = res["out_tokens"].reshape(n, K + 1)
    al = res["accept_len"]
    assert res["near_tie_accept"].sum() == 0 and res["near_tie_sample"].sum() == 0
    cell = Fraction(1, 16 ** (K + 1))
    got = {}
    for i, (_, _, w) in enumerate(reqs):
        key = (int(al[i]),) + tuple(int(t) for t in out[i, : al[i]])
        got[key] = got.get(key, 0) + w * cell
    want = _proof_law(P, Q, K, V)
    assert got == want
    # corollary printed on the page: the first emitted token follows p exactly
    first = {}
    for key, pr in got.items():
        first[key[1]] = first.get(key[1], 0) + pr
    assert first == {v: Fraction(P[0][v], 16) for v in range(V) if P[0][v]}


# --------------------------------------------------------------------------
# statistical laws at 10^6 trials (V <= 16)
# --------------------------------------------------------------------------
def _trial_batch(z, q, n, rng):
    K = q.shape[0]
    V = z.shape[1]
    draft = np.stack([rng.choice(V, size=n, p=q[j].astype(np.float64) / q[j].astype(np.float64).sum())
                      for j in range(K)], axis=1).astype(np.int32)
    uni = rng.random((n, K + 1)).astype(np.float32)
    uni = np.clip(uni, np.float32(2 ** -24), np.float32(1 - 2 ** -24))
    logits = np.ascontiguousarray(np.broadcast_to(z, (n, K + 1, V)).reshape(-1, V)).astype(np.float32)
    qq = np.ascontiguousarray(np.broadcast_to(q, (n, K, V)).reshape(-1, V)).astype(np.float32)
    return logits, qq, draft.reshape(-1), uni.reshape(-1)


def _q_variants(z, rng):
    V = z.shape[1]
    K = z.shape[0] - 1
    def sm(x):
        e = np.exp(x - x.max(axis=-1, keepdims=True))
        return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)
    near = sm(z[:K] + rng.normal(0, 1.0, size=(K, V)))
    onehot = np.zeros((K, V), np.float32)
    onehot[np.arange(K), rng.integers(0, V, size=K)] = 1.0
    zeros = sm(z[:K] + rng.normal(0, 1.0, size=(K, V)))
    zeros[:, ::2] = 0.0
    zeros /= zeros.sum(axis=1, keepdims=True)
    far = sm(-2.0 * z[:K])
    return {"near": near, "onehot": onehot.astype(np.float32), "zeros": zeros.astype(np.float32), "far": far}


def _chisq_pvalue(counts, probs):
    from scipy import stats
    n = counts.sum()
    exp = probs * n
    keep = exp >= 5
    c = np.concatenate([counts[keep], [counts[~keep].sum()]])
    e = np.concatenate([exp[keep], [exp[~keep].sum()]])
    if e[-1] == 0:
        c, e = c[:-1], e[:-1]
    e = e * c.sum() / e.sum()
    return stats.chisquare(c, e).pvalue


@pytest.mark.parametrize("variant", ["near", "onehot", "zeros", "far"])
def test_emitted_token_law_is_p_chisquare(variant):
    """10^6 trials, V = 16, K = 2: the first emitted token follows p_0, and
    the token at position j given positions < j accepted follows p_j."""
    rng = np.random.default_rng(123)
    V, K, T, n = 16, 2, 1.0, 1_000_000
    z = rng.normal(0, 1.0, size=(K + 1, V))
    q = _q_variants(z, rng)[variant]
    logits, qq, draft, uni = _trial_batch(z, q, n, rng)
    res = oracle.verify_fixed(logits, qq, draft, uni, n, K, T)
    out = res["out_tokens"].reshape(n, K + 1)
    al = res["accept_len"]
    p = oracle.softmax_rows(z.astype(np.float32), T)
    for j in range(K + 1):
        sel = al > j
        counts = np.bincount(out[sel, j], minlength=V).astype(np.float64)
        assert _chisq_pvalue(counts, p[j]) > 1e-3, (variant, j)


def test_acceptance_rate_and_mean_al():
    """Per-position acceptance frequency -> beta_j = sum min(p_j, q_j); mean AL
    -> sum_k prod_{j<k} beta_j; both inside a 5 sigma binomial band."""
    rng = np.random.default_rng(7)
    V, K, T, n = 16, 3, 0.8, 400_000
    z = rng.normal(0, 1.5, size=(K + 1, V))
    q = _q_variants(z, rng)["near"]
    logits, qq, draft, uni = _trial_batch(z, q, n, rng)
    res = oracle.verify_fixed(logits, qq, draft, uni, n, K, T)
    al = res["accept_len"]
    p = oracle.softmax_rows(z.astype(np.float32), T)
    betas = [speedup.acceptance_beta(p[j], q[j]) for j in range(K)]
    for j in range(K):
        reached = al > j           # position j was tested
        acc = al > j + 1           # and accepted
        k = reached.sum()
        freq = acc.sum() / k
        sd = math.sqrt(betas[j] * (1 - betas[j]) / k)
        assert abs(freq - betas[j]) < 5 * sd, (j, freq, betas[j])
    mean_al = al.mean()
    want = speedup.mean_accept_length(betas)
    sd = al.std() / math.sqrt(n)
    assert abs(mean_al - want) < 5 * sd


@pytest.mark.parametrize("alpha", [0.3, 0.875])
def test_mean_al_matches_page_closed_form(alpha):
    """Equal acceptance rate alpha at every position: mean AL must approach
    E[N] = (1 - alpha^(gamma+1)) / (1 - alpha) with gamma = K = 5.  Rows are
    built with p = (alpha, 1-alpha, 0...) and q = (1, 0, ...) so that
    beta = sum min(p, q) = alpha exactly."""
    rng = np.random.default_rng(11)
    V, K, n = 8, 5, 300_000
    prow = np.zeros(V)
    prow[0], prow[1] = alpha, 1 - alpha
    with np.errstate(divide="ignore"):
        z = np.tile(np.log(prow), (K + 1, 1))
    q = np.zeros((K, V), np.float32)
    q[:, 0] = 1.0
    logits, qq, draft, uni = _trial_batch(z, q, n, rng)
    res = oracle.verify_fixed(logits.astype(np.float64), qq, draft, uni, n, K, 1.0)
    al = res["accept_len"]
    want = speedup.expected_tokens(alpha, K)
    assert abs(al.mean() - want) < 5 * al.std() / math.sqrt(n)


# --------------------------------------------------------------------------
# special cases
# --------------------------------------------------------------------------
def test_q_equals_p_accepts_everything():
    rng = np.random.default_rng(5)
    B, K, V, T = 200, 4, 64, 0.9
    z = rng.normal(0, 2, size=(B * (K + 1), V)).astype(np.float32)
    p = oracle.softmax_rows(z, T).reshape(B, K + 1, V)
    q = p[:, :K].reshape(B * K, V).astype(np.float32)
    draft = np.array([rng.choice(V, p=row / row.sum()) for row in q.astype(np.float64)], np.int32)
    uni = rng.random(B * (K + 1)).astype(np.float32)
    res = oracle.verify_fixed(z, q, draft, uni, B, K, T)
    full = res["accept_len"] == K + 1
    # a rejection can only come from q's fp32 rounding above p: a counted near tie
    assert np.all(full | (res["near_tie_accept"] > 0))


def test_q_zero_at_drafted_token_accepts():
    V = 4
    z = np.log(np.array([[0.25, 0.25, 0.25, 0.25]] * 2))
    q = np.array([[0.0, 0.5, 0.5, 0.0]], np.float32)
    res = oracle.verify_fixed(z, q, np.array([0], np.int32), np.array([0.99, 0.5], np.float32), 1, 1, 1.0)
    assert res["accept_len"][0] == 2 and res["out_tokens"][0] == 0


def test_residual_excludes_rejected_token_and_uses_final_uniform():
    """p = (1/2, 1/4, 1/4), q = (0, 0, 1): drafting token 2 accepts with
    probability 1/4; on rejection the residual is (1/2, 1/4, 0) / (3/4), and
    the correction is drawn with u_K, not with the rejected position's u."""
    z = np.log(np.array([[0.5, 0.25, 0.25], [0.5, 0.25, 0.25]]))
    q = np.array([[0.0, 0.0, 1.0]], np.float32)
    for u0 in [0.3, 0.9]:
        for uK, tok in [(0.1, 0), (0.6, 0), (0.7, 1), (0.95, 1)]:
            res = oracle.verify_fixed(z, q, np.array([2], np.int32), np.array([u0, uK], np.float32), 1, 1, 1.0)
            assert res["accept_len"][0] == 1
            assert res["out_tokens"][0] == tok, (u0, uK)
            assert abs(res["residual_mass"][0] - 0.75) < 1e-15
    res = oracle.verify_fixed(z, q, np.array([2], np.int32), np.array([0.2, 0.9], np.float32), 1, 1, 1.0)
    # accepted (0.2 <= 1/4), bonus from p_1 = (1/2, 1/4, 1/4): 0.9 lies in the third bin
    assert res["accept_len"][0] == 2 and res["out_tokens"][0] == 2 and res["out_tokens"][1] == 2


def test_zero_residual_falls_back_to_p():
    """q above p everywhere (q rows not normalised): after a rejection the
    residual is empty; the oracle samples from p and flags it."""
    z = np.log(np.array([[0.5, 0.5], [0.5, 0.5]]))
    q = np.array([[0.6, 0.6]], np.float32)
    res = oracle.verify_fixed(z, q, np.array([0], np.int32), np.array([0.99, 0.75], np.float32), 1, 1, 1.0)
    assert res["accept_len"][0] == 1 and res["zero_residual"][0] == 1
    assert res["out_tokens"][0] == 1


def test_invalid_draft_id_invalidates_request():
    z = np.zeros((4, 5), np.float32)
    q = np.full((2, 5), 0.2, np.float32)
    res = oracle.verify_fixed(z, q, np.array([1, 7], np.int32), np.full(4, 0.5, np.float32), 2, 1, 1.0)
    assert res["invalid"] == 1
    assert res["accept_len"][1] == 0 and list(res["out_tokens"][2:]) == [-1, -1]
    assert res["accept_len"][0] >= 1


def test_greedy_reproduces_argmax_decoding():
    """Greedy verification emits exactly the plain argmax decode of rows 0..AL-1
    ("Co-Designing AI Models...": same output as standard decoding)."""
    rng = np.random.default_rng(3)
    B, K, V = 300, 5, 50
    z = np.round(rng.normal(0, 1, size=(B * (K + 1), V)) * 4) / 4  # many ties
    z = z.astype(np.float32)
    am = z.reshape(B, K + 1, V).argmax(axis=2)  # numpy: first index on ties
    draft = am[:, :K].copy()
    flip = rng.random((B, K)) < 0.3
    draft[flip] = rng.integers(0, V, size=flip.sum())
    res = oracle.verify_fixed(z, None, draft.reshape(-1).astype(np.int32), None, B, K, 0.0, greedy=True)
    out = res["out_tokens"].reshape(B, K + 1)
    al = res["accept_len"]
    for b in range(B):
        L = al[b]
        assert 1 <= L <= K + 1
        assert list(out[b, :L]) == list(am[b, :L])
        assert all(t == -1 for t in out[b, L:])
        mism = [j for j in range(K) if draft[b, j] != am[b, j]]
        assert L == (mism[0] + 1 if mism else K + 1)


def test_ragged_k_zero_goes_straight_to_bonus():
    V = 3
    ro = np.array([0, 1, 3], np.int32)  # K_0 = 0, K_1 = 1
    z = np.log(np.array([[0.2, 0.3, 0.5], [0.5, 0.25, 0.25], [0.1, 0.1, 0.8]]))
    q = np.array([[1.0, 0.0, 0.0]], np.float32)
    uni = np.array([0.45, 0.1, 0.95], np.float32)
    res = oracle.verify(z, q, np.array([0], np.int32), uni, ro, 1.0)
    assert res["accept_len"][0] == 1 and res["out_tokens"][0] == 1   # 0.45 -> cdf .2,.5
    assert res["accept_len"][1] == 2 and list(res["out_tokens"][1:]) == [0, 2]


def test_accept_length_bounds_random():
    rng = np.random.default_rng(9)
    B, K, V = 500, 6, 32
    z = rng.normal(0, 2, size=(B * (K + 1), V)).astype(np.float32)
    qz = z.reshape(B, K + 1, V)[:, :K].reshape(B * K, V) + rng.normal(0, 1, size=(B * K, V))
    q = (np.exp(qz) / np.exp(qz).sum(1, keepdims=True)).astype(np.float32)
    draft = np.array([rng.choice(V, p=r / r.sum()) for r in q.astype(np.float64)], np.int32)
    uni = rng.random(B * (K + 1)).astype(np.float32)
    res = oracle.verify_fixed(z, q, draft, uni, B, K, 1.0)
    al = res["accept_len"]
    assert al.min() >= 1 and al.max() <= K + 1
    out = res["out_tokens"].reshape(B, K + 1)
    d = draft.reshape(B, K)
    for b in range(B):
        assert list(out[b, : al[b] - 1]) == list(d[b, : al[b] - 1])


# --------------------------------------------------------------------------
# LM-head GEMM orientation
# --------------------------------------------------------------------------
def test_lmhead_logits_direct_sum():
    g = torch.Generator().manual_seed(0)
    M, d, V = 3, 5, 7
    h = torch.randn(M, d, generator=g).to(torch.bfloat16)
    wt = torch.randn(V, d, generator=g).to(torch.bfloat16)
    z = oracle.lmhead_logits(h, wt, v_chunk=3)
    hf = h.float().tolist()
    wf = wt.float().tolist()
    for i in range(M):
        for v in range(V):
            s = 0.0
            for k in range(d):
                s += hf[i][k] * wf[v][k]
            assert abs(z[i, v] - s) < 1e-12


# --------------------------------------------------------------------------
# speedup model: the worked numbers printed on the page
# --------------------------------------------------------------------------
def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "speedup_worked_examples.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, alo, ahi, g, c, en, cost, s = line.split()
                rows.append((name, float(alo), float(ahi), int(g), float(c), float(en), float(cost), float(s)))
    return rows


def _trunc2(x):
    return math.floor(x * 100 + 1e-9) / 100


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_speedup_worked_examples(row):
    name, alo, ahi, g, c, en, cost, s = row
    assert abs((1 + g * c) - cost) < 1e-12
    if alo == ahi:
        # E[N] from the closed form, carried to two decimals as the page does
        assert _trunc2(speedup.expected_tokens(alo, g)) == en
        assert _trunc2(en / cost) == s
        assert abs(speedup.cycle_speedup(alo, g, c) - speedup.expected_tokens(alo, g) / cost) < 1e-15
    else:
        # E[N] ~ 4.4 must be reachable inside the printed alpha range
        assert speedup.expected_tokens(alo, g) < en < speedup.expected_tokens(ahi, g)
        assert abs(en / cost - s) < 1e-12


def test_expected_tokens_limits():
    # E[N] in [1, gamma + 1]: AL lies between 1 and 1 + D ("Co-Designing AI Models Using Speculative
    # Decoding for Faster LLM Inference", "What is speculative decoding?")
    for g in range(0, 9):
        assert speedup.expected_tokens(0.0, g) == 1.0
        assert speedup.expected_tokens(1.0, g) == g + 1
        assert abs(speedup.expected_tokens(0.999999, g) - (g + 1)) < 1e-4
    # that section's speedup formula gives AL when verifying B(1+D) tokens costs
    # the same as verifying B and drafting is free
    assert speedup.measured_speedup(2.0, 2.0, 0.0, 3.7) == pytest.approx(3.7)


# --------------------------------------------------------------------------
# batch layout, input rules and the draw's edges
# --------------------------------------------------------------------------
def _ragged_case(seed, ks, V, dtype=np.float32):
    rng = np.random.default_rng(seed)
    ro = np.concatenate([[0], np.cumsum(np.asarray(ks) + 1)]).astype(np.int32)
    R, nq = int(ro[-1]), int(ro[-1]) - len(ks)
    z = rng.normal(0, 2.0, size=(R, V)).astype(dtype)
    zq = rng.normal(0, 2.0, size=(nq, V))
    q = (np.exp(zq) / np.exp(zq).sum(1, keepdims=True)).astype(np.float32)
    x = np.array([rng.choice(V, p=q[i].astype(np.float64) / q[i].astype(np.float64).sum()) for i in range(nq)],
                 dtype=np.int32)
    u = rng.uniform(0.001, 0.999, size=R).astype(np.float32)
    return z, q, x, u, ro


@pytest.mark.parametrize("greedy", [False, True])
def test_ragged_batch_equals_its_requests_one_by_one(greedy):
    """Request b of a CSR batch owns logits rows, uniforms and output slots
    ro[b] .. ro[b+1]-1 and q rows / draft ids ro[b]-b .. ro[b+1]-b-2: the batch
    gives what each request gives alone."""
    ks = [3, 0, 5, 1, 0, 2, 4]
    z, q, x, u, ro = _ragged_case(5, ks, 40)
    res = oracle.verify(z, q, x, u, ro, 0.9, greedy=greedy)
    for b, k in enumerate(ks):
        r0, d0 = int(ro[b]), int(ro[b]) - b
        one = oracle.verify_fixed(z[r0:r0 + k + 1], q[d0:d0 + k], x[d0:d0 + k], u[r0:r0 + k + 1], 1, k, 0.9,
                                  greedy=greedy)
        assert res["accept_len"][b] == one["accept_len"][0], b
        assert np.array_equal(res["out_tokens"][r0:r0 + k + 1], one["out_tokens"]), b


def test_malformed_offsets_are_refused():
    z = np.zeros((5, 8), np.float32)
    q = np.full((3, 8), 0.125, np.float32)
    x = np.zeros(3, np.int32)
    u = np.full(5, 0.5, np.float32)
    for ro in ([0, 3, 3, 5], [0, 4, 3, 5], [1, 3, 5]):  # an empty request, decreasing, not from 0
        with pytest.raises(ValueError):
            oracle.verify(z, q, x, u, np.array(ro, np.int32), 1.0)


def test_drafted_id_equal_to_vocab_size_is_invalid():
    V = 6
    z = np.zeros((3, V), np.float32)
    q = np.full((2, V), 1.0 / V, np.float32)
    u = np.full(3, 0.5, np.float32)
    res = oracle.verify_fixed(z, q, np.array([0, V], np.int32), u, 1, 2, 1.0)
    assert res["invalid"] == 1 and res["accept_len"][0] == 0 and list(res["out_tokens"]) == [-1, -1, -1]
    res = oracle.verify_fixed(z, q, np.array([0, V - 1], np.int32), u, 1, 2, 1.0)
    assert res["invalid"] == 0 and res["accept_len"][0] >= 1


def test_draw_with_no_boundary_above_u_takes_the_last_positive_token():
    """The reading for a draw that rounding leaves without a boundary above
    u R: the largest token with r > 0.  A final uniform of exactly 1 makes
    that happen (u R = R = C(V-1)); the tokens after the last positive one
    have z = -inf, so p and r are 0 there."""
    z = np.array([[0.3, -1.0, 2.0, 0.0, 1.5, -0.5, 0.7, -np.inf, -np.inf, -np.inf]])
    res = oracle.verify_fixed(z, np.zeros((0, 10), np.float32), np.zeros(0, np.int32),
                              np.array([1.0], np.float32), 1, 0, 1.0)
    assert res["out_tokens"][0] == 6 and res["near_tie_sample"][0] == 1


def test_accept_near_tie_is_measured_on_p_over_q():
    """p(x) = 1/4 (four equal logits), q(x) = 1/2: the accept threshold p/q is
    1/2.  A uniform 6e-8 above it is a near tie; one at 0.6 is not."""
    z = np.zeros((2, 4))
    q = np.array([[0.5, 0.5 / 3, 0.5 / 3, 0.5 / 3]], np.float32)
    u_near = np.nextafter(np.float32(0.5), np.float32(1.0))
    for u0, tie in ((u_near, 1), (np.float32(0.6), 0)):
        res = oracle.verify_fixed(z, q, np.array([0], np.int32), np.array([u0, 0.3], np.float32), 1, 1, 1.0)
        assert res["near_tie_accept"][0] == tie, u0
        assert res["accept_len"][0] == 1  # u > 1/2: rejected either way


def test_zero_residual_draws_from_p_not_uniformly():
    """q = 1 everywhere leaves an empty residual after every rejection; the
    token is the inverse-CDF draw from the (non-uniform) p with the final
    uniform, computed here with numpy from the page's softmax."""
    rng = np.random.default_rng(11)
    B, V = 40, 64
    z = rng.normal(0, 2.0, size=(2 * B, V))
    q = np.ones((B, V), np.float32)
    x = rng.integers(0, V, size=B).astype(np.int32)
    u = rng.uniform(0.01, 0.99, size=2 * B).astype(np.float32)
    res = oracle.verify_fixed(z, q, x, u, B, 1, 1.0)
    checked = 0
    for b in range(B):
        assert res["accept_len"][b] == 1 and res["zero_residual"][b] == 1
        p = np.exp(z[2 * b] - z[2 * b].max())
        c = np.cumsum(p) / p.sum()
        uf = float(u[2 * b + 1])
        if np.min(np.abs(c - uf)) < 1e-9:
            continue
        assert res["out_tokens"][2 * b] == int(np.searchsorted(c, uf, side="right")), b
        checked += 1
    assert checked >= B - 2


def test_results_do_not_change_when_every_logit_is_shifted():
    """softmax(z + c) = softmax(z): fp64 logits shifted by 1000 (exp(1000)
    overflows fp64 without the max subtraction) give the same results."""
    z, q, x, u, ro = _ragged_case(9, [2, 3, 0, 1], 30, dtype=np.float64)
    a = oracle.verify(z, q, x, u, ro, 0.8)
    b = oracle.verify(z + 1000.0, q, x, u, ro, 0.8)
    assert np.array_equal(a["accept_len"], b["accept_len"]) and np.array_equal(a["out_tokens"], b["out_tokens"])
    assert np.allclose(a["p_draft"], b["p_draft"], rtol=1e-9, atol=0, equal_nan=True)
    assert np.allclose(oracle.softmax_rows(z + 1000.0, 0.8), oracle.softmax_rows(z, 0.8), rtol=1e-9, atol=1e-300)


@pytest.mark.parametrize("alpha,gamma,c", [(0.6, 4, 0.05), (0.8, 7, 0.1), (0.3, 2, 0.02)])
def test_measured_speedup_reduces_to_the_cycle_model(alpha, gamma, c):
    """With the cycle model's costs (one target call of unit time at either
    batch size, as the memory-bound verification makes it, gamma draft steps
    of c each) and AL = E[N], the measured-times formula of "Co-Designing AI
    Models..." equals the closed form of "Speculative Decoding in Large
    Language Models", section 2."""
    got = speedup.measured_speedup(1.0, 1.0, gamma * c, speedup.expected_tokens(alpha, gamma))
    assert abs(got - speedup.cycle_speedup(alpha, gamma, c)) < 1e-12
