"""Pins of the draft-side oracle (oracle/draft.py and the C functions under it)
against facts outside its own code: published Philox4x32-10 known-answer
vectors, exact rational enumeration of the inverse-CDF draw, a chi-square test
of the draws against q, and plain argmax for greedy drafting.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import draft as D
from speculative_decoding_verification_11_gb300 import workloads as W

from test_oracle_pins import _chisq_pvalue

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        w = [int(t, 16) for t in line.split()]
        rows.append((w[0:4], w[4:6], w[6:10]))
    return rows


def test_philox_known_answer_vectors():
    rows = _kat()
    assert len(rows) == 3
    for ctr, key, want in rows:
        assert [int(v) for v in D.philox4x32_10(ctr, key)] == want


def test_uniform_mapping_and_the_input_generator_agree():
    """The oracle's uniform of (seed, index, stream) equals the one the seeded
    input generator (numpy, written separately) makes for the same counter."""
    seed = 0x1234_5678_9ABC
    got = np.array([D.philox_uniform(seed, 1000 + i, stream=1) for i in range(64)])
    ref = W.philox_uniforms(seed, 64, stream=1, offset=1000).astype(np.float64)
    assert np.array_equal(got, ref)
    assert np.all(got > 0) and np.all(got < 1)
    assert np.array_equal(got.astype(np.float32).astype(np.float64), got)  # exact in fp32


def test_draft_uniforms_follow_their_counters():
    """Draw r of a call with counter offset o uses Philox counter (o + r,
    stream 1): the uniforms draft_sample reports equal the input generator's
    (numpy, written separately) for that stream and offset, and another offset
    gives other uniforms."""
    g = torch.Generator().manual_seed(17)
    M, d, V = 6, 64, 300
    h = torch.randn(M, d, generator=g).to(torch.bfloat16)
    w = (torch.randn(V, d, generator=g) * 0.1).to(torch.bfloat16)
    seed = 0xABCDEF012345
    for offset in (0, 777, 2**33 + 5):
        got = D.draft_sample(h, w, 1.0, seed, offset)["u"]
        ref = W.philox_uniforms(seed, M, stream=1, offset=offset).astype(np.float64)
        assert np.array_equal(got, ref), offset
    assert not np.array_equal(D.draft_sample(h, w, 1.0, seed, 0)["u"], D.draft_sample(h, w, 1.0, seed, 1)["u"])


def test_draw_matches_exact_rational_enumeration():
    rng = np.random.default_rng(3)
    for _ in range(300):
        V = int(rng.integers(1, 7))
        w = rng.integers(0, 5, size=V)
        if w.sum() == 0:
            w[int(rng.integers(0, V))] = 1
        u = float(rng.integers(1, 2**20)) / 2**20
        # exact: the smallest v whose cumulative weight exceeds u * total
        tot = Fraction(int(w.sum()))
        cum = Fraction(0)
        want = None
        for v in range(V):
            cum += int(w[v])
            if cum > Fraction(u) * tot:
                want = v
                break
        got, _ = D.draw_inverse_cdf(w.astype(np.float64), u)
        assert got == want, (w, u)
    # u exactly on a boundary: C(v) = u R picks the next token (strictly greater)
    for w, u, want in (([1, 1], 0.5, 1), ([2, 1, 1], 0.5, 1), ([1, 1, 2, 4], 0.25, 2), ([3, 0, 1], 0.75, 2),
                       ([1, 3], 0.25, 1)):
        assert D.draw_inverse_cdf(np.array(w, dtype=np.float64), u)[0] == want, (w, u)


def test_draws_follow_q_chisquare():
    rng = np.random.default_rng(8)
    V, n = 16, 200_000
    q = rng.dirichlet(np.ones(V) * 0.7)
    u = W.philox_uniforms(99, n, stream=1).astype(np.float64)
    draws = np.array([D.draw_inverse_cdf(q, float(x))[0] for x in u[:n]])
    counts = np.bincount(draws, minlength=V).astype(np.float64)
    assert _chisq_pvalue(counts, q) > 1e-3


def test_draft_sample_small_case():
    g = torch.Generator().manual_seed(5)
    M, d, V = 6, 64, 40
    h = torch.randn(M, d, generator=g).to(torch.bfloat16)
    w = (torch.randn(V, d, generator=g) * 0.3).to(torch.bfloat16)
    res = D.draft_sample(h, w, 0.8, seed=77, offset=10)
    z = h.double() @ w.double().T
    q = torch.softmax(z / 0.8, dim=1).numpy()
    assert np.allclose(res["q"], q, rtol=1e-12, atol=0)
    assert np.allclose(res["q"].sum(1), 1.0, rtol=0, atol=1e-12)
    for r in range(M):
        c = np.cumsum(q[r])
        v = int(res["x"][r])
        assert (v == 0 or c[v - 1] <= res["u"][r] * c[-1] + 1e-12) and c[v] > res["u"][r] * c[-1] - 1e-12
    greedy = D.draft_sample(h, w, 0.0, seed=77)
    assert np.array_equal(greedy["x"], np.argmax(z.numpy(), axis=1))
