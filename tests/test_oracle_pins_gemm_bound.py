"""Pins of the GEMM accumulation bound, the bands it induces and the
accumulation model (oracle/gemm_bound.py), each against something other than
the code under test:

  - simulated fp32 accumulations (one rounding per 16-product step, to nearest
    and toward zero) and the model's own accumulation stay inside beta on
    mixed-sign and one-signed operands;
  - a hand-built case where every product of every step falls just below the
    alignment grid (all dropped) reaches 78% of beta, and a bound without the
    dropped-bits term, or taken over 64-product steps, is exceeded there;
  - the model gives, on hand-worked operands, the values its statement
    implies (guard bits, rounding toward zero, alignment to the accumulator);
  - the fp64 logits equal an exactly rounded direct sum (math.fsum);
  - logits perturbed anywhere inside beta move p, and the partial masses of
    max(0, p - q), inside the derived bands, and an adversarial perturbation
    comes close to them;
  - greedy: no perturbation inside beta changes the argmax of a row the
    function calls safe, and a constructed one does change it where it calls a
    flip possible;
  - the C oracle's near-tie tests widen by exactly the stated amounts.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import gemm_bound as G

U1 = 2.0 ** -23   # ulp of 1.0 in fp32


def _bf16(a):
    t = torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    assert np.array_equal(t.double().numpy(), np.asarray(a, dtype=np.float64)), "not bf16-exact"
    return t


def _operands(seed, M, d, V, w_sigma=0.05, positive=False):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn(M, d, generator=g)
    w = torch.randn(V, d, generator=g) * w_sigma
    if positive:
        h, w = h.abs(), w.abs()
    return h.to(torch.bfloat16), w.to(torch.bfloat16)


def _simulate(h, w, mode, step=16):
    """fp32 accumulation of every (row, column) product sum in steps of `step`
    exact products, one rounding per step: 'rn' to nearest, 'rz' toward zero."""
    hh = h.to(torch.float64).numpy()
    ww = w.to(torch.float64).numpy()
    M, d = hh.shape
    V = ww.shape[0]
    acc = np.zeros((M, V), dtype=np.float32)
    for j in range(0, d, step):
        block = hh[:, j:j + step] @ ww[:, j:j + step].T      # exact: 16-bit products, few terms
        exact = acc.astype(np.float64) + block
        r = exact.astype(np.float32)                          # round to nearest
        if mode == "rz":
            over = np.abs(r.astype(np.float64)) > np.abs(exact)
            r[over] = np.nextafter(r[over], np.float32(0))
        acc = r
    return acc.astype(np.float64)


@pytest.mark.parametrize("d", [64, 256, 1024])
@pytest.mark.parametrize("mode", ["rn", "rz", "model"])
@pytest.mark.parametrize("positive", [False, True])
def test_bound_holds_for_simulated_accumulations(d, mode, positive):
    h, w = _operands(11 + d, 8, d, 200, positive=positive)
    z, beta = G.accumulation_bound(h, w)
    got = G.emulate(h, w) if mode == "model" else _simulate(h, w, mode)
    err = np.abs(got - z)
    assert np.all(err <= beta), (err / beta).max()


def _all_dropped(d=1024):
    """Accumulator 1.0 after the first step, then 16 products of 255 2^-33 per
    step: just below the grid 2^-25 of an accumulator of 1, so all dropped."""
    w = np.zeros((1, d))
    w[0, 0] = 1.0
    w[0, 16:] = 255 * 2.0 ** -33
    return _bf16(np.ones((1, d))), _bf16(w)


def test_dropped_bits_worst_case_reaches_the_bound():
    h, w = _all_dropped()
    z, beta = G.accumulation_bound(h, w)
    got = G.emulate(h, w)
    assert got[0, 0] == 1.0                      # nothing was ever added
    ratio = abs(got[0, 0] - z[0, 0]) / beta[0, 0]
    assert 0.75 <= ratio <= 1.0, ratio


def test_bound_without_the_dropped_bits_term_fails():
    """2u sum_j |S_j| alone (one faithful rounding of an exact step sum) is
    exceeded almost four times over on the same case."""
    h, w = _all_dropped()
    z, _ = G.accumulation_bound(h, w)
    ww = w.double().numpy()[0]
    S = np.cumsum([ww[j:j + 16].sum() for j in range(0, ww.size, 16)])
    assert abs(G.emulate(h, w)[0, 0] - z[0, 0]) > 3 * (2 * G.U32 * np.abs(S).sum())


def test_bound_over_the_wrong_step_fails():
    """beta taken over 64-product steps (four times fewer partial sums) does not
    bound the 16-product accumulation: the step is part of it."""
    h, w = _all_dropped()
    z, beta64 = G.accumulation_bound(h, w, step=64)
    assert abs(G.emulate(h, w)[0, 0] - z[0, 0]) > beta64[0, 0]


def test_final_rounding_worst_case_inside_the_bound():
    """Each step adds 255/256 of an ulp of the accumulator (1.0), which the
    rounding toward zero drops: inside beta (the final-rounding share, 2u per
    step, is a fifth of it here)."""
    d = 1024
    w = np.zeros((1, d))
    w[0, 0] = 1.0
    w[0, 16::16] = 255 * 2.0 ** -31
    h, w = _bf16(np.ones((1, d))), _bf16(w)
    z, beta = G.accumulation_bound(h, w)
    got = G.emulate(h, w)
    assert got[0, 0] == 1.0
    assert 0.15 <= abs(got[0, 0] - z[0, 0]) / beta[0, 0] <= 1.0


@pytest.mark.parametrize("entries,expected", [
    ([(0, 1.0)] + [(k, 2.0 ** -24) for k in range(1, 16)], 1.0 + 7 * U1),   # 1 + 7.5 ulp, toward zero
    ([(0, 1.0)] + [(k, 2.0 ** -25) for k in range(1, 16)], 1.0 + 3 * U1),   # 2^-25: on the grid (2 guard bits)
    ([(0, 1.0)] + [(k, 2.0 ** -26) for k in range(1, 16)], 1.0),            # 2^-26: below the grid, dropped
    ([(0, 1.0)] + [(k, -2.0 ** -26) for k in range(1, 16)], 1.0),           # negatives dropped toward zero
    ([(0, 1.0)] + [(k, -2.0 ** -25) for k in range(1, 16)], 1.0 - 8 * 2.0 ** -24),
    ([(0, 1.0)] + [(k, 2.0 ** -26) for k in range(16, 32)], 1.0),           # the accumulator sets the grid
    ([(k, 2.0 ** -26) for k in range(0, 16)] + [(16, 1.0)], 1.0 + 2 * U1),  # a small accumulator survives
    ([(0, 2.0 ** 20), (1, -2.0 ** 20), (2, 2.0 ** -10)], 0.0),              # grid 2^-5 after the cancellation
    ([(0, 2.0 ** 20), (1, -2.0 ** 20), (2, 2.0 ** -5)], 2.0 ** -5),
    ([(0, -1.0), (1, 3 * 2.0 ** -25)], -(1.0 - 2 * 2.0 ** -24)),            # toward zero for a negative sum
])
def test_model_on_hand_worked_operands(entries, expected):
    w = np.zeros((1, 64))
    for k, v in entries:
        w[0, k] = v
    got = G.emulate(_bf16(np.ones((1, 64))), _bf16(w))
    assert got[0, 0] == expected, (got[0, 0], expected)


def test_model_is_exact_when_every_addend_is_on_the_grid():
    """Small integers: every addend and partial sum is exact, so the model
    returns the exact sum."""
    rng = np.random.default_rng(1)
    h = rng.integers(-8, 9, size=(4, 256)).astype(np.float64)
    w = rng.integers(-8, 9, size=(6, 256)).astype(np.float64)
    assert np.array_equal(G.emulate(_bf16(h), _bf16(w)), h @ w.T)


def test_logits_equal_an_exactly_rounded_direct_sum():
    h, w = _operands(7, 3, 128, 5)
    z, _ = G.accumulation_bound(h, w)
    hh, ww = h.double().numpy(), w.double().numpy()
    for r in range(3):
        for v in range(5):
            assert z[r, v] == math.fsum(hh[r, k] * ww[v, k] for k in range(128))


def test_bound_value_on_a_hand_computed_case():
    """32 products of 1 x 1 in two steps: S = (16, 32), largest product 1 per
    step, previous sums (0, 16); the bound written out by hand."""
    h = _bf16(np.ones((1, 32)))
    w = _bf16(np.ones((1, 32)))
    z, beta = G.accumulation_bound(h, w)
    assert z[0, 0] == 32.0
    u = G.U32
    c1 = 2 * u * 16 + 8 * u * (1 + 2 * u) * max(0.0, 1.0)
    c2 = 2 * u * 32 + 8 * u * (1 + 2 * u) * max(16.0, 1.0)
    rho = (1 + 2 * u) * (1 + 8 * u)
    assert beta[0, 0] == pytest.approx(rho ** 2 * (1 + 2.0 ** -20) * (c1 + c2), rel=1e-14)

def _perturbations(beta, rng, n):
    yield beta.copy()
    yield -beta
    for _ in range(n):
        yield beta * rng.uniform(-1, 1, size=beta.shape)


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_p_moves_inside_its_band(T):
    rng = np.random.default_rng(3)
    V = 400
    z = rng.normal(0, 2, size=(6, V))
    beta = rng.uniform(1e-5, 5e-3, size=(6, V))
    p = G.softmax64(z, T)
    e_p, E = G.p_error_bounds(z, beta, T, p)
    e_gemm = (1 + e_p) / (1 + G.REL) - 1          # the GEMM share of the band
    q = G.softmax64(z + rng.normal(0, 0.5, size=z.shape), 1.0)
    r0 = np.maximum(0, p - q)
    worst = 0.0
    for dz in _perturbations(beta, rng, 50):
        pt = G.softmax64(z + dz, T)
        rel = np.abs(pt / p - 1)
        assert np.all(rel <= e_gemm * (1 + 1e-9))
        worst = max(worst, (rel / e_gemm).max())
        # partial masses of the residual and of p itself
        for r_new, r_old in ((np.maximum(0, pt - q), r0), (pt, p)):
            dC = np.abs(np.cumsum(r_new, axis=1) - np.cumsum(r_old, axis=1)).max(axis=1)
            assert np.all(dC <= E)
    # adversarial: +beta at one token, -beta elsewhere, moves p(v) by nearly the band
    v = 17
    dz = -beta.copy()
    dz[:, v] = beta[:, v]
    pt = G.softmax64(z + dz, T)
    rel_v = np.abs(pt[:, v] / p[:, v] - 1)
    assert np.all(rel_v >= 0.5 * e_gemm[:, v])
    assert worst <= 1.0


def test_greedy_flip_detection():
    rng = np.random.default_rng(9)
    z = rng.normal(0, 1, size=(200, 50))
    beta = np.full_like(z, 2e-3)
    # plant near ties in half of the rows
    top = np.argmax(z, axis=1)
    for r in range(0, 200, 2):
        v = (top[r] + 1) % 50
        z[r, v] = z[r, top[r]] - rng.uniform(0, 6e-3)
    flip = G.greedy_flip_possible(z, beta)
    assert flip[0::2].any() and not flip.all()
    for r in range(200):
        vs = np.argmax(z[r])
        if not flip[r]:
            for _ in range(20):
                assert np.argmax(z[r] + beta[r] * rng.uniform(-1, 1, 50)) == vs
        else:
            # the closest challenger, pushed up while v* is pushed down, wins or ties
            gap = z[r, vs] - z[r] - beta[r, vs] - beta[r]
            gap[vs] = np.inf
            c = int(np.argmin(gap))
            zz = z[r].copy()
            zz[vs] -= beta[r, vs]
            zz[c] += beta[r, c]
            assert zz[c] >= zz[vs]


def test_oracle_near_tie_bands_widen_as_stated():
    """One request, K = 1: the accept test's near-tie band grows by e_p p/q and
    the draw's by 2E/(R - E)."""
    z = np.log(np.array([[0.3, 0.2, 0.1, 0.1, 0.1, 0.1, 0.05, 0.05],
                         [0.125] * 8]))
    q = np.array([[0.2, 0.3, 0.1, 0.1, 0.1, 0.1, 0.05, 0.05]], dtype=np.float32)
    x = np.array([0], dtype=np.int32)
    ro = np.array([0, 2], dtype=np.int32)
    x1 = np.array([1], dtype=np.int32)  # p/q = 0.2/0.3 = 2/3
    ratio = 0.2 / float(q[0, 1])
    for du, ep, flagged in ((2e-6, 0.0, False), (2e-6, 4e-6, True), (-2e-6, 4e-6, True), (2e-5, 4e-6, False)):
        u = np.array([ratio + du, 0.5], dtype=np.float32)
        res = oracle.verify(z, q, x1, u, ro, 1.0, p_rel_err=[ep], mass_err=[0.0, 0.0])
        assert bool(res["near_tie_accept"][0]) == flagged, (du, ep)
    # the draw: bonus from p of row 1 (uniform over 8), u_K = 0.5 + 3e-6 lies 3e-6 past the boundary C(3)/R
    u = np.array([0.01, 0.5 + 3e-6], dtype=np.float32)
    ub = float(u[1]) - 0.5
    e0 = (ub - 1e-6) / 2      # band = 1e-6 + 2E / (1 - E) reaches ub at E ~ e0
    for E, flagged in ((0.0, False), (e0 * 1.01, True), (e0 * 0.98, False), (1.5, True)):
        res = oracle.verify(z, q, x, u, ro, 1.0, p_rel_err=[0.0], mass_err=[0.0, E])
        assert res["accept_len"][0] == 2
        assert bool(res["near_tie_sample"][0]) == flagged, E
