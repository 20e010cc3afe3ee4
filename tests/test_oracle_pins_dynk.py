"""Pins of the dynamic-K controller oracle (oracle/dynk.py) against facts
outside its own code: the closed form of the expected accepted length, the
estimator's convergence on simulated acceptance, the pages' worked rule (K 5
-> 2 when the average of the last 10 falls below 1.5), and brute-force argmax
on well-separated goodput curves.
"""
from __future__ import annotations

import numpy as np
import pytest

from oracle import dynk, speedup


@pytest.mark.parametrize("alpha", [0.0, 0.3, 0.6, 0.85, 0.99])
def test_expected_al_matches_the_closed_form(alpha):
    for K in range(0, 12):
        got = float(dynk.expected_al_f32(alpha, K))
        want = speedup.expected_tokens(alpha, K)
        assert abs(got - want) <= 1e-6 * want, (alpha, K, got, want)


def test_alpha_estimate_converges_on_simulated_acceptance():
    """Drafts accepted independently with probability alpha, stopping at the
    first rejection: S / (S + F) estimates alpha."""
    rng = np.random.default_rng(4)
    for alpha in (0.2, 0.55, 0.8):
        entries = []
        for _ in range(20000):
            K = int(rng.integers(1, 8))
            acc = 0
            while acc < K and rng.random() < alpha:
                acc += 1
            entries.append((acc + 1, K))
        est = float(dynk.alpha_estimate(entries, 0.5))
        assert abs(est - alpha) < 0.01, (alpha, est)


def test_window_rule_of_the_pages():
    """K = 5 while the average accepted length over the last 10 stays at or
    above 1.5; K = 2 once it falls below; back to 5 when it recovers."""
    W, B = 10, 1
    hist = np.zeros((B, W, 2), dtype=np.int32)
    count = np.zeros(B, dtype=np.int32)
    seq = [3] * 10 + [1] * 7 + [1, 1, 1] + [4] * 10
    ks = []
    for al in seq:
        k, _ = dynk.update([al], [5], hist, count, W, dynk.WINDOW, 1.5, 2, 5)
        ks.append(int(k[0]))
    means = [np.mean(seq[max(0, i - 9):i + 1]) for i in range(len(seq))]
    assert ks == [2 if m < 1.5 else 5 for m in means]
    assert ks[:10] == [5] * 10 and 2 in ks and ks[-1] == 5


def test_goodput_argmax_matches_brute_force_when_separated():
    rng = np.random.default_rng(9)
    checked = 0
    for _ in range(300):
        alpha = float(rng.uniform(0.05, 0.95))
        k_hi = int(rng.integers(1, 10))
        base = float(rng.uniform(5, 20))
        slope = float(rng.uniform(0.0, 4.0))
        itl = np.array([base + slope * k for k in range(k_hi + 1)], dtype=np.float32)
        g = [speedup.expected_tokens(alpha, k) / float(itl[k]) for k in range(k_hi + 1)]
        order = np.sort(g)
        if len(g) > 1 and order[-1] - order[-2] < 1e-4 * order[-1]:
            continue  # near tie: either K is right
        got = dynk.choose_goodput([], itl, 0, k_hi, alpha)
        assert got == int(np.argmax(g)), (alpha, k_hi, base, slope)
        checked += 1
    assert checked > 200


def test_goodput_edges():
    itl = np.array([10, 10, 10, 10], dtype=np.float32)
    assert dynk.choose_goodput([], itl, 0, 3, 0.9) == 3      # flat cost: more drafts never hurt
    assert dynk.choose_goodput([], itl, 1, 3, 0.0) == 1      # nothing accepted: the smallest allowed K
    steep = np.array([10, 40, 80, 120], dtype=np.float32)
    assert dynk.choose_goodput([], steep, 0, 3, 0.5) == 0


def test_ring_keeps_the_last_w_results_and_skips_invalid():
    W = 3
    hist = np.zeros((1, W, 2), dtype=np.int32)
    count = np.zeros(1, dtype=np.int32)
    for al in (2, 0, 3, 4, 5):
        dynk.update([al], [4], hist, count, W, dynk.WINDOW, 1.5, 1, 4)
    assert int(count[0]) == 4
    assert sorted(a for a, _ in dynk.ring(hist, count, 0, W)) == [3, 4, 5]


def test_offsets_for_ragged_verification():
    W = 2
    hist = np.zeros((3, W, 2), dtype=np.int32)
    count = np.zeros(3, dtype=np.int32)
    k, offs = dynk.update([1, 4, 2], [3, 3, 3], hist, count, W, dynk.WINDOW, 2.0, 1, 6)
    assert list(k) == [1, 6, 6]
    assert list(offs) == [0, 2, 9, 16]
