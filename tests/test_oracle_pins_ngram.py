"""Pins of the n-gram drafter oracle (oracle/ngram.py) against facts outside its
own code: Python's str.rfind over an encoding of the tokens (one character per
token), the closed form of a periodic stream, and special cases.
"""
from __future__ import annotations

import numpy as np
import pytest

from oracle import ngram


def _rfind_propose(ctx, K, n_min, n_max):
    s = "".join(chr(0x100 + t) for t in ctx)
    L = len(s)
    for n in range(n_max, n_min - 1, -1):
        if n <= 0 or n > L - 1:
            continue
        i = s.rfind(s[L - n:], 0, L - 1)  # the window lies inside s[0 : L-1]
        if i >= 0:
            return [ord(c) - 0x100 for c in s[i + n:i + n + K]]
    return []


@pytest.mark.parametrize("alphabet", [2, 3, 8])
def test_matches_rfind_on_random_streams(alphabet):
    rng = np.random.default_rng(alphabet)
    for _ in range(400):
        L = int(rng.integers(1, 40))
        ctx = rng.integers(0, alphabet, size=L).tolist()
        K = int(rng.integers(1, 8))
        n_max = int(rng.integers(1, 6))
        n_min = int(rng.integers(1, n_max + 1))
        got, _ = ngram.propose(ctx, K, n_min, n_max)
        assert got == _rfind_propose(ctx, K, n_min, n_max), (ctx, K, n_min, n_max)


def test_periodic_stream_proposes_the_next_period_tokens():
    period = [5, 9, 2, 7, 7, 1]
    for L in range(len(period) * 2, len(period) * 6):
        ctx = [period[i % len(period)] for i in range(L)]
        got, _ = ngram.propose(ctx, 4, 2, 4)
        assert got == [period[(L + j) % len(period)] for j in range(4)]


def test_no_repetition_proposes_nothing():
    got, e = ngram.propose(list(range(50)), 5, 1, 3)
    assert got == [] and e == -1


def test_proposal_is_cut_at_the_context_end():
    ctx = [1, 2, 3, 1, 2]   # suffix [1, 2] occurs at 0..1; only 3 tokens follow before the end
    got, e = ngram.propose(ctx, 8, 1, 2)
    assert e == 1 and got == [3, 1, 2]


def test_longer_match_wins_over_later_shorter_one():
    #          0  1  2  3  4  5  6  7  8
    ctx = [4, 6, 8, 0, 9, 8, 3, 4, 6, 8]
    # suffix 3 = [4, 6, 8] occurs at 0..2 (followed by 0); suffix 1 = [8] also at 5 (later)
    got, e = ngram.propose(ctx, 2, 1, 3)
    assert e == 2 and got == [0, 9]
    got, e = ngram.propose(ctx, 2, 1, 1)
    assert e == 5 and got == [3, 4]


def test_short_contexts_and_bounds():
    assert ngram.propose([], 3, 1, 2) == ([], -1)
    assert ngram.propose([7], 3, 1, 2) == ([], -1)
    assert ngram.propose([7, 7], 3, 1, 2) == ([7], 0)
    assert ngram.propose([1, 2, 1, 2], 3, 3, 3) == ([], -1)  # n = 3 has no earlier occurrence
