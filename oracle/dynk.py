"""Oracle of the dynamic draft-length (K) controller run after verification.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): plain Python per request.

What it follows: "Hardware Aware Dynamic Speculative Decoding", section
"Dynamic speculative decoding" (the number of draft tokens is adapted; the metric is goodput = AL / ITL, with ITL the
inter-token latency, largely draft plus verify time; the optimal K is kept in
a table that can take live AL and ITL statistics), and "Speculative Decoding
in Production: Accelerating LLM Inference via Custom Draft Models",
"Production Failure Modes and Mitigation Strategies", item 1 (dynamic window
sizing: when the running average of accepted tokens over the last 10 falls
below 1.5, K drops from 5 to 1 or 2).

Readings:
  - State per request: a ring of its last W verification results (AL, K used),
    and how many results were pushed.  A result with AL = 0 (an invalid
    request) is not pushed.
  - Window rule: K_next = k_low if the mean AL over the ring is below the
    threshold, else k_high (k_high while the ring is empty).  The pages'
    "last 10 requests" is read as the request's last W steps, so that each
    request's K_i adapts.
  - Goodput rule: each result gives AL - 1 accepted drafts (successes) and one
    failure if AL - 1 < K (a rejection stopped it); alpha = S / (S + F) over
    the ring (alpha_prior when S + F = 0).  Expected AL with K drafts:
    E(0) = 1, E(K) = E(K - 1) + alpha^K (the truncated geometric sum of
    "Speculative Decoding in Large Language Models", E[N] = (1 - a^(K+1)) /
    (1 - a)), accumulated in fp32 in that order; K_next = the K in
    [k_low, k_high] maximising E(K) / itl[K] in fp32 (the smaller K on ties),
    itl[K] the caller's profiled step time with K drafts.
  - Row offsets for a ragged verification: offsets[b] = sum_{i<b} (K_i + 1).
Decisions are taken in fp32 on both sides (the kernel's precision), so they
agree exactly.

Parity: exact; pinned by the closed form of E[N], the estimator's convergence
on simulated acceptance, and hand-worked cases (tests/test_oracle_pins_dynk.py).
"""
from __future__ import annotations

import numpy as np

WINDOW, GOODPUT = 0, 1


def push(hist, count, b, al, k, W):
    """Append (al, k) to request b's ring (in place)."""
    if al <= 0:
        return
    slot = int(count[b]) % W
    hist[b, slot, 0] = al
    hist[b, slot, 1] = k
    count[b] += 1


def ring(hist, count, b, W):
    n = min(int(count[b]), W)
    return [(int(hist[b, i, 0]), int(hist[b, i, 1])) for i in range(n)]


def expected_al_f32(alpha, K):
    """E(K) accumulated in fp32: 1 + alpha + ... + alpha^K."""
    a = np.float32(alpha)
    e = np.float32(1.0)
    p = np.float32(1.0)
    for _ in range(K):
        p = np.float32(p * a)
        e = np.float32(e + p)
    return e


def choose_window(entries, threshold, k_low, k_high):
    if not entries:
        return k_high
    tot = np.float32(sum(al for al, _ in entries))
    mean = np.float32(tot / np.float32(len(entries)))
    return k_low if mean < np.float32(threshold) else k_high


def alpha_estimate(entries, alpha_prior):
    S = sum(al - 1 for al, _ in entries)
    F = sum(1 for al, k in entries if al - 1 < k)
    if S + F == 0:
        return np.float32(alpha_prior)
    return np.float32(np.float32(S) / np.float32(S + F))


def choose_goodput(entries, itl, k_low, k_high, alpha_prior):
    a = alpha_estimate(entries, alpha_prior)
    best_k, best_g = k_low, None
    e = np.float32(1.0)
    p = np.float32(1.0)
    for K in range(0, k_high + 1):
        if K > 0:
            p = np.float32(p * a)
            e = np.float32(e + p)
        if K < k_low:
            continue
        g = np.float32(e / np.float32(itl[K]))
        if best_g is None or g > best_g:
            best_k, best_g = K, g
    return best_k


def update(accept_len, k_used, hist, count, W, policy, threshold, k_low, k_high, itl=None, alpha_prior=0.5):
    """One controller step for a batch.  hist (B, W, 2) and count (B,) are
    updated in place; returns (k_next (B,), row_offsets (B + 1,))."""
    B = len(accept_len)
    k_next = np.zeros(B, dtype=np.int32)
    for b in range(B):
        push(hist, count, b, int(accept_len[b]), int(k_used[b]), W)
        entries = ring(hist, count, b, W)
        if policy == WINDOW:
            k_next[b] = choose_window(entries, threshold, k_low, k_high)
        else:
            k_next[b] = choose_goodput(entries, itl, k_low, k_high, alpha_prior)
    offs = np.zeros(B + 1, dtype=np.int32)
    offs[1:] = np.cumsum(k_next + 1)
    return k_next, offs
