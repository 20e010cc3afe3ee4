"""The seeded input generators against the input recipe they state: shapes,
layouts, value laws and structure, at reduced sizes.  The generators hold no
verification arithmetic; these tests keep their inputs what the workload
descriptions say they are."""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import pytest
import torch

from oracle import draft as D
from speculative_decoding_verification_11_gb300 import workloads as W


def _check_batch_layout(b, ks):
    ro = b.row_offsets.numpy()
    assert ro[0] == 0 and np.array_equal(np.diff(ro), np.asarray(ks) + 1)
    R, nq = int(ro[-1]), int(ro[-1]) - len(ks)
    assert b.logits.shape == (R, b.V)
    assert b.draft.shape == (nq,) and b.draft.dtype == torch.int32
    assert int(b.draft.min()) >= 0 and int(b.draft.max()) < b.V
    if b.q is not None:
        assert b.q.shape == (nq, b.V) and b.q.dtype == torch.float32
        assert torch.allclose(b.q.double().sum(1), torch.ones(nq, dtype=torch.float64), atol=1e-5)
        assert b.uniforms.shape == (R,) and b.uniforms.dtype == torch.float32


def test_sampling_recipe():
    b = W.sampling(B=6, K=4, V=4096)
    _check_batch_layout(b, [4] * 6)
    assert b.temperature == 0.7 and b.logits.dtype == torch.float32
    z = b.logits.numpy().astype(np.float64)
    # N(0, 2^2) plus 32 entries per row raised by 8: the rest of the row keeps the normal law
    body = np.sort(z, axis=1)[:, :-64]
    assert 1.8 < z[:, :].std() < 2.4 and abs(float(np.median(z))) < 0.1
    assert body.std() < 2.1
    # entries above 5.5 per row: 32 boosted ones from N(8, 2^2), the rest from the N(0, 2^2) tail
    phi = lambda t: 0.5 * (1.0 + math.erf(t / math.sqrt(2.0)))
    expect = 32 * phi((8.0 - 5.5) / 2.0) + (4096 - 32) * (1.0 - phi(5.5 / 2.0))
    assert abs((z > 5.5).sum(1).mean() - expect) < 3.0, expect


def test_boosted_entries_are_distinct_and_uniformly_placed():
    b = W.make_sampling_batch("probe", 3, B=64, K=1, V=512, T=1.0, logit_sigma=1.0, noise_sigma=1.0, boost=32,
                              boost_value=1000.0)
    z = b.logits.numpy()
    hit = z > 500
    assert np.all(hit.sum(1) == 32)  # exactly 32 distinct indices per row
    per_index = hit.sum(0)            # 128 rows x 32 hits spread over 512 indices: 8 per index on average
    assert per_index.max() < 30 and (per_index > 0).mean() > 0.9


def test_sampling_uniforms_are_philox_stream_zero():
    """The verifier's uniforms: Philox4x32-10 at counter (row, stream 0), the
    same values the oracle's own Philox gives for those counters."""
    seed = 1002
    b = W.sampling(seed=seed, B=2, K=4, V=256)
    want = np.array([D.philox_uniform(seed, r, stream=0) for r in range(b.rows)])
    assert np.array_equal(b.uniforms.numpy().astype(np.float64), want)
    assert np.all(want > 0) and np.all(want < 1)


def test_drafts_follow_q():
    """x ~ q: over many rows, the count of each drafted id matches the sum of
    that id's probability over the rows (5 sigma)."""
    b = W.make_sampling_batch("probe", 8, B=4000, K=1, V=8, T=1.0, logit_sigma=0.0, noise_sigma=1.0)
    # logit_sigma 0: target rows are 0, so each draft row is N(0, 1) noise and q varies by row
    q = b.q.numpy().astype(np.float64)
    x = b.draft.numpy()
    expect = q.sum(0)
    counts = np.bincount(x, minlength=8).astype(np.float64)
    assert np.all(np.abs(counts - expect) < 5 * np.sqrt(expect) + 1)


def test_ragged_recipe():
    b = W.ragged(B=400, V=64)
    ks = (np.diff(b.row_offsets.numpy()) - 1).tolist()
    _check_batch_layout(b, ks)
    assert min(ks) == 0 and max(ks) == 8 and set(ks) == set(range(9))
    assert abs(np.mean(ks) - 4.0) < 0.5
    assert b.K is None and b.temperature == 1.0


def test_greedy_recipe():
    b = W.greedy(B=8, K=5, V=3000)
    _check_batch_layout(b, [5] * 8)
    assert b.logits.dtype == torch.bfloat16 and b.q is None and b.uniforms is None and b.temperature == 0.0
    z = b.logits.float().numpy()
    assert 2.8 < z.std() < 3.2
    # x_j = argmax(z_j + N(0, 1.5^2)): z at the drafted id sits in the row's top tail
    idx = W._draft_rows_index(b.row_offsets).numpy()
    zx = z[idx, b.draft.numpy()]
    assert np.mean(zx) > 6.0


def test_tiny_recipe():
    b = W.tiny(steps=30)
    _check_batch_layout(b, [4] * 30)
    assert b.V == 1024 and b.temperature == 1.0


def test_lmhead_recipe():
    b = W.lmhead(seed=5, B=2, K=3, d=256, V=1000, d_draft=128, T=1.0)
    M = 2 * 4
    assert b.hidden.shape == (M, 256) and b.hidden.dtype == torch.bfloat16
    assert b.w_vocab_t.shape == (1000, 256) and b.w_vocab_t.dtype == torch.bfloat16
    assert 0.9 < b.hidden.float().std() < 1.1
    assert 0.018 < b.w_vocab_t.float().std() < 0.022
    # no logits in this workload (the GEMM makes them): check the rest of the layout with a stand-in
    _check_batch_layout(dataclasses.replace(b, logits=torch.zeros(M, b.V)), [3, 3])


@pytest.mark.parametrize("L", [3000, 8192])
def test_repetitive_streams_recipe(L):
    """Streams of L tokens over a 32000-token vocabulary where about 5% of the
    steps copy a span of 8-64 earlier tokens: about two thirds of the tokens
    are copies, so 8-grams repeat far more often than chance allows."""
    tokens, offs = W.repetitive_streams(seed=1006, B=6, L=L)
    assert np.array_equal(offs, np.arange(7) * L) and tokens.dtype == np.int32
    assert tokens.min() >= 0 and tokens.max() < 32000
    for b in range(6):
        s = tokens[offs[b]:offs[b + 1]]
        grams = {}
        for i in range(len(s) - 7):
            grams.setdefault(s[i:i + 8].tobytes(), 0)
            grams[s[i:i + 8].tobytes()] += 1
        repeated = sum(c for c in grams.values() if c > 1) / (len(s) - 7)
        assert 0.3 < repeated < 0.9, repeated
