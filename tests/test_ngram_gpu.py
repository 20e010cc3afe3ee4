"""GPU parity of the n-gram (prompt lookup) drafter (spec_ngram_draft) against
the oracle (oracle/ngram.py): integer work, so drafts and counts are equal."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import ngram
from speculative_decoding_verification_11_gb300 import binding as B_, workloads as W

pytestmark = pytest.mark.gpu


def _gpu(dev, tokens, offs, K, n_min, n_max):
    B = len(offs) - 1
    t = torch.from_numpy(np.ascontiguousarray(tokens, dtype=np.int32)).to(dev) if len(tokens) else \
        torch.zeros(1, dtype=torch.int32, device=dev)
    o = torch.from_numpy(np.asarray(offs, dtype=np.int32)).to(dev)
    d = torch.full((B, K), -7, dtype=torch.int32, device=dev)
    k = torch.full((B,), -7, dtype=torch.int32, device=dev)
    B_.spec_ngram_draft(t, o, K, n_min, n_max, d, k)
    torch.cuda.synchronize()
    return d.cpu().numpy(), k.cpu().numpy()


def _oracle(tokens, offs, K, n_min, n_max):
    ctxs = [list(tokens[offs[b]:offs[b + 1]]) for b in range(len(offs) - 1)]
    d, k = ngram.propose_batch(ctxs, K, n_min, n_max)
    return np.asarray(d, dtype=np.int32).reshape(len(ctxs), K), np.asarray(k, dtype=np.int32)


@pytest.mark.parametrize("alphabet,K,n_min,n_max", [(2, 4, 1, 3), (5, 8, 2, 4), (50, 6, 1, 1), (3, 1, 3, 32)])
def test_random_streams_match_oracle(cuda_device, alphabet, K, n_min, n_max):
    rng = np.random.default_rng(alphabet * 100 + K)
    lens = [0, 1, 2, 3] + rng.integers(4, 700, size=60).tolist()
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tokens = rng.integers(0, alphabet, size=int(offs[-1])).astype(np.int32)
    d, k = _gpu(cuda_device, tokens, offs, K, n_min, n_max)
    od, ok = _oracle(tokens, offs, K, n_min, n_max)
    assert np.array_equal(k, ok) and np.array_equal(d, od)


def test_repetitive_streams_workload(cuda_device):
    tokens, offs = W.repetitive_streams(seed=1006, B=32, L=3000)
    d, k = _gpu(cuda_device, tokens, offs, 8, 1, 4)
    od, ok = _oracle(tokens, offs, 8, 1, 4)
    assert np.array_equal(k, ok) and np.array_equal(d, od)
    assert (k > 0).mean() > 0.5  # the streams repeat: most requests find a match


@pytest.mark.parametrize("L", [8192, 32768])
def test_timed_workload_at_full_size(cuda_device, L):
    """The timed drafting workload at its own sizes (B = 256 contexts of L
    tokens, K = 8, n = 1..4): every request against the oracle."""
    tokens, offs = W.repetitive_streams(seed=1006, B=256, L=L)
    d, k = _gpu(cuda_device, tokens, offs, 8, 1, 4)
    od, ok = _oracle(tokens, offs, 8, 1, 4)
    assert np.array_equal(k, ok) and np.array_equal(d, od)
    assert 0 < (k > 0).mean() < 1  # both outcomes occur


def test_decreasing_offsets_propose_nothing(cuda_device):
    tokens = np.array([1, 2, 1, 2, 1, 2], dtype=np.int32)
    d, k = _gpu(cuda_device, tokens, [0, 6, 2], 3, 1, 2)
    assert k[0] == 2 and list(d[0]) == [1, 2, -1]
    assert k[1] == 0 and list(d[1]) == [-1, -1, -1]


def test_negative_start_proposes_nothing(cuda_device):
    """A context whose first offset is negative is empty: nothing proposed,
    no token read; the next request is unaffected."""
    tokens = np.array([1, 2, 1, 2, 1, 2], dtype=np.int32)
    d, k = _gpu(cuda_device, tokens, [-3, 0, 6], 3, 1, 2)
    assert k[0] == 0 and list(d[0]) == [-1, -1, -1]
    assert k[1] == 2 and list(d[1]) == [1, 2, -1]


def test_ngram_argument_errors(cuda_device):
    dev = cuda_device
    t = torch.zeros(4, dtype=torch.int32, device=dev)
    o = torch.tensor([0, 4], dtype=torch.int32, device=dev)
    d = torch.zeros(1, 2, dtype=torch.int32, device=dev)
    k = torch.zeros(1, dtype=torch.int32, device=dev)
    for n_min, n_max in ((0, 2), (3, 2), (1, 33)):
        with pytest.raises(B_.SpecVerifyError):
            B_.spec_ngram_draft(t, o, 2, n_min, n_max, d, k)


@pytest.mark.parametrize("shift", [0, 1, 2, 3])
def test_long_contexts_at_every_alignment(cuda_device, shift):
    """Contexts that wrap each CTA's ring of shared-memory stages (several
    stages per CTA) and start at every 4-byte position of a 16-byte group: the
    token buffer itself starts `shift` elements into an allocation, and the
    context lengths are odd, so both ends of each stage's bulk copy fall at
    every alignment.  Short contexts (no aligned interior at all) sit between
    them."""
    dev = cuda_device
    rng = np.random.default_rng(77 + shift)
    lens = [2, 3, 4, 5, 6, 7, 8, 9, 31, 33, 8193, 24577, 30001] + rng.integers(10, 40000, size=5).tolist()
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tokens = rng.integers(0, 3, size=int(offs[-1])).astype(np.int32)
    full = torch.zeros(len(tokens) + shift, dtype=torch.int32, device=dev)
    full[shift:] = torch.from_numpy(tokens).to(dev)
    t = full[shift:]
    o = torch.from_numpy(offs).to(dev)
    K, n_min, n_max = 8, 2, 7
    d = torch.full((len(lens), K), -7, dtype=torch.int32, device=dev)
    k = torch.full((len(lens),), -7, dtype=torch.int32, device=dev)
    B_.spec_ngram_draft(t, o, K, n_min, n_max, d, k)
    torch.cuda.synchronize()
    od, ok = _oracle(tokens, offs, K, n_min, n_max)
    assert np.array_equal(k.cpu().numpy(), ok) and np.array_equal(d.cpu().numpy(), od)


@pytest.mark.parametrize("n_max", [4, 32])
def test_dense_matches(cuda_device, n_max):
    """Contexts where most or all candidate ends equal the last token: a
    constant context, short periods, and a long periodic run after random
    tokens (every warp pass holds matches, up to 128 per 32-group block, and
    the extensions run to n_max).  Lengths span one to several shared-memory
    stages per CTA."""
    rng = np.random.default_rng(90 + n_max)
    ctxs = []
    for L in (40, 2049, 9000, 30001):
        ctxs.append(np.full(L, 7, dtype=np.int32))                                   # constant
        for p in (2, 5, 31):
            base = rng.integers(0, 1000, size=p).astype(np.int32)
            ctxs.append(np.resize(base, L))                                          # period p
        head = rng.integers(0, 1000, size=L // 2).astype(np.int32)
        ctxs.append(np.concatenate([head, np.resize(np.array([3, 9, 3], np.int32), L - L // 2)]))
    lens = [len(c) for c in ctxs]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tokens = np.concatenate(ctxs).astype(np.int32)
    d, k = _gpu(cuda_device, tokens, offs, 8, 1, n_max)
    od, ok = _oracle(tokens, offs, 8, 1, n_max)
    assert np.array_equal(k, ok) and np.array_equal(d, od)
