"""The bounded-wait path on the GPU, made to expire on purpose.

Every wait of the streaming verifier and of the LM-head GEMM on work that
other warps or CTAs produce gives up after the wait budget
(spec_set_wait_budget), flags SV_FLAG_TIMEOUT in the status word, lets the
CTA's own copies and MMAs land, releases its tensor memory and returns.  These
tests set a budget of a few cycles, so that the first wait expires, and check
that the call reports SV_ERR_TIMEOUT, that the context stays usable, and that
after re-zeroing the workspace and restoring the budget the same call matches
the oracle (and, for the GEMM, leaves no tensor memory held: a second GEMM
allocates it again).  No kernel traps, faults or hangs: the waits that expire
here are bounded by construction.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import gemm_bound as G
from speculative_decoding_verification_11_gb300 import binding as B_, workloads as W

from paritylib import compare_sampling

pytestmark = pytest.mark.gpu

TINY_BUDGET = 4  # SM cycles


@pytest.fixture
def streaming_only():
    prev_small = B_.spec_set_small_kernel_limit(0)
    prev_cluster = B_.spec_set_cluster_kernel(False)
    yield
    B_.spec_set_small_kernel_limit(prev_small)
    B_.spec_set_cluster_kernel(prev_cluster)
    B_.spec_set_wait_budget(0)


def _sample(dev, b, ws):
    rows = b.rows
    out = torch.full((rows,), -9, dtype=torch.int32, device=dev)
    al = torch.full((b.B,), -9, dtype=torch.int32, device=dev)
    dg = torch.full((rows + b.B,), float("nan"), device=dev)
    B_.spec_verify_sample(b.logits.to(dev), b.q.to(dev), b.B, b.K, b.V, b.temperature, b.draft.to(dev),
                          b.uniforms.to(dev), out, al, ws, diag=dg)
    return out, al, dg


def test_streaming_verifier_times_out_then_recovers(cuda_device, streaming_only):
    dev = cuda_device
    b = W.make_sampling_batch("timeout", 71, B=8, K=3, V=40000, T=1.0, logit_sigma=2.0, noise_sigma=1.0)
    ws = B_.workspace(B_.spec_verify_workspace_size(b.B, b.rows, b.V), dev)
    assert B_.spec_set_wait_budget(TINY_BUDGET) == 4000000000
    _sample(dev, b, ws)
    assert B_.spec_last_kernel() == "stream"
    st, flags = B_.spec_verify_last_device_status(ws)
    assert st == B_.SV_ERR_TIMEOUT and flags & B_.SV_FLAG_TIMEOUT, (st, flags)
    # the context is usable; re-zero the workspace, restore the budget, run again
    B_.spec_set_wait_budget(0)
    ws.zero_()
    out, al, dg = _sample(dev, b, ws)
    torch.cuda.synchronize()
    st, flags = B_.spec_verify_last_device_status(ws)
    assert st == B_.SV_OK and not flags & B_.SV_FLAG_TIMEOUT
    orc = oracle.verify(b.logits, b.q, b.draft, b.uniforms, b.row_offsets, b.temperature)
    compare_sampling("after a timeout: stream B=8 K=3 V=40000", b.row_offsets, out.cpu().numpy(),
                     al.cpu().numpy(), dg.cpu().numpy(), orc)


def test_lmhead_gemm_times_out_then_recovers(cuda_device):
    dev = cuda_device
    g = torch.Generator().manual_seed(5)
    M, d, V = 64, 512, 9000
    h = torch.randn(M, d, generator=g).to(torch.bfloat16)
    w = (torch.randn(V, d, generator=g) * 0.05).to(torch.bfloat16)
    hd, wd = h.to(dev), w.to(dev)
    out = torch.zeros(M, V, device=dev)
    ws = B_.workspace(B_.spec_draft_workspace_size(M, d, V), dev)
    try:
        B_.spec_set_wait_budget(TINY_BUDGET)
        B_.spec_lmhead_logits(hd, wd, out, ws)
        st, flags = B_.spec_verify_last_device_status(ws)
        assert st == B_.SV_ERR_TIMEOUT and flags & B_.SV_FLAG_TIMEOUT, (st, flags)
    finally:
        B_.spec_set_wait_budget(0)
    z, beta = G.accumulation_bound(h, w)
    for _ in range(2):  # each GEMM allocates tensor memory on every SM it runs on again
        ws.zero_()
        out.fill_(float("nan"))
        B_.spec_lmhead_logits(hd, wd, out, ws)
        st, flags = B_.spec_verify_last_device_status(ws)
        assert st == B_.SV_OK, (st, flags)
        assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - z) <= beta)
