"""GPU parity of the draft side (spec_draft_sample: tcgen05 GEMM, q in place,
Philox inverse-CDF draw) against the fp64 oracle (oracle/draft.py).

  u   bit-exact (both sides implement Philox4x32-10 from its definition);
  q   within e_p(v) relative of the fp64 softmax, element by element: the
      bound oracle/gemm_bound.py derives from the a-priori bound beta on the
      GEMM's fp32 accumulation error (exp(b_v + L)(1 + 1e-5) - 1, b = beta/T);
  x   identical except rows the oracle flags as near ties (a CDF boundary
      within 1e-6 + 2E/(1 - E) of u, E = sum_v e_p(v) q(v) the bound on the
      error of the row's masses); greedy: identical except rows where some
      v != argmax has z_argmax - z_v <= beta_argmax + beta_v.
The measured error / bound ratios are reported.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import draft as D
from oracle import gemm_bound as G
from speculative_decoding_verification_11_gb300 import binding as B_

from paritylib import record

pytestmark = pytest.mark.gpu


def _inputs(seed, M, d, V, w_sigma=0.02):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn(M, d, generator=g).to(torch.bfloat16)
    w = (torch.randn(V, d, generator=g) * w_sigma).to(torch.bfloat16)
    return h, w


def _gpu(dev, h, w, T, seed, offset):
    M, V = h.shape[0], w.shape[0]
    q = torch.full((M, V), float("nan"), device=dev) if T > 0 else None
    x = torch.full((M,), -9, dtype=torch.int32, device=dev)
    u = torch.full((M,), float("nan"), device=dev)
    ws = B_.workspace(B_.spec_draft_workspace_size(M, h.shape[1], V), dev)
    B_.spec_draft_sample(h.to(dev), w.to(dev), T, seed, offset, q, x, ws, u_out=u)
    torch.cuda.synchronize()
    return (q.cpu().numpy() if q is not None else None), x.cpu().numpy(), u.cpu().numpy()


@pytest.mark.parametrize("M,d,V,T,w_sigma", [(16, 256, 4000, 0.9, 0.1), (128, 1024, 20000, 1.0, 0.05),
                                             (128, 2048, 128256, 1.0, 0.02), (3, 64, 1028, 0.5, 0.2)])
def test_draft_sampling_matches_oracle(cuda_device, M, d, V, T, w_sigma):
    h, w = _inputs(M + d + V, M, d, V, w_sigma)
    seed, offset = 0xC0FFEE + M, 1234
    q, x, u = _gpu(cuda_device, h, w, T, seed, offset)
    bands = G.bands(h, w, T)
    orc = D.draft_sample(h, w, T, seed, offset, bands=bands)
    assert np.array_equal(u.astype(np.float64), orc["u"])
    qo = orc["q"]
    big = qo > 1e-30
    assert np.all(np.isfinite(q))
    rel = np.abs(q[big] - qo[big]) / qo[big]
    ratio = rel / bands.e_p[big]
    assert ratio.max() <= 1.0, ratio.max()
    same = x == orc["x"]
    assert np.all(same | orc["near_tie"]), np.nonzero(~same & ~orc["near_tie"])
    record(f"draft sample M={M} d={d} V={V} T={T}", {"q_max_rel_err": float(rel.max()),
                                                     "q_err_over_bound": float(ratio.max()),
                                                     "x_mismatch": int((~same).sum()),
                                                     "near_ties": int(orc["near_tie"].sum())})


@pytest.mark.parametrize("M,d,V", [(16, 256, 4000), (128, 1024, 20000), (128, 2048, 128256)])
def test_greedy_drafting_is_argmax(cuda_device, M, d, V):
    h, w = _inputs(7 + M, M, d, V, 0.05)
    _, x, _ = _gpu(cuda_device, h, w, 0.0, 0, 0)
    z, beta = G.accumulation_bound(h, w)
    orc = D.draft_sample(h, w, 0.0, 0, bands=G.Bands(logits=z, beta=beta, T=0.0))
    flip = G.greedy_flip_possible(z, beta)
    same = x == orc["x"]
    assert np.all(same | flip), np.nonzero(~same & ~flip)
    record(f"draft greedy M={M} d={d} V={V}", {"x_mismatch": int((~same).sum()), "near_ties": int(flip.sum())})


def test_offsets_give_independent_draws(cuda_device):
    """The same rows at two counter offsets draw different uniforms, each the
    oracle's for its counter."""
    h, w = _inputs(99, 8, 128, 2048, 0.1)
    _, _, u1 = _gpu(cuda_device, h, w, 1.0, 5, 0)
    _, _, u2 = _gpu(cuda_device, h, w, 1.0, 5, 8)
    assert not np.array_equal(u1, u2)
    assert np.array_equal(u2.astype(np.float64), [D.philox_uniform(5, 8 + r) for r in range(8)])


def test_draft_argument_errors(cuda_device):
    dev = cuda_device
    h = torch.zeros(16, 128, dtype=torch.bfloat16, device=dev)
    x = torch.zeros(16, dtype=torch.int32, device=dev)
    ws = B_.workspace(B_.spec_draft_workspace_size(16, 128, 1000), dev)
    for V, dd in ((1002, 128), (1000, 100)):  # V not a multiple of 4; d not a multiple of 64
        w = torch.zeros(V, dd, dtype=torch.bfloat16, device=dev)
        hh = torch.zeros(16, dd, dtype=torch.bfloat16, device=dev)
        q = torch.zeros(16, V, device=dev)
        with pytest.raises(B_.SpecVerifyError) as e:
            B_.spec_draft_sample(hh, w, 1.0, 0, 0, q, x, ws)
        assert e.value.status == B_.SV_ERR_INVALID
    big = torch.zeros(129, 128, dtype=torch.bfloat16, device=dev)  # M > 128
    w = torch.zeros(1000, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(B_.SpecVerifyError):
        B_.spec_draft_sample(big, w, 1.0, 0, 0, torch.zeros(129, 1000, device=dev),
                             torch.zeros(129, dtype=torch.int32, device=dev), ws)
    del h
