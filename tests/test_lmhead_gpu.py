"""GPU parity of the fused LM-head front end (tcgen05 GEMM + verifier) against
the fp64 oracle (fp64 GEMM of the bf16 operands, then the same steps).

The GPU's logits come from an fp32 accumulation on the tensor cores, so they
differ from the fp64 GEMM by a rounding error that grows with d.  The parity
rule is the verifier's with its bands widened to cover that error:
  LM_REL   relative tolerance on p_j(x_j) and on the residual quantities;
  LM_BAND  near-tie band for the accept test and the final draw (oracle-side,
           in fp64);
  greedy   tokens identical except rows whose fp64 top-2 logits lie within
           LM_GAP (then either order is a valid argmax of the GPU's logits).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_11_gb300 import api, binding as B_, workloads as W

from paritylib import record

pytestmark = pytest.mark.gpu

LM_REL = 1e-4
LM_BAND = 1e-4
LM_GAP = 1e-3


def _run(batch, dev, T):
    h = batch.hidden.to(dev)
    w = batch.w_vocab_t.to(dev)
    q = batch.q.to(dev) if T > 0 else None
    u = batch.uniforms.to(dev) if T > 0 else None
    out, al, dg = api.lmhead_verify(h, w, q, batch.draft.to(dev), u, batch.K, T, diag=T > 0)
    torch.cuda.synchronize()
    return out.cpu().numpy(), al.cpu().numpy(), (dg.cpu().numpy() if dg is not None else None)


def _compare(name, batch, T, dev):
    out, al, dg = _run(batch, dev, T)
    orc = oracle.lmhead_verify(batch.hidden, batch.w_vocab_t, batch.q, batch.draft, batch.uniforms,
                               batch.B, batch.K, T, tie_band=LM_BAND)
    K1 = batch.K + 1
    mism, tie_mism, ties = [], 0, 0
    z = orc["logits"]
    for b in range(batch.B):
        sl = slice(b * K1, (b + 1) * K1)
        if T == 0:
            top2 = np.sort(z[sl], axis=1)[:, -2:]
            tie = bool(np.any(top2[:, 1] - top2[:, 0] < LM_GAP))
        else:
            tie = orc["near_tie_accept"][b] > 0 or orc["near_tie_sample"][b] > 0
        ties += int(tie)
        same = al[b] == orc["accept_len"][b] and np.array_equal(out[sl], orc["out_tokens"][sl])
        if not same:
            if tie:
                tie_mism += 1
            else:
                mism.append(b)
    info = {"requests": batch.B, "mismatch": len(mism), "near_ties": ties, "near_tie_mismatch": tie_mism,
            "mean_al": float(al.mean())}
    if T > 0:
        nd = batch.rows - batch.B
        po = orc["p_draft"]
        ev = ~np.isnan(po)
        rel = np.abs(dg[:nd][ev] - po[ev]) / np.maximum(po[ev], 1e-30)
        info["p_max_rel_err"] = float(rel.max()) if rel.size else 0.0
        assert info["p_max_rel_err"] <= LM_REL, name
        Rg = dg[nd::2][: batch.B]
        ok = np.array([al[b] == orc["accept_len"][b] and np.array_equal(out[b * K1:(b + 1) * K1],
                                                                          orc["out_tokens"][b * K1:(b + 1) * K1])
                       for b in range(batch.B)])
        relR = np.abs(Rg[ok] - orc["residual_mass"][ok]) / np.maximum(orc["residual_mass"][ok], 1e-30)
        info["R_max_rel_err"] = float(relR.max()) if relR.size else 0.0
        assert info["R_max_rel_err"] <= LM_REL + 4e-7 / np.maximum(orc["residual_mass"][ok], 1e-30).min()
    record(name, info)
    assert not mism, f"{name}: requests {mism[:5]} differ without a near tie"
    assert tie_mism <= max(1, batch.B // 10)


def test_lmhead_small_sampling(cuda_device):
    b = W.lmhead_small()
    _compare("lmhead B=4 K=3 d=512 V=4000 T=1", b, 1.0, cuda_device)


@pytest.fixture(scope="module")
def m128_batch():
    return W.lmhead(seed=3303, B=16, K=7, d=1024, V=20000, d_draft=256, T=0.8)


def test_lmhead_m128_sampling(cuda_device, m128_batch):
    _compare("lmhead B=16 K=7 d=1024 V=20000 T=0.8", m128_batch, 0.8, cuda_device)


def test_lmhead_m128_greedy(cuda_device, m128_batch):
    _compare("lmhead greedy B=16 K=7 d=1024 V=20000", m128_batch, 0.0, cuda_device)


def test_lmhead_full_workload(cuda_device):
    b = W.lmhead()
    _compare("lmhead B=16 K=7 d=8192 V=128256 T=1", b, 1.0, cuda_device)


def _lm_status(dev):
    ws = api._default_ws[(str(dev), torch.cuda.current_stream(dev).cuda_stream)].buf
    return B_.spec_verify_last_device_status(ws)


def test_lmhead_k_zero_is_bonus_only(cuda_device):
    """Plain decoding through the same call: one row per request, the token
    drawn from p."""
    b = W.lmhead(seed=3311, B=12, K=0, d=512, V=6000, d_draft=256)
    _compare("lmhead K=0 B=12 d=512 V=6000 T=1", b, 1.0, cuda_device)


def test_lmhead_vocab_not_multiple_of_4(cuda_device):
    """Element-wise logits copy in the GEMM epilogue and the two-kernel finish."""
    b = W.lmhead(seed=3313, B=5, K=3, d=512, V=4001, d_draft=256, T=0.9)
    _compare("lmhead B=5 K=3 d=512 V=4001 T=0.9", b, 0.9, cuda_device)


@pytest.fixture(scope="module")
def wide_batch():
    return W.lmhead(seed=3315, B=4, K=3, d=256, V=300000, d_draft=256, T=1.0)


def test_lmhead_vocab_past_the_cluster_finish(cuda_device, wide_batch):
    """V = 300000 is past the largest vocabulary the one-cluster-per-request
    finish takes (8 CTAs x 96 segments x 256 tokens = 196608): the GEMM runs
    ~9 tiles per CTA and the call finishes with the decide and residual
    kernels over the logits copy (three launches in all)."""
    _compare("lmhead wide B=4 K=3 d=256 V=300000 T=1", wide_batch, 1.0, cuda_device)
    assert B_.spec_last_launch_count() == 3


def test_lmhead_vocab_past_the_cluster_finish_greedy(cuda_device, wide_batch):
    _compare("lmhead wide greedy B=4 K=3 d=256 V=300000", wide_batch, 0.0, cuda_device)
    assert B_.spec_last_launch_count() == 2


def test_lmhead_zero_residual_falls_back_to_p(cuda_device):
    """q >= p everywhere: every residual is empty, so the token is drawn from
    p and the call flags it."""
    b = W.lmhead(seed=3312, B=6, K=3, d=512, V=8192, d_draft=256)
    b = dataclasses.replace(b, q=torch.ones_like(b.q))
    _lm_status(cuda_device)  # clears the status word
    _compare("lmhead zero residual B=6 K=3 d=512 V=8192", b, 1.0, cuda_device)
    st, flags = _lm_status(cuda_device)
    assert st == B_.SV_OK and flags & B_.SV_FLAG_ZERO_RESIDUAL


def test_lmhead_residual_at_one_token_forces_it(cuda_device):
    """q = 1 except q(t) = 0 for one token t per request: the draft is
    rejected (u q(x) > p(x)) and r > 0 at t alone, so the token drawn is t
    whatever u is.  The targets sit in different slices of the finish
    cluster, on both sides of a slice boundary and in the ragged last
    segment."""
    V = 20000
    targets = [5, 2559, 2560, 7777, 12345, 17999, 19968, 19999]
    b = W.lmhead(seed=3314, B=len(targets), K=1, d=512, V=V, d_draft=256)
    q = torch.ones_like(b.q)
    for i, t in enumerate(targets):
        q[i, t] = 0.0
    b = dataclasses.replace(b, q=q)
    out, al, _ = _run(b, cuda_device, 1.0)
    for i, t in enumerate(targets):
        if int(b.draft[i]) != t:
            assert al[i] == 1 and out[2 * i] == t, (i, t, al[i], out[2 * i])
    _compare("lmhead one-token residual B=8 K=1 d=512 V=20000", b, 1.0, cuda_device)


def test_lmhead_argument_errors(cuda_device):
    dev = cuda_device
    h = torch.zeros(16, 100, dtype=torch.bfloat16, device=dev)  # d not a multiple of 64
    w = torch.zeros(300, 100, dtype=torch.bfloat16, device=dev)
    x = torch.zeros(12, dtype=torch.int32, device=dev)
    with pytest.raises(B_.SpecVerifyError) as e:
        api.lmhead_verify(h, w, None, x, None, 3, 0.0)
    assert e.value.status == B_.SV_ERR_INVALID
    h = torch.zeros(160, 128, dtype=torch.bfloat16, device=dev)  # M = 160 > 128
    w = torch.zeros(300, 128, dtype=torch.bfloat16, device=dev)
    x = torch.zeros(128, dtype=torch.int32, device=dev)
    with pytest.raises(B_.SpecVerifyError) as e:
        api.lmhead_verify(h, w, None, x, None, 4, 0.0)
    assert e.value.status == B_.SV_ERR_INVALID
