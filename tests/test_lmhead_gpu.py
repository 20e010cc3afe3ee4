"""GPU parity of the fused LM-head front end (tcgen05 GEMM + verifier) against
the fp64 oracle (fp64 GEMM of the bf16 operands, then the same steps).

The GPU's logits come from an fp32 accumulation on the tensor cores, so they
differ from the fp64 GEMM by a rounding error.  The parity rule is the
verifier's, with every band derived from an a-priori bound beta on that error
(oracle/gemm_bound.py, computed from the operands alone), element by element:
  p_j(x_j)   within e_p(x_j) = exp(b_x + L)(1 + 1e-5) - 1 relative (b = beta/T,
             L = log sum_w p_w exp(b_w): the log-normaliser's largest move);
  R          within E = sum_w e_p(w) p_w (+ the logits-in rule's 4e-7 for fp32
             cancellation in p - q) of the selected row;
  near ties  the oracle widens its accept band by e_p(x) p/q and its draw band
             by 2E/(R - E) for the row it draws from;
  greedy     tokens identical except requests where, at a position the oracle
             evaluated, some v != argmax has z_argmax - z_v <= beta_argmax + beta_v
             (only there can the fp32 product order the two differently).
The measured error / bound ratios are reported.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle import gemm_bound as G
from speculative_decoding_verification_11_gb300 import api, binding as B_, workloads as W

from paritylib import compare_greedy, compare_sampling, record

pytestmark = pytest.mark.gpu


def _run(batch, dev, T):
    h = batch.hidden.to(dev)
    w = batch.w_vocab_t.to(dev)
    q = batch.q.to(dev) if T > 0 else None
    u = batch.uniforms.to(dev) if T > 0 else None
    out, al, dg = api.lmhead_verify(h, w, q, batch.draft.to(dev), u, batch.K, T, diag=T > 0)
    torch.cuda.synchronize()
    return out.cpu().numpy(), al.cpu().numpy(), (dg.cpu().numpy() if dg is not None else None)


def _compare(name, batch, T, dev, bands=None):
    out, al, dg = _run(batch, dev, T)
    if bands is None or bands.T != T:
        bands = G.bands(batch.hidden, batch.w_vocab_t, T)
    orc = oracle.lmhead_verify(batch.hidden, batch.w_vocab_t, batch.q, batch.draft, batch.uniforms,
                               batch.B, batch.K, T, bands=bands)
    K1 = batch.K + 1
    mism, tie_mism, ties = [], 0, 0
    flip = G.greedy_flip_possible(bands.logits, bands.beta) if T == 0 else None
    for b in range(batch.B):
        sl = slice(b * K1, (b + 1) * K1)
        if T == 0:
            n_eval = max(int(orc["accept_len"][b]), 1)   # positions 0..k* decide the output
            tie = bool(flip[b * K1:b * K1 + n_eval].any())
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
            "mean_al": float(al.mean()), "median_beta": float(np.median(bands.beta))}
    if T > 0:
        nd = batch.rows - batch.B
        po = orc["p_draft"]
        ev = ~np.isnan(po)
        tol = bands.p_rel_err_at(batch.draft, batch.B, batch.K)
        rel = np.abs(dg[:nd][ev] - po[ev]) / np.maximum(po[ev], 1e-30)
        info["p_max_rel_err"] = float(rel.max()) if rel.size else 0.0
        info["p_err_over_bound"] = float((rel / tol[ev]).max()) if rel.size else 0.0
        assert info["p_err_over_bound"] <= 1.0, name
        Rg = dg[nd::2][: batch.B]
        ok = np.array([al[b] == orc["accept_len"][b] and np.array_equal(out[b * K1:(b + 1) * K1],
                                                                          orc["out_tokens"][b * K1:(b + 1) * K1])
                       for b in range(batch.B)])
        sel = np.arange(batch.B) * K1 + np.maximum(orc["accept_len"], 1) - 1   # the row each draw used
        allow = bands.mass_err[sel] + 4e-7
        errR = np.abs(Rg - orc["residual_mass"])
        info["R_err_over_bound"] = float((errR[ok] / allow[ok]).max()) if ok.any() else 0.0
        assert info["R_err_over_bound"] <= 1.0, name
    record(name, info)
    assert not mism, f"{name}: requests {mism[:5]} differ without a near tie"
    assert tie_mism <= max(1, batch.B // 10)


_MODEL_CASES = {}


def _model_case(which):
    """(batch, the accumulation model's fp32 logits of it), built once per case."""
    if which not in _MODEL_CASES:
        b = {"small": lambda: W.lmhead_small(),
             "k0": lambda: W.lmhead(seed=3311, B=12, K=0, d=512, V=6000, d_draft=256),
             "v4001": lambda: W.lmhead(seed=3313, B=5, K=3, d=512, V=4001, d_draft=256, T=0.9),
             "b16_v20000": lambda: W.lmhead(seed=3317, B=16, K=3, d=256, V=20000, d_draft=256)}[which]()
        _MODEL_CASES[which] = (b, G.emulate(b.hidden, b.w_vocab_t).astype(np.float32))
    return _MODEL_CASES[which]


def _compare_model_logits(name, batch, z32, T, dev):
    """The strict rule: the oracle verifies the accumulation model's fp32
    logits (bit-identical to the GEMM's, tests/test_lmhead_logits_gpu.py) with
    the logits-in parity rule (p within 1e-5, near ties within 1e-6)."""
    out, al, dg = _run(batch, dev, T)
    if T == 0:
        orc = oracle.verify_fixed(z32, None, batch.draft, None, batch.B, batch.K, 1.0, greedy=True)
        compare_greedy(name, batch.row_offsets, out, al, orc)
    else:
        orc = oracle.verify_fixed(z32, batch.q, batch.draft, batch.uniforms, batch.B, batch.K, T)
        compare_sampling(name, batch.row_offsets, out, al, dg, orc)


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


def test_lmhead_full_workload(cuda_device, lmhead_full):
    b, bands = lmhead_full
    _compare("lmhead B=16 K=7 d=8192 V=128256 T=1", b, 1.0, cuda_device, bands)


def test_lmhead_full_workload_greedy(cuda_device, lmhead_full):
    b, bands = lmhead_full
    _compare("lmhead greedy B=16 K=7 d=8192 V=128256", b, 0.0, cuda_device,
             dataclasses.replace(bands, T=0.0, e_p=None, mass_err=None))


@pytest.mark.parametrize("which", ["small", "k0", "v4001", "b16_v20000"])
@pytest.mark.parametrize("T", [1.0, 0.0])
def test_lmhead_on_model_logits_strict(cuda_device, which, T):
    """Small fused batches, every decision compared under the logits-in rule
    with the oracle run on the accumulation model's logits."""
    b, z32 = _model_case(which)
    _compare_model_logits(f"lmhead on model logits {which} B={b.B} K={b.K} V={b.V} T={T}", b, z32, T, cuda_device)


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
