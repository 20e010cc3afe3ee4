"""GPU parity of the dynamic-K controller (spec_dynk_update) against the oracle
(oracle/dynk.py): every decision is taken in fp32 in the same order on both
sides, so k_next, the row offsets and the controller state are equal."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import dynk
from speculative_decoding_verification_11_gb300 import api, binding as B_, workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("policy", [dynk.WINDOW, dynk.GOODPUT])
@pytest.mark.parametrize("B,Wn", [(37, 10), (2500, 4), (4096, 10)])
def test_controller_matches_oracle_over_steps(cuda_device, policy, B, Wn):
    dev = cuda_device
    rng = np.random.default_rng(B * 10 + policy)
    k_low, k_high = 1, 7
    itl = (10.0 + 1.7 * np.arange(k_high + 1) + rng.uniform(0, 0.5, k_high + 1)).astype(np.float32)
    hist_o = np.zeros((B, Wn, 2), dtype=np.int32)
    count_o = np.zeros(B, dtype=np.int32)
    hist_g = torch.zeros(B, Wn, 2, dtype=torch.int32, device=dev)
    count_g = torch.zeros(B, dtype=torch.int32, device=dev)
    itl_g = torch.from_numpy(itl).to(dev)
    k_used = np.full(B, k_high, dtype=np.int32)
    alpha = rng.uniform(0.1, 0.95, size=B)
    for step in range(12):
        al = np.array([1 + min(int(rng.geometric(1 - a)) - 1, k) for a, k in zip(alpha, k_used)], dtype=np.int32)
        al[rng.random(B) < 0.03] = 0  # a few invalid requests
        k_o, offs_o = dynk.update(al, k_used, hist_o, count_o, Wn, policy, 1.5, k_low, k_high, itl, 0.5)
        k_g = torch.empty(B, dtype=torch.int32, device=dev)
        offs_g = torch.empty(B + 1, dtype=torch.int32, device=dev)
        B_.spec_dynk_update(torch.from_numpy(al).to(dev), torch.from_numpy(k_used).to(dev), hist_g, count_g, policy,
                            k_low, k_high, k_g, threshold=1.5, itl=itl_g, alpha_prior=0.5, row_offsets=offs_g)
        torch.cuda.synchronize()
        assert np.array_equal(k_g.cpu().numpy(), k_o), step
        assert np.array_equal(offs_g.cpu().numpy(), offs_o), step
        assert np.array_equal(count_g.cpu().numpy(), count_o)
        assert np.array_equal(hist_g.cpu().numpy(), hist_o)
        k_used = k_o


def test_offsets_drive_a_ragged_verification(cuda_device):
    """K_i chosen on the device shape the next ragged verification directly."""
    dev = cuda_device
    B, V = 48, 3000
    al = torch.randint(1, 6, (B,), dtype=torch.int32, device=dev)
    hist = torch.zeros(B, 10, 2, dtype=torch.int32, device=dev)
    count = torch.zeros(B, dtype=torch.int32, device=dev)
    k = torch.empty(B, dtype=torch.int32, device=dev)
    offs = torch.empty(B + 1, dtype=torch.int32, device=dev)
    B_.spec_dynk_update(al, torch.full((B,), 4, dtype=torch.int32, device=dev), hist, count, B_.SV_DYNK_WINDOW, 2,
                        5, k, threshold=2.5, row_offsets=offs)
    torch.cuda.synchronize()
    ks = k.cpu().tolist()
    b = W.make_sampling_batch("dynk", 12, B=B, K=None, V=V, T=1.0, logit_sigma=2.0, noise_sigma=1.0, k_list=ks)
    assert np.array_equal(offs.cpu().numpy(), b.row_offsets.numpy())
    out, acc, _ = api.verify_ragged(b.logits.to(dev), b.q.to(dev), offs, b.draft.to(dev), b.uniforms.to(dev), 1.0)
    torch.cuda.synchronize()
    a = acc.cpu().numpy()
    assert np.all(a >= 1) and np.all(a <= np.array(ks) + 1)


def test_dynk_argument_errors(cuda_device):
    dev = cuda_device
    z = torch.zeros(4, dtype=torch.int32, device=dev)
    h = torch.zeros(4, 3, 2, dtype=torch.int32, device=dev)
    for kl, kh, pol in ((3, 2, 0), (0, 256, 0), (0, 3, 7)):
        with pytest.raises(B_.SpecVerifyError):
            B_.spec_dynk_update(z, z, h, z, pol, kl, kh, z)
    with pytest.raises(B_.SpecVerifyError):  # the goodput rule needs the step-time table
        B_.spec_dynk_update(z, z, h, z, B_.SV_DYNK_GOODPUT, 0, 3, z)
