"""GPU parity of the paged KV-cache bookkeeping (spec_kv_reserve /
spec_kv_rollback) against the oracle (oracle/kv_blocks.py): integer work, so
every table entry, length, free-list slot and the free count must be equal.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import kv_blocks as kv
from speculative_decoding_verification_11_gb300 import api, binding as B_, workloads as W

from test_oracle_pins_kv import _state

pytestmark = pytest.mark.gpu


def _to(dev, *arrays):
    return [torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in arrays]


def _run(dev, bt, seq, free, fc, K, al, bs):
    """reserve(K) then rollback(K, al) on the GPU; returns host copies after each call and the status."""
    g_bt, g_seq, g_free, g_K, g_al = _to(dev, bt, seq, free, K.astype(np.int32), al.astype(np.int32))
    g_fc = torch.tensor([fc], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B_.spec_kv_reserve(g_bt, g_seq, g_free, g_fc, g_K, bs, st)
    torch.cuda.synchronize()
    after_reserve = (g_bt.cpu().numpy(), int(g_fc.item()), int(st.item()))
    B_.spec_kv_rollback(g_bt, g_seq, g_free, g_fc, g_K, g_al, bs, st)
    torch.cuda.synchronize()
    return after_reserve, (g_bt.cpu().numpy(), g_seq.cpu().numpy(), g_free.cpu().numpy(), int(g_fc.item()),
                           int(st.item()))


@pytest.mark.parametrize("B,max_blocks,bs,kmax", [(64, 40, 16, 8), (7, 9, 1, 6), (300, 12, 3, 20),
                                                  (2500, 6, 32, 64), (4096, 264, 16, 4)])
def test_reserve_and_rollback_match_oracle(cuda_device, B, max_blocks, bs, kmax):
    rng = np.random.default_rng(B + bs)
    bt, seq, free, fc = _state(rng, B, max_blocks, bs, fill=0.55)
    K = np.minimum(rng.integers(0, kmax + 1, size=B), max_blocks * bs - seq).astype(np.int32)
    al = np.array([rng.integers(0, k + 2) for k in K], dtype=np.int32)
    (g_bt1, g_fc1, st1), (g_bt2, g_seq2, g_free2, g_fc2, st2) = _run(cuda_device, bt, seq, free, fc, K, al, bs)
    o_bt1, o_fc1, o_st1 = kv.reserve(bt, seq, free, fc, K, bs)
    assert o_st1 == kv.OK and st1 == 0
    assert np.array_equal(g_bt1, o_bt1) and g_fc1 == o_fc1
    o_bt2, o_seq2, o_free2, o_fc2, o_st2 = kv.rollback(o_bt1, seq, free, o_fc1, K, al, bs)
    assert o_st2 == kv.OK and st2 == 0
    assert np.array_equal(g_bt2, o_bt2) and np.array_equal(g_seq2, o_seq2) and g_fc2 == o_fc2
    assert np.array_equal(g_free2[:g_fc2], o_free2[:o_fc2])


def test_out_of_blocks_changes_nothing(cuda_device):
    dev = cuda_device
    rng = np.random.default_rng(3)
    bt, seq, free, fc = _state(rng, 50, 10, 4, n_ids=50 * 10)
    K = np.full(50, 30, dtype=np.int32)
    K = np.minimum(K, 40 - seq).astype(np.int32)
    small_fc = 3
    g_bt, g_seq, g_free, g_K = _to(dev, bt, seq, free, K)
    g_fc = torch.tensor([small_fc], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B_.spec_kv_reserve(g_bt, g_seq, g_free, g_fc, g_K, 4, st)
    torch.cuda.synchronize()
    assert kv.reserve(bt, seq, free, small_fc, K, 4)[2] == kv.OUT_OF_BLOCKS
    assert st.item() & B_.SV_FLAG_KV_OUT_OF_BLOCKS
    assert np.array_equal(g_bt.cpu().numpy(), bt) and g_fc.item() == small_fc


def test_bad_inputs_change_nothing(cuda_device):
    dev = cuda_device
    bs = 4
    bt = np.array([[1, -1], [2, -1]], dtype=np.int32)
    seq = np.array([3, 4], dtype=np.int32)
    free = np.array([5, 6, 7, -1], dtype=np.int32)
    cases = [("reserve", np.array([9, 0]), None), ("reserve", np.array([-1, 0]), None),
             ("rollback", np.array([1, 0]), np.array([3, 1])), ("rollback", np.array([3, 0]), np.array([1, 1]))]
    for kind, K, al in cases:
        g_bt, g_seq, g_free, g_K = _to(dev, bt, seq, free, K.astype(np.int32))
        g_fc = torch.tensor([3], dtype=torch.int32, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        if kind == "reserve":
            B_.spec_kv_reserve(g_bt, g_seq, g_free, g_fc, g_K, bs, st)
            orc = kv.reserve(bt, seq, free, 3, K, bs)[2]
        else:
            g_al = _to(dev, al.astype(np.int32))[0]
            B_.spec_kv_rollback(g_bt, g_seq, g_free, g_fc, g_K, g_al, bs, st)
            orc = kv.rollback(bt, seq, free, 3, K, al, bs)[4]
        torch.cuda.synchronize()
        assert orc == kv.BAD_INPUT
        assert st.item() & B_.SV_FLAG_KV_BAD_INPUT, (kind, K, al)
        assert np.array_equal(g_bt.cpu().numpy(), bt) and np.array_equal(g_seq.cpu().numpy(), seq)
        assert g_fc.item() == 3 and np.array_equal(g_free.cpu().numpy(), free)


def test_rollback_after_verification_on_device(cuda_device):
    """The verification's accept lengths feed the rollback without leaving the GPU."""
    dev = cuda_device
    b = W.make_sampling_batch("kvpipe", 55, B=48, K=6, V=5000, T=1.0, logit_sigma=2.0, noise_sigma=1.0)
    bs, max_blocks = 8, 20
    rng = np.random.default_rng(9)
    bt, seq, free, fc = _state(rng, b.B, max_blocks, bs, fill=0.5)
    K = np.full(b.B, b.K, dtype=np.int32)
    g_bt, g_seq, g_free, g_K = _to(dev, bt, seq, free, K)
    g_fc = torch.tensor([fc], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B_.spec_kv_reserve(g_bt, g_seq, g_free, g_fc, g_K, bs, st)
    out, al, _ = api.verify_sample(b.logits.to(dev), b.q.to(dev), b.draft.to(dev), b.uniforms.to(dev), b.K,
                                   b.temperature)
    B_.spec_kv_rollback(g_bt, g_seq, g_free, g_fc, g_K, al, bs, st)
    torch.cuda.synchronize()
    al_h = al.cpu().numpy()
    o_bt1, o_fc1, _ = kv.reserve(bt, seq, free, fc, K, bs)
    o_bt2, o_seq2, o_free2, o_fc2, o_st = kv.rollback(o_bt1, seq, free, o_fc1, K, al_h, bs)
    assert o_st == kv.OK and st.item() == 0
    assert np.array_equal(g_bt.cpu().numpy(), o_bt2) and np.array_equal(g_seq.cpu().numpy(), o_seq2)
    assert g_fc.item() == o_fc2 and np.array_equal(g_free.cpu().numpy()[:o_fc2], o_free2[:o_fc2])
    assert np.array_equal(g_seq.cpu().numpy(), seq + al_h - 1)
