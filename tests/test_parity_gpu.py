"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
identical seeded inputs, at the full workload sizes and at small shapes that
span several chunks/tiles with ragged tails, plus the edge cases."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_11_gb300 import api, binding as B_, workloads as W

from paritylib import compare_greedy, compare_sampling, record

pytestmark = pytest.mark.gpu


def _oracle(batch, temperature=None):
    T = batch.temperature if temperature is None else temperature
    greedy = T == 0
    return oracle.verify(batch.logits, batch.q, batch.draft, batch.uniforms, batch.row_offsets,
                         T if not greedy else 1.0, greedy=greedy)


def _gpu_fixed(batch, dev, diag=True):
    logits = batch.logits.to(dev)
    draft = batch.draft.to(dev)
    if batch.temperature == 0:
        out, al = api.verify_greedy(logits, draft, batch.K)
        torch.cuda.synchronize()
        return out.cpu().numpy(), al.cpu().numpy(), None
    out, al, dg = api.verify_sample(logits, batch.q.to(dev), draft, batch.uniforms.to(dev), batch.K,
                                    batch.temperature, diag=diag)
    torch.cuda.synchronize()
    return out.cpu().numpy(), al.cpu().numpy(), (dg.cpu().numpy() if dg is not None else None)


def _gpu_ragged(batch, dev, T=None, diag=True):
    T = batch.temperature if T is None else T
    q = batch.q.to(dev) if batch.q is not None else None
    u = batch.uniforms.to(dev) if batch.uniforms is not None else None
    out, al, dg = api.verify_ragged(batch.logits.to(dev), q, batch.row_offsets.to(dev),
                                    batch.draft.to(dev), u, T, diag=diag and T > 0)
    torch.cuda.synchronize()
    return out.cpu().numpy(), al.cpu().numpy(), (dg.cpu().numpy() if dg is not None else None)


@pytest.fixture(params=["small", "stream", "cluster"])
def kernel(request, cuda_device):
    """Runs a test on each kernel: "small" raises the request-per-CTA kernel's
    limit to 192 KB of logits per request (so that every shape that fits its
    shared memory takes it), "stream" sends every call to the persistent
    streaming kernel, "cluster" lets every shape the cluster-per-request
    kernel takes run on it (the others stream)."""
    prev = B_.spec_set_small_kernel_limit(192 * 1024 if request.param == "small" else 0)
    prev_c = B_.spec_set_cluster_kernel(request.param != "stream")
    yield request.param
    B_.spec_set_small_kernel_limit(prev)
    B_.spec_set_cluster_kernel(prev_c)


def _status(dev):
    ws = api._default_ws[(str(dev), torch.cuda.current_stream(dev).cuda_stream)].buf
    return B_.spec_verify_last_device_status(ws)


# --------------------------------------------------------------------------
# the five workloads at full size
# --------------------------------------------------------------------------
def test_greedy_workload_bit_exact(cuda_device):
    b = W.greedy()
    out, al, _ = _gpu_fixed(b, cuda_device)
    compare_greedy("greedy B=32 K=5 V=32000 bf16", b.row_offsets, out, al, _oracle(b))
    assert _status(cuda_device) == (B_.SV_OK, 0)


def test_tiny_workload_batched(cuda_device):
    b = W.tiny()
    out, al, dg = _gpu_fixed(b, cuda_device)
    compare_sampling("tiny B=1x1000 K=4 V=1024", b.row_offsets, out, al, dg, _oracle(b))


def test_tiny_workload_as_single_calls(cuda_device):
    """The 1000 independent steps as B=1 calls give the batched results."""
    b = W.tiny()
    dev = cuda_device
    logits, q, x, u = b.logits.to(dev), b.q.to(dev), b.draft.to(dev), b.uniforms.to(dev)
    outs, als = [], []
    for s in range(100):
        o, a, _ = api.verify_sample(logits[5 * s:5 * s + 5], q[4 * s:4 * s + 4], x[4 * s:4 * s + 4],
                                    u[5 * s:5 * s + 5], 4, 1.0)
        outs.append(o)
        als.append(a)
    torch.cuda.synchronize()
    o_all, a_all, _ = api.verify_sample(logits[:500], q[:400], x[:400], u[:500], 4, 1.0)
    assert torch.equal(torch.cat(outs), o_all) and torch.equal(torch.cat(als), a_all)


def test_sampling_workload_full(cuda_device):
    b = W.sampling()
    out, al, dg = _gpu_fixed(b, cuda_device)
    compare_sampling("sampling B=64 K=4 V=128256 T=0.7", b.row_offsets, out, al, dg, _oracle(b))
    st, flags = _status(cuda_device)
    assert st == B_.SV_OK and flags & ~B_.SV_FLAG_ZERO_RESIDUAL == 0


@pytest.fixture(scope="module")
def ragged_batch():
    return W.ragged()


def test_ragged_workload_full(cuda_device, ragged_batch):
    b = ragged_batch
    out, al, dg = _gpu_ragged(b, cuda_device)
    compare_sampling("ragged B=256 K_i~U{0..8} V=151936", b.row_offsets, out, al, dg, _oracle(b))


def test_ragged_workload_greedy(cuda_device, ragged_batch):
    b = ragged_batch
    out, al, _ = _gpu_ragged(b, cuda_device, T=0.0)
    compare_greedy("ragged greedy B=256 V=151936", b.row_offsets, out, al, _oracle(b, temperature=0.0))


# --------------------------------------------------------------------------
# shapes: several chunks / tiles, ragged tails, vector and scalar paths
# --------------------------------------------------------------------------
def _rand_batch(seed, B, K, V, dtype, T, sigma=2.0, noise=1.0, ties=False):
    g = torch.Generator().manual_seed(seed)
    R = B * (K + 1)
    z = torch.randn(R, V, generator=g) * sigma
    if ties:
        z = torch.round(z * 2) / 2
    z = z.to(dtype)
    ro = W.fixed_offsets(B, K)
    if T == 0:
        idx = W._draft_rows_index(ro)
        noisy = z[idx].float() + torch.randn(len(idx), V, generator=g) * noise
        x = torch.argmax(noisy, 1).to(torch.int32)
        return W.Batch("rand", z, None, x, None, ro, B, K, V, 0.0)
    idx = W._draft_rows_index(ro)
    q = W._softmax_rows_f32(z[idx].float() + torch.randn(len(idx), V, generator=g) * noise, T)
    x = W._draw_from(q, g) if len(idx) else torch.empty(0, dtype=torch.int32)
    u = torch.from_numpy(W.philox_uniforms(seed, R))
    return W.Batch("rand", z, q, x, u, ro, B, K, V, T)


GREEDY_SHAPES = [(1, 3), (7, 2), (1000, 5), (8191, 1), (8192, 4), (16385, 3), (40001, 2), (65536, 0)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V,K", GREEDY_SHAPES)
def test_greedy_shapes_with_ties(cuda_device, kernel, dtype, V, K):
    b = _rand_batch(10 + V + K, B=9, K=K, V=V, dtype=dtype, T=0.0, ties=True)
    out, al, _ = _gpu_fixed(b, cuda_device)
    compare_greedy(f"greedy V={V} K={K} {dtype} {kernel}", b.row_offsets, out, al, _oracle(b))


SAMPLE_SHAPES = [(5, 2, 1.0), (1000, 4, 0.7), (4097, 3, 1.3), (8192, 4, 1.0), (10007, 5, 0.9),
                 (25000, 7, 1.0), (70001, 2, 0.5), (131072, 1, 1.0)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V,K,T", SAMPLE_SHAPES)
def test_sampling_shapes(cuda_device, kernel, dtype, V, K, T):
    b = _rand_batch(100 + V + K, B=24, K=K, V=V, dtype=dtype, T=T)
    out, al, dg = _gpu_fixed(b, cuda_device)
    compare_sampling(f"sample V={V} K={K} T={T} {dtype} {kernel}", b.row_offsets, out, al, dg, _oracle(b))


@pytest.mark.parametrize("dtype,V", [(torch.float32, 100000), (torch.bfloat16, 200000)])
def test_sampling_batch_too_large_to_keep_rows(cuda_device, dtype, V):
    """B x V x element size above a quarter of L2: no logits row is kept in L2
    through the stats stream, and residual claims start during it."""
    b = _rand_batch(77 + V, B=96, K=3, V=V, dtype=dtype, T=1.0)
    out, al, dg = _gpu_fixed(b, cuda_device)
    compare_sampling(f"sample B=96 K=3 V={V} {dtype} (early residual)", b.row_offsets, out, al, dg, _oracle(b))


def test_sampling_k_zero_is_bonus_only(cuda_device, kernel):
    b = _rand_batch(5, B=40, K=0, V=3000, dtype=torch.float32, T=1.0)
    out, al, dg = _gpu_fixed(b, cuda_device)
    assert np.all(al == 1)
    compare_sampling("sample K=0", b.row_offsets, out, al, dg, _oracle(b))


def test_ragged_small_mixed(cuda_device, kernel):
    g = torch.Generator().manual_seed(77)
    ks = [0, 3, 0, 8, 1, 255, 2]
    b = W.make_sampling_batch("r", 77, B=len(ks), K=None, V=3001, T=0.8, logit_sigma=2.0,
                              noise_sigma=0.7, k_list=ks)
    out, al, dg = _gpu_ragged(b, cuda_device)
    compare_sampling("ragged small incl. K=255", b.row_offsets, out, al, dg, _oracle(b))


def test_ragged_small_vocab_long_requests(cuda_device, kernel):
    """V = 40: even a request of 256 rows fits the request-per-CTA kernel."""
    ks = [0, 3, 255, 17, 1, 64, 0]
    b = W.make_sampling_batch("rs", 91, B=len(ks), K=None, V=40, T=1.1, logit_sigma=1.5,
                              noise_sigma=0.6, k_list=ks)
    out, al, dg = _gpu_ragged(b, cuda_device)
    compare_sampling(f"ragged V=40 incl. K=255 {kernel}", b.row_offsets, out, al, dg, _oracle(b))
    out, al, _ = _gpu_ragged(b, cuda_device, T=0.0)
    compare_greedy(f"ragged greedy V=40 incl. K=255 {kernel}", b.row_offsets, out, al, _oracle(b, temperature=0.0))


# --------------------------------------------------------------------------
# special cases and errors
# --------------------------------------------------------------------------
def test_q_equals_p_accepts_everything(cuda_device, kernel):
    B, K, V, T = 64, 4, 5000, 0.9
    g = torch.Generator().manual_seed(8)
    z = torch.randn(B * (K + 1), V, generator=g) * 2
    ro = W.fixed_offsets(B, K)
    idx = W._draft_rows_index(ro)
    q = W._softmax_rows_f32(z[idx], T)
    x = W._draw_from(q, g)
    u = torch.from_numpy(W.philox_uniforms(8, B * (K + 1)))
    b = W.Batch("qp", z, q, x, u, ro, B, K, V, T)
    out, al, dg = _gpu_fixed(b, cuda_device)
    orc = _oracle(b)
    full = al == K + 1
    assert np.all(full | (orc["near_tie_accept"] > 0))
    compare_sampling("q == p", b.row_offsets, out, al, dg, orc)


def test_invalid_draft_id_is_isolated(cuda_device, kernel):
    b = _rand_batch(3, B=6, K=3, V=2000, dtype=torch.float32, T=1.0)
    x = b.draft.clone()
    x[5] = 2000  # request 1, position 2
    x[13] = -4   # request 4, position 1
    b.draft = x
    out, al, dg = _gpu_fixed(b, cuda_device)
    orc = _oracle(b)
    assert orc["invalid"] == 2
    assert al[1] == 0 and al[4] == 0 and np.all(out[4:8] == -1) and np.all(out[16:20] == -1)
    st, flags = _status(cuda_device)
    assert st == B_.SV_ERR_DEVICE_INPUT and flags & B_.SV_FLAG_BAD_TOKEN
    keep = [0, 2, 3, 5]
    assert np.array_equal(al[keep], orc["accept_len"][keep])
    # the status word was cleared by the read
    assert _status(cuda_device) == (B_.SV_OK, 0)


def test_malformed_offsets_invalidate_call(cuda_device, kernel):
    dev = cuda_device
    V = 500
    z = torch.randn(10, V, device=dev)
    q = torch.full((7, V), 1.0 / V, device=dev)
    x = torch.zeros(7, dtype=torch.int32, device=dev)
    u = torch.full((10,), 0.5, device=dev)
    for bad in ([0, 4, 3, 10], [1, 4, 7, 10], [0, 4, 7, 9]):
        ro = torch.tensor(bad, dtype=torch.int32, device=dev)
        out, al, _ = api.verify_ragged(z, q, ro, x, u, 1.0)
        torch.cuda.synchronize()
        assert torch.all(al == 0) and torch.all(out == -1)
        st, flags = _status(dev)
        assert st == B_.SV_ERR_DEVICE_INPUT and flags & B_.SV_FLAG_BAD_OFFSETS
    # a good call right after works (workspace left reusable)
    ro = torch.tensor([0, 4, 7, 10], dtype=torch.int32, device=dev)
    out, al, _ = api.verify_ragged(z, q, ro, x, u, 1.0)
    torch.cuda.synchronize()
    assert torch.all(al >= 1)


def test_zero_residual_falls_back_to_p(cuda_device, kernel):
    dev = cuda_device
    z = torch.log(torch.tensor([[0.5, 0.5], [0.5, 0.5]])).to(dev)
    q = torch.tensor([[0.6, 0.6]], device=dev)
    x = torch.tensor([0], dtype=torch.int32, device=dev)
    u = torch.tensor([0.99, 0.75], device=dev)
    out, al, _ = api.verify_sample(z, q, x, u, 1, 1.0)
    torch.cuda.synchronize()
    assert al.item() == 1 and out[0].item() == 1
    st, flags = _status(dev)
    assert st == B_.SV_OK and flags & B_.SV_FLAG_ZERO_RESIDUAL


def test_empty_batch(cuda_device):
    dev = cuda_device
    z = torch.empty(0, 100, device=dev)
    out, al = api.verify_greedy(z, torch.empty(0, dtype=torch.int32, device=dev), 3)
    assert out.numel() == 0 and al.numel() == 0


def test_repeat_calls_identical_and_canaries(cuda_device, kernel):
    dev = cuda_device
    b = _rand_batch(21, B=16, K=4, V=9000, dtype=torch.float32, T=1.0)
    logits, q, x, u = b.logits.to(dev), b.q.to(dev), b.draft.to(dev), b.uniforms.to(dev)
    R, Bn = b.rows, b.B
    sentinel = -777
    out_buf = torch.full((R + 64,), sentinel, dtype=torch.int32, device=dev)
    al_buf = torch.full((Bn + 64,), sentinel, dtype=torch.int32, device=dev)
    dg_buf = torch.full((R + Bn + 64,), 12345.0, device=dev)
    ws = B_.workspace(B_.spec_verify_workspace_size(Bn, R, b.V) + 4096, dev)
    ws_guard = ws[-4096:]
    ws_guard.fill_(0xA5)
    results = []
    for _ in range(3):
        B_.spec_verify_sample(logits, q, Bn, 4, b.V, 1.0, x, u, out_buf[32:32 + R], al_buf[32:32 + Bn],
                              ws[:-4096], diag=dg_buf[32:32 + R + Bn])
        torch.cuda.synchronize()
        results.append((out_buf.clone(), al_buf.clone()))
    for o, a in results[1:]:
        assert torch.equal(o, results[0][0]) and torch.equal(a, results[0][1])
    assert torch.all(out_buf[:32] == sentinel) and torch.all(out_buf[32 + R:] == sentinel)
    assert torch.all(al_buf[:32] == sentinel) and torch.all(al_buf[32 + Bn:] == sentinel)
    assert torch.all(dg_buf[:32] == 12345.0) and torch.all(dg_buf[32 + R + Bn:] == 12345.0)
    assert torch.all(ws_guard == 0xA5)


# --------------------------------------------------------------------------
# the emitted token's law on the GPU (10^6 trials, V = 16)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("variant", ["near", "onehot", "zeros", "far"])
def test_emitted_token_law_chisquare_gpu(cuda_device, kernel, variant):
    from test_oracle_pins import _chisq_pvalue, _q_variants
    rng = np.random.default_rng(321)
    V, K, T, n = 16, 2, 1.0, 1_000_000
    z = rng.normal(0, 1.0, size=(K + 1, V))
    q = _q_variants(z, rng)[variant]
    draft = np.stack([rng.choice(V, size=n, p=q[j].astype(np.float64) / q[j].astype(np.float64).sum())
                      for j in range(K)], axis=1).astype(np.int32).reshape(-1)
    uni = torch.from_numpy(W.philox_uniforms(4242, n * (K + 1)))
    dev = cuda_device
    logits = torch.from_numpy(z.astype(np.float32)).to(dev).repeat(n, 1)
    qq = torch.from_numpy(q).to(dev).repeat(n, 1)
    out, al, _ = api.verify_sample(logits, qq, torch.from_numpy(draft).to(dev), uni.to(dev), K, T)
    out = out.view(n, K + 1).cpu().numpy()
    al = al.cpu().numpy()
    p = oracle.softmax_rows(z.astype(np.float32), T)
    pv = []
    for j in range(K + 1):
        sel = al > j
        counts = np.bincount(out[sel, j], minlength=V).astype(np.float64)
        pv.append(_chisq_pvalue(counts, p[j]))
    record(f"chi-square GPU {variant} {kernel}", {"pvalues": pv, "trials": n, "mean_al": float(al.mean())})
    assert min(pv) > 1e-3


def test_one_workspace_serves_calls_of_any_shape(cuda_device):
    """A workspace zero-filled once and then used by calls of other shapes
    (it holds their leftovers) gives the same results as a fresh one."""
    dev = cuda_device
    shapes = [(40, 4, 9000), (3, 2, 1000), (64, 7, 20000), (1, 0, 300), (50, 5, 12000)]
    batches = [_rand_batch(300 + i, B=Bn, K=K, V=V, dtype=torch.float32, T=1.0)
               for i, (Bn, K, V) in enumerate(shapes)]
    big = max(B_.spec_verify_workspace_size(b.B, b.rows, b.V) for b in batches)
    shared = B_.workspace(big, dev)
    for rep in range(2):
        for b in batches:
            args = (b.logits.to(dev), b.q.to(dev), b.B, b.K, b.V, 1.0, b.draft.to(dev), b.uniforms.to(dev))
            o1 = torch.empty(b.rows, dtype=torch.int32, device=dev)
            a1 = torch.empty(b.B, dtype=torch.int32, device=dev)
            B_.spec_verify_sample(*args, o1, a1, shared)
            o2 = torch.empty_like(o1)
            a2 = torch.empty_like(a1)
            B_.spec_verify_sample(*args, o2, a2, B_.workspace(B_.spec_verify_workspace_size(b.B, b.rows, b.V), dev))
            torch.cuda.synchronize()
            assert torch.equal(o1, o2) and torch.equal(a1, a2), (rep, b.B, b.K, b.V)


def test_graph_replay_over_rotating_inputs(cuda_device, kernel):
    """Calls captured in one CUDA graph, as the small workloads are timed:
    sampling and greedy calls over different inputs, back to back on one
    workspace.  Two replays give the oracle's results for every call."""
    dev = cuda_device
    samp = [_rand_batch(700 + i, B=12, K=3, V=9000, dtype=torch.float32, T=1.0) for i in range(3)]
    gre = [_rand_batch(710 + i, B=12, K=3, V=9000, dtype=torch.bfloat16, T=0.0) for i in range(2)]
    order = [samp[0], gre[0], samp[1], samp[2], gre[1]]
    ws = B_.workspace(max(B_.spec_verify_workspace_size(b.B, b.rows, b.V) for b in order), dev)
    ins = [(b.logits.to(dev), b.q.to(dev) if b.q is not None else None, b.draft.to(dev),
            b.uniforms.to(dev) if b.uniforms is not None else None) for b in order]
    outs = [(torch.empty(b.rows, dtype=torch.int32, device=dev), torch.empty(b.B, dtype=torch.int32, device=dev))
            for b in order]

    def calls(st):
        for b, (lg, q, x, u), (o, a) in zip(order, ins, outs):
            if b.temperature == 0:
                B_.spec_verify_greedy(lg, x, b.B, b.K, b.V, o, a, ws, stream=st)
            else:
                B_.spec_verify_sample(lg, q, b.B, b.K, b.V, b.temperature, x, u, o, a, ws, stream=st)

    stream = torch.cuda.current_stream(dev)
    calls(stream)  # eager first: the same kernels, and the workspace's state carried into the graph
    torch.cuda.synchronize()
    gs = torch.cuda.Stream(dev)
    gs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        calls(gs)
    orcs = [_oracle(b) for b in order]
    for rep in range(2):
        for o, a in outs:
            o.fill_(-5)
            a.fill_(-5)
        g.replay()
        torch.cuda.synchronize()
        for i, (b, (o, a), orc) in enumerate(zip(order, outs, orcs)):
            name = f"graph replay {rep} call {i} {kernel}"
            if b.temperature == 0:
                compare_greedy(name, b.row_offsets, o.cpu().numpy(), a.cpu().numpy(), orc)
            else:
                compare_sampling(name, b.row_offsets, o.cpu().numpy(), a.cpu().numpy(), None, orc)
    st, flags = B_.spec_verify_last_device_status(ws)
    assert st == B_.SV_OK and flags & ~B_.SV_FLAG_ZERO_RESIDUAL == 0


def test_more_than_2_32_logits_with_planted_maxima(cuda_device):
    """16 bf16 rows of V = 2^28 + 8 logits (4.3e9 elements, past 2^32) and 12
    fp32 q rows (3.2e9 elements, past 2^31), so that every row, gather and
    residual offset past the first rows needs 64-bit indexing.  Each row is 0
    except a planted +100 at t_r, so p is one-hot at t_r in fp32 (the other
    tokens get e^-100 / S < 4e-44) and the results follow by construction:
    drafts equal to t_j with q one-hot there are accepted; a draft elsewhere
    with q one-hot at it is rejected, and its residual max(0, p - q) is
    one-hot at t_j again.  So request b emits t_0 .. t_{a_b} and AL = a_b + 1,
    where a_b is the first position whose draft misses.  Greedy verification
    of the same logits gives the same result."""
    dev = cuda_device
    B, K, V = 4, 3, (1 << 28) + 8
    R, Nq = B * (K + 1), B * K
    miss = [0, 1, 2, K]  # first drafted position that misses t; K: every draft matches (bonus)
    t = [(V - 1 - 1009 * r) if r % 2 else (1000003 * r + 4099) % V for r in range(R)]
    x = []
    for b in range(B):
        for j in range(K):
            tj = t[b * (K + 1) + j]
            x.append(tj if j < miss[b] else (tj + 12345) % V)
    logits = torch.zeros(R, V, dtype=torch.bfloat16, device=dev)
    logits[torch.arange(R, device=dev), torch.tensor(t, device=dev)] = 100.0
    q = torch.zeros(Nq, V, dtype=torch.float32, device=dev)
    q[torch.arange(Nq, device=dev), torch.tensor(x, device=dev)] = 1.0
    draft = torch.tensor(x, dtype=torch.int32, device=dev)
    u = torch.from_numpy(W.philox_uniforms(4321, R)).to(dev)
    exp_out = np.full(R, -1, dtype=np.int32)
    for b in range(B):
        exp_out[b * (K + 1):b * (K + 1) + miss[b] + 1] = t[b * (K + 1):b * (K + 1) + miss[b] + 1]
    exp_al = np.array(miss, dtype=np.int32) + 1
    ws = B_.workspace(B_.spec_verify_workspace_size(B, R, V), dev)
    out = torch.full((R,), -9, dtype=torch.int32, device=dev)
    al = torch.full((B,), -9, dtype=torch.int32, device=dev)
    B_.spec_verify_sample(logits, q, B, K, V, 1.0, draft, u, out, al, ws)
    torch.cuda.synchronize()
    assert B_.spec_last_kernel() == "stream"
    assert np.array_equal(al.cpu().numpy(), exp_al) and np.array_equal(out.cpu().numpy(), exp_out)
    out.fill_(-9)
    al.fill_(-9)
    B_.spec_verify_greedy(logits, draft, B, K, V, out, al, ws)
    torch.cuda.synchronize()
    assert np.array_equal(al.cpu().numpy(), exp_al) and np.array_equal(out.cpu().numpy(), exp_out)
    st, flags = B_.spec_verify_last_device_status(ws)
    assert st == B_.SV_OK and flags == 0
    del logits, q
    torch.cuda.empty_cache()


def test_kernel_choice_follows_the_knobs(cuda_device):
    """The path a call takes, as spec_last_kernel() reports it, follows the
    size rules and the two process-wide knobs; every path gives the oracle's
    result (checked above), so this pins only the dispatch."""
    dev = cuda_device
    prev_s = B_.spec_set_small_kernel_limit(48 * 1024)
    prev_c = B_.spec_set_cluster_kernel(True)
    try:
        def kind(V, K, B, dtype=torch.float32):
            b = _rand_batch(3 + V, B=B, K=K, V=V, dtype=dtype, T=1.0)
            _gpu_fixed(b, dev)
            return B_.spec_last_kernel()

        assert kind(1024, 4, 8) == "small"                 # 20 KB of logits per request
        assert kind(32000, 5, 16) == "cluster"             # 768 KB per request, 16 requests
        assert kind(32000, 5, 64) == "stream"              # 64 x 8 CTAs exceed two per SM
        assert kind(4097, 3, 8) == "scalar"                # rows not 16-byte aligned
        B_.spec_set_cluster_kernel(False)
        assert kind(32000, 5, 16) == "stream"
        B_.spec_set_small_kernel_limit(0)
        assert kind(1024, 4, 8) == "stream"
    finally:
        B_.spec_set_small_kernel_limit(prev_s)
        B_.spec_set_cluster_kernel(prev_c)


@pytest.mark.parametrize("V", [4096, 20000])
def test_empty_residual_on_aligned_rows(cuda_device, kernel, V):
    """q = 1 everywhere: every draft is rejected and every residual is empty,
    so each request draws from p and the call sets the flag; on all paths
    (the cluster kernel's retry included), against the oracle."""
    dev = cuda_device
    b = _rand_batch(900 + V, B=6, K=2, V=V, dtype=torch.float32, T=1.0)
    b = W.Batch(b.name, b.logits, torch.ones_like(b.q), b.draft, b.uniforms, b.row_offsets, b.B, b.K, b.V,
                b.temperature)
    _gpu_fixed(b, dev)
    _status(dev)  # clears the status word of the call's workspace
    out, al, dg = _gpu_fixed(b, dev)
    compare_sampling(f"empty residual V={V} {kernel}", b.row_offsets, out, al, dg, _oracle(b))
    st, flags = _status(dev)
    assert st == B_.SV_OK and flags & B_.SV_FLAG_ZERO_RESIDUAL


def test_residual_at_one_token_is_drawn(cuda_device, kernel):
    """q = 1 except q(t) = 0 at one token t per request: the draft is rejected
    and r > 0 at t alone, so t is drawn whatever the uniform.  The targets lie
    in different slices of the cluster kernel, on both sides of a slice
    boundary (2560 tokens at V = 20000) and in the ragged last segment."""
    dev = cuda_device
    V = 20000
    targets = [5, 2559, 2560, 7777, 12345, 17999, 19968, 19999]
    b = _rand_batch(77, B=len(targets), K=1, V=V, dtype=torch.float32, T=1.0)
    q = torch.ones_like(b.q)
    for i, t in enumerate(targets):
        q[i, t] = 0.0
    b = W.Batch(b.name, b.logits, q, b.draft, b.uniforms, b.row_offsets, b.B, b.K, b.V, b.temperature)
    out, al, dg = _gpu_fixed(b, dev)
    for i, t in enumerate(targets):
        if int(b.draft[i]) != t:
            assert al[i] == 1 and out[2 * i] == t, (kernel, i, t, al[i], out[2 * i])
    compare_sampling(f"one-token residual V={V} {kernel}", b.row_offsets, out, al, dg, _oracle(b))
