"""The allocation-free sampling entry point, spec_verify_sample_noalloc.

Some callers of this library cannot allocate device memory: a plugin loaded
into an inference server whose device memory is all held by the server's
caching allocator, or a loop that must not call cudaMalloc because it can
synchronise the whole device.  They still own their inputs and outputs, and
this entry point gives them the sampling verification with scratch taken from
a fixed array inside the library instead of a caller-provided workspace.

These tests call it through the C ABI and check that it gives what
spec_verify_sample gives with a workspace of its own, within the tolerance
the parity tests use (token ids and accepted lengths exactly, diagnostics
within 1e-5 relative): twice in a row on one shape, and over a sequence of
shapes that take every kernel path in turn, so that each call finds the
shared scratch as a call of another shape left it.  The file is collected
last so that a run stopping at its first failure has already run every other
test.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from speculative_decoding_verification_11_gb300 import binding as B_, build, workloads as W

pytestmark = pytest.mark.gpu


def _with_workspace(dev, logits, q, x, u, B, K, V, T):
    rows = B * (K + 1)
    out = torch.full((rows,), -9, dtype=torch.int32, device=dev)
    al = torch.full((B,), -9, dtype=torch.int32, device=dev)
    dg = torch.full((rows + B,), float("nan"), device=dev)
    ws = B_.workspace(B_.spec_verify_workspace_size(B, rows, V), dev)
    B_.spec_verify_sample(logits, q, B, K, V, T, x, u, out, al, ws, diag=dg)
    return out, al, dg, B_.spec_last_kernel()


def _noalloc(ref_out, ref_al, ref_dg, logits, q, x, u, B, K, V, T):
    out = torch.full_like(ref_out, -9)
    al = torch.full_like(ref_al, -9)
    dg = torch.full_like(ref_dg, float("nan"))
    B_.spec_verify_sample_noalloc(logits, q, B, K, V, T, x, u, out, al, diag=dg)
    return out, al, dg, B_.spec_last_kernel()


def _check_same(got, ref):
    out, al, dg, _ = got
    ref_out, ref_al, ref_dg, _ = ref
    assert torch.equal(out, ref_out)
    assert torch.equal(al, ref_al)
    torch.testing.assert_close(dg, ref_dg, rtol=1e-5, atol=0.0, equal_nan=True)


@pytest.mark.parametrize("which", ["sampling B=64 K=4 V=128256", "small B=9 K=3 V=10007"])
def test_noalloc_matches_the_workspace_entry_point_twice(cuda_device, which):
    build.build()
    dev = cuda_device
    if which.startswith("sampling"):
        b = W.sampling()
    else:
        b = W.make_sampling_batch("noalloc", 31, B=9, K=3, V=10007, T=1.0, logit_sigma=2.0, noise_sigma=1.0)
    B, K, V, T = b.B, b.K, b.V, b.temperature
    logits, q, x, u = b.logits.to(dev), b.q.to(dev), b.draft.to(dev), b.uniforms.to(dev)
    ref = _with_workspace(dev, logits, q, x, u, B, K, V, T)
    for _ in range(2):
        got = _noalloc(*ref[:3], logits, q, x, u, B, K, V, T)
        torch.cuda.synchronize()
        _check_same(got, ref)
        assert got[3] == ref[3]


# (B, K, V, logits dtype, kernel path the call takes)
SEQUENCE = [
    (64, 4, 128256, torch.float32, "stream"),
    (9, 3, 1024, torch.float32, "small"),
    (8, 4, 32000, torch.bfloat16, "cluster"),
    (40, 6, 50000, torch.bfloat16, "stream"),
    (9, 3, 10007, torch.float32, "scalar"),
    (200, 2, 4096, torch.bfloat16, "small"),
]


def test_noalloc_over_a_sequence_of_shapes_and_paths(cuda_device):
    """Calls of different shapes, logits types and kernel paths one after
    another on the one scratch array, the whole sequence twice: each call
    matches spec_verify_sample with its own workspace, takes the same kernel
    path, and the calls leave the device's free memory unchanged (nothing is
    allocated)."""
    build.build()
    dev = cuda_device
    cases = []
    for i, (B, K, V, dt, path) in enumerate(SEQUENCE):
        b = W.make_sampling_batch("noalloc-seq", 40 + i, B=B, K=K, V=V, T=0.8, logit_sigma=2.0,
                                  noise_sigma=1.0)
        logits = b.logits.to(dt).to(dev)
        args = (logits, b.q.to(dev), b.draft.to(dev), b.uniforms.to(dev), B, K, V, b.temperature)
        ref = _with_workspace(dev, *args)
        assert ref[3] == path, (B, K, V, dt, ref[3])
        cases.append((args, ref))
    # the first call on the device looks up the scratch address (and may load the module)
    _noalloc(*cases[0][1][:3], *cases[0][0])
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info(dev)[0]
    for _ in range(2):
        for args, ref in cases:
            got = _noalloc(*ref[:3], *args)
            torch.cuda.synchronize()
            _check_same(got, ref)
            assert got[3] == ref[3]
    assert torch.cuda.mem_get_info(dev)[0] == free_before


def test_noalloc_refuses_calls_beyond_its_scratch(cuda_device):
    """A call that would need more than the fixed scratch is refused on the host
    (SV_ERR_WORKSPACE) before any launch; the pointers are never touched."""
    lib = B_.load()
    B, K, V = 20000, 4, 128256
    assert B_.spec_verify_workspace_size(B, B * (K + 1), V) > B_.NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x1000)
    st = lib.spec_verify_sample_noalloc(fake, B_.SV_F32, fake, B, K, V, 1.0, fake, fake, fake, fake, None,
                                        None)
    assert st == B_.SV_ERR_WORKSPACE
