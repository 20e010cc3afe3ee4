"""Host-side checks of the C ABI (no GPU): the library builds for sm_103a,
loads, exports every entry point the header declares, and rejects bad
arguments before any launch."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from speculative_decoding_verification_11_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_and_binding_agree():
    assert sorted(binding.EXPORTS) == _declared()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(6):
        assert lib.spec_status_string(code)
    assert lib.spec_status_string(99) == b"unknown status"


def test_workspace_size_grows_with_problem(lib):
    small = lib.spec_verify_workspace_size(64, 320, 128256)
    big = lib.spec_verify_workspace_size(256, 1280, 151936)
    assert small % 256 == 0 and big > small
    # partials: one (M, s) pair per 8192-token chunk of every row
    assert small >= 320 * 16 * 8


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails on the host
ALIGNED_WS = ctypes.c_void_p(0x10000)


def test_argument_errors_return_before_launch(lib):
    I = binding
    ws_bytes = 1 << 20
    # K out of range
    assert lib.spec_verify_greedy(FAKE, 0, 4, -1, 100, FAKE, FAKE, FAKE, ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID
    assert lib.spec_verify_greedy(FAKE, 0, 4, 256, 100, FAKE, FAKE, FAKE, ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID
    # bad dtype, bad V, null logits
    assert lib.spec_verify_greedy(FAKE, 7, 4, 2, 100, FAKE, FAKE, FAKE, ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID
    assert lib.spec_verify_greedy(FAKE, 0, 4, 2, 0, FAKE, FAKE, FAKE, ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID
    assert lib.spec_verify_greedy(None, 0, 4, 2, 100, FAKE, FAKE, FAKE, ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID
    # sampling needs T > 0 and finite, uniforms and q
    for T in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.spec_verify_sample(FAKE, 0, FAKE, 4, 2, 100, T, FAKE, FAKE, FAKE, FAKE, None,
                                      ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID
    assert lib.spec_verify_sample(FAKE, 0, None, 4, 2, 100, 1.0, FAKE, FAKE, FAKE, FAKE, None,
                                  ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID
    assert lib.spec_verify_sample(FAKE, 0, FAKE, 4, 2, 100, 1.0, FAKE, None, FAKE, FAKE, None,
                                  ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID
    # ragged: null offsets, negative temperature
    assert lib.spec_verify_ragged(FAKE, 0, FAKE, None, 4, 10, 100, 1.0, FAKE, FAKE, FAKE, FAKE, None,
                                  ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID
    assert lib.spec_verify_ragged(FAKE, 0, FAKE, FAKE, 4, 10, 100, -0.5, FAKE, FAKE, FAKE, FAKE, None,
                                  ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID
    # rows fewer than requests
    assert lib.spec_verify_ragged(FAKE, 0, FAKE, FAKE, 4, 3, 100, 1.0, FAKE, FAKE, FAKE, FAKE, None,
                                  ALIGNED_WS, ws_bytes, None) == I.SV_ERR_INVALID


def test_workspace_errors(lib):
    I = binding
    need = lib.spec_verify_workspace_size(4, 12, 100)
    assert lib.spec_verify_greedy(FAKE, 0, 4, 2, 100, FAKE, FAKE, FAKE, ALIGNED_WS, need - 1, None) == I.SV_ERR_WORKSPACE
    assert lib.spec_verify_greedy(FAKE, 0, 4, 2, 100, FAKE, FAKE, FAKE, ctypes.c_void_p(0x10010), need, None) == I.SV_ERR_WORKSPACE


def test_empty_batch_is_a_no_op(lib):
    assert lib.spec_verify_greedy(FAKE, 0, 0, 3, 100, FAKE, FAKE, FAKE, ALIGNED_WS, 256, None) == binding.SV_OK
    assert lib.spec_lmhead_workspace_size(16, 7, 8192, 128256) >= 128 * 128256 * 4
    assert lib.spec_last_launch_count() == 0


def test_profile_hook_arguments(lib):
    assert lib.spec_profile_set_events(FAKE, None) == binding.SV_ERR_INVALID
    assert lib.spec_profile_set_events(None, None) == binding.SV_OK


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        binding.load()


def test_kv_argument_errors_return_before_launch(lib):
    """Argument errors of the KV-cache calls come back synchronously, with no
    launch (the pointers are never touched)."""
    P = ctypes.c_void_p(0x1000)
    ok_args = dict(B=4, max_blocks=8, bs=16)
    assert lib.spec_kv_reserve(P, P, P, P, P, 4, 0, 16, P, None) == binding.SV_ERR_INVALID   # max_blocks
    assert lib.spec_kv_reserve(P, P, P, P, P, 4, 8, 0, P, None) == binding.SV_ERR_INVALID    # block size
    assert lib.spec_kv_reserve(P, None, P, P, P, 4, 8, 16, P, None) == binding.SV_ERR_INVALID
    assert lib.spec_kv_reserve(P, P, P, P, P, -1, 8, 16, P, None) == binding.SV_ERR_INVALID
    assert lib.spec_kv_reserve(None, None, None, None, None, 0, 8, 16, None, None) == binding.SV_OK  # empty
    assert lib.spec_kv_rollback(P, P, P, P, P, P, 4, 8, 16, -1, P, None) == binding.SV_ERR_INVALID  # capacity
    assert lib.spec_kv_rollback(P, P, P, P, P, None, 4, 8, 16, 10, P, None) == binding.SV_ERR_INVALID
    assert lib.spec_kv_rollback(P, P, P, P, P, P, 4, 8, 16, 10, None, None) == binding.SV_ERR_INVALID
    assert lib.spec_kv_rollback(None, None, None, None, None, None, 0, 8, 16, 0, None, None) == binding.SV_OK
    del ok_args


def test_ngram_refuses_a_misaligned_token_buffer(lib):
    """The n-gram drafter's bulk copies need 4-byte-aligned int32 tokens: a
    pointer off by two bytes is refused before any launch."""
    P = ctypes.c_void_p(0x1000)
    assert lib.spec_ngram_draft(ctypes.c_void_p(0x1002), P, 4, 8, 1, 4, P, P, None) == binding.SV_ERR_INVALID
    assert lib.spec_ngram_draft(P, P, 4, 8, 1, 33, P, P, None) == binding.SV_ERR_INVALID  # n_max


def test_noalloc_scratch_size_matches_the_header():
    """The binding's copy of SV_NOALLOC_SCRATCH_BYTES is the header's value."""
    src = open(HEADER).read()
    m = re.search(r"#define\s+SV_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", src)
    assert m, "SV_NOALLOC_SCRATCH_BYTES not found in the header"
    assert binding.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_noalloc_refuses_bad_arguments_before_touching_its_scratch(lib):
    """Every argument rule of the allocation-free call is checked on the host
    before its scratch is cleared: a refused call enqueues nothing (here no
    CUDA call at all: this machine has no GPU, so reaching one would return
    SV_ERR_CUDA instead of the refusal)."""
    I = binding
    call = lib.spec_verify_sample_noalloc
    # B (K + 1) past INT_MAX: refused, not wrapped to a small or negative count
    assert call(FAKE, 0, FAKE, 1 << 30, 1, 128, 1.0, FAKE, FAKE, FAKE, FAKE, None, None) == I.SV_ERR_INVALID
    assert call(FAKE, 0, FAKE, (1 << 31) - 1, 255, 128, 1.0, FAKE, FAKE, FAKE, FAKE, None, None) == I.SV_ERR_INVALID
    # null logits, outputs, draft, uniforms or q
    assert call(None, 0, FAKE, 4, 2, 100, 1.0, FAKE, FAKE, FAKE, FAKE, None, None) == I.SV_ERR_INVALID
    assert call(FAKE, 0, FAKE, 4, 2, 100, 1.0, FAKE, FAKE, None, FAKE, None, None) == I.SV_ERR_INVALID
    assert call(FAKE, 0, FAKE, 4, 2, 100, 1.0, FAKE, FAKE, FAKE, None, None, None) == I.SV_ERR_INVALID
    assert call(FAKE, 0, FAKE, 4, 2, 100, 1.0, None, FAKE, FAKE, FAKE, None, None) == I.SV_ERR_INVALID
    assert call(FAKE, 0, FAKE, 4, 2, 100, 1.0, FAKE, None, FAKE, FAKE, None, None) == I.SV_ERR_INVALID
    assert call(FAKE, 0, None, 4, 2, 100, 1.0, FAKE, FAKE, FAKE, FAKE, None, None) == I.SV_ERR_INVALID
    # bad dtype, V, K, temperature
    assert call(FAKE, 7, FAKE, 4, 2, 100, 1.0, FAKE, FAKE, FAKE, FAKE, None, None) == I.SV_ERR_INVALID
    assert call(FAKE, 0, FAKE, 4, 2, 0, 1.0, FAKE, FAKE, FAKE, FAKE, None, None) == I.SV_ERR_INVALID
    assert call(FAKE, 0, FAKE, 4, 256, 100, 1.0, FAKE, FAKE, FAKE, FAKE, None, None) == I.SV_ERR_INVALID
    for T in (0.0, -1.0, float("inf"), float("nan")):
        assert call(FAKE, 0, FAKE, 4, 2, 100, T, FAKE, FAKE, FAKE, FAKE, None, None) == I.SV_ERR_INVALID
    # a valid call too large for the scratch: refused as a workspace error
    assert call(FAKE, 0, FAKE, 20000, 4, 128256, 1.0, FAKE, FAKE, FAKE, FAKE, None, None) == I.SV_ERR_WORKSPACE


def test_fixed_k_calls_refuse_row_counts_past_int_max(lib):
    """B (K + 1) is formed in 64 bits: a product past INT_MAX is an argument
    error, not a wrapped row count."""
    I = binding
    ws = ctypes.c_void_p(0x10000)
    assert lib.spec_verify_greedy(FAKE, 0, 1 << 30, 1, 128, FAKE, FAKE, FAKE, ws, 1 << 20, None) == I.SV_ERR_INVALID
    assert lib.spec_verify_sample(FAKE, 0, FAKE, 1 << 30, 3, 128, 1.0, FAKE, FAKE, FAKE, FAKE, None, ws, 1 << 20,
                                  None) == I.SV_ERR_INVALID


def test_wait_budget_knob(lib):
    """spec_set_wait_budget: returns the previous value, 0 restores the default,
    a negative value is refused and changes nothing (host only, no launch)."""
    default = 4000000000
    prev = binding.spec_set_wait_budget(1234)
    try:
        assert prev == default
        assert lib.spec_set_wait_budget(-5) == -1
        assert binding.spec_set_wait_budget(0) == 1234
        assert binding.spec_set_wait_budget(0) == default
    finally:
        binding.spec_set_wait_budget(0)
