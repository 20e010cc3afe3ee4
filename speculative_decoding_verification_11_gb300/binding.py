"""Thin Python binding of libspecverify.so (ctypes).

Argument marshalling only: every function passes device pointers, sizes and
the current CUDA stream straight to the C entry point of the same name in
``include/specverify.h``.  No step of the verification runs here, and there is
no CPU fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

SV_OK, SV_ERR_INVALID, SV_ERR_CUDA, SV_ERR_DEVICE_INPUT, SV_ERR_TIMEOUT, SV_ERR_WORKSPACE = range(6)
SV_F32, SV_BF16 = 0, 1
SV_FLAG_BAD_TOKEN, SV_FLAG_BAD_OFFSETS, SV_FLAG_ZERO_RESIDUAL, SV_FLAG_TIMEOUT = 1, 2, 4, 8
SV_FLAG_KV_OUT_OF_BLOCKS, SV_FLAG_KV_BAD_INPUT = 0x10, 0x20
SV_DYNK_WINDOW, SV_DYNK_GOODPUT = 0, 1
SV_MAX_K = 255

EXPORTS = (
    "spec_verify_workspace_size", "spec_verify_greedy", "spec_verify_sample", "spec_verify_ragged",
    "spec_lmhead_workspace_size", "spec_lmhead_verify", "spec_verify_last_device_status",
    "spec_status_string", "spec_profile_set_events", "spec_last_launch_count", "spec_last_kernel",
    "spec_verify_sample_noalloc", "spec_set_small_kernel_limit", "spec_set_cluster_kernel",
    "spec_kv_reserve", "spec_kv_rollback",
    "spec_draft_workspace_size", "spec_draft_sample", "spec_ngram_draft", "spec_dynk_update",
    "spec_lmhead_logits", "spec_set_wait_budget",
)

_lock = threading.Lock()
_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load the built library (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sig = {
            "spec_verify_workspace_size": (Z, [I, I, I]),
            "spec_verify_greedy": (I, [P, I, I, I, I, P, P, P, P, Z, P]),
            "spec_verify_sample": (I, [P, I, P, I, I, I, F, P, P, P, P, P, P, Z, P]),
            "spec_verify_ragged": (I, [P, I, P, P, I, I, I, F, P, P, P, P, P, P, Z, P]),
            "spec_lmhead_workspace_size": (Z, [I, I, I, I]),
            "spec_lmhead_verify": (I, [P, P, I, P, I, I, I, F, P, P, P, P, P, P, Z, P]),
            "spec_verify_last_device_status": (I, [P, P, P]),
            "spec_status_string": (ctypes.c_char_p, [I]),
            "spec_profile_set_events": (I, [P, P]),
            "spec_last_launch_count": (I, []),
            "spec_last_kernel": (ctypes.c_char_p, []),
            "spec_verify_sample_noalloc": (I, [P, I, P, I, I, I, F, P, P, P, P, P, P]),
            "spec_set_small_kernel_limit": (Z, [Z]),
            "spec_set_cluster_kernel": (I, [I]),
            "spec_kv_reserve": (I, [P, P, P, P, P, I, I, I, P, P]),
            "spec_kv_rollback": (I, [P, P, P, P, P, P, I, I, I, I, P, P]),
            "spec_draft_workspace_size": (Z, [I, I, I]),
            "spec_draft_sample": (I, [P, P, I, I, I, F, ctypes.c_uint64, ctypes.c_uint64, P, P, P, P, Z, P]),
            "spec_ngram_draft": (I, [P, P, I, I, I, I, P, P, P]),
            "spec_dynk_update": (I, [P, P, P, P, I, I, I, F, I, I, P, F, P, P, P]),
            "spec_lmhead_logits": (I, [P, P, I, I, I, P, P, Z, P]),
            "spec_set_wait_budget": (ctypes.c_longlong, [ctypes.c_longlong]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().spec_status_string(int(status)).decode()
    except Exception:  # library not loadable: plain number
        return f"status {status}"


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------
def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libspecverify must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libspecverify must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _check(t, dtype, numel=None, name="tensor"):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: expected {numel} elements, got {t.numel()}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise TypeError(f"logits must be fp32 or bf16, got {t.dtype}")


def _raise(status, where):
    if status != SV_OK:
        raise SpecVerifyError(status, where)


# --------------------------------------------------------------------------
# the C entry points, same names
# --------------------------------------------------------------------------
def spec_verify_workspace_size(B: int, rows: int, V: int) -> int:
    return int(load().spec_verify_workspace_size(B, rows, V))


def spec_lmhead_workspace_size(B: int, K: int, d: int, V: int) -> int:
    return int(load().spec_lmhead_workspace_size(B, K, d, V))


def spec_verify_greedy(logits, draft, B, K, V, out_tokens, accept_len, ws, stream=None):
    _check(draft, torch.int32, B * K, "draft")
    _check(out_tokens, torch.int32, B * (K + 1), "out_tokens")
    _check(accept_len, torch.int32, B, "accept_len")
    st = load().spec_verify_greedy(_ptr(logits), _dtype_code(logits), B, K, V, _ptr(draft),
                                   _ptr(out_tokens), _ptr(accept_len), _ptr(ws), ws.numel(),
                                   _stream(stream))
    _raise(st, "spec_verify_greedy")


def spec_verify_sample(logits, q, B, K, V, temperature, draft, uniforms, out_tokens, accept_len,
                       ws, diag=None, stream=None):
    _check(q, torch.float32, B * K * V, "q")
    _check(draft, torch.int32, B * K, "draft")
    _check(uniforms, torch.float32, B * (K + 1), "uniforms")
    _check(out_tokens, torch.int32, B * (K + 1), "out_tokens")
    _check(accept_len, torch.int32, B, "accept_len")
    st = load().spec_verify_sample(_ptr(logits), _dtype_code(logits), _ptr(q), B, K, V,
                                   float(temperature), _ptr(draft), _ptr(uniforms),
                                   _ptr(out_tokens), _ptr(accept_len), _ptr(diag), _ptr(ws),
                                   ws.numel(), _stream(stream))
    _raise(st, "spec_verify_sample")


def spec_verify_ragged(logits, q, row_offsets, B, rows, V, temperature, draft, uniforms,
                       out_tokens, accept_len, ws, diag=None, stream=None):
    _check(row_offsets, torch.int32, B + 1, "row_offsets")
    _check(out_tokens, torch.int32, rows, "out_tokens")
    _check(accept_len, torch.int32, B, "accept_len")
    st = load().spec_verify_ragged(_ptr(logits), _dtype_code(logits), _ptr(q), _ptr(row_offsets),
                                   B, rows, V, float(temperature), _ptr(draft), _ptr(uniforms),
                                   _ptr(out_tokens), _ptr(accept_len), _ptr(diag), _ptr(ws),
                                   ws.numel(), _stream(stream))
    _raise(st, "spec_verify_ragged")


def spec_lmhead_verify(hidden, w_vocab_t, d, q, B, K, V, temperature, draft, uniforms,
                       out_tokens, accept_len, ws, diag=None, stream=None):
    _check(hidden, torch.bfloat16, B * (K + 1) * d, "hidden")
    _check(w_vocab_t, torch.bfloat16, V * d, "w_vocab_t")
    _check(out_tokens, torch.int32, B * (K + 1), "out_tokens")
    _check(accept_len, torch.int32, B, "accept_len")
    st = load().spec_lmhead_verify(_ptr(hidden), _ptr(w_vocab_t), d, _ptr(q), B, K, V,
                                   float(temperature), _ptr(draft), _ptr(uniforms),
                                   _ptr(out_tokens), _ptr(accept_len), _ptr(diag), _ptr(ws),
                                   ws.numel(), _stream(stream))
    _raise(st, "spec_lmhead_verify")


def spec_verify_sample_noalloc(logits, q, B, K, V, temperature, draft, uniforms, out_tokens, accept_len,
                               diag=None, stream=None):
    """spec_verify_sample without a workspace: for callers that cannot allocate
    device memory; the library's own fixed scratch array is used instead."""
    _check(q, torch.float32, B * K * V, "q")
    _check(draft, torch.int32, B * K, "draft")
    _check(uniforms, torch.float32, B * (K + 1), "uniforms")
    _check(out_tokens, torch.int32, B * (K + 1), "out_tokens")
    _check(accept_len, torch.int32, B, "accept_len")
    st = load().spec_verify_sample_noalloc(_ptr(logits), _dtype_code(logits), _ptr(q), B, K, V,
                                           float(temperature), _ptr(draft), _ptr(uniforms),
                                           _ptr(out_tokens), _ptr(accept_len), _ptr(diag),
                                           _stream(stream))
    _raise(st, "spec_verify_sample_noalloc")


NOALLOC_SCRATCH_BYTES = 2 << 20


def spec_verify_last_device_status(ws, stream=None):
    """Returns (status, flags); synchronises the stream and clears the word."""
    flags = ctypes.c_uint32(0)
    st = load().spec_verify_last_device_status(_ptr(ws), _stream(stream), ctypes.byref(flags))
    return int(st), int(flags.value)


def spec_profile_set_events(begin=None, end=None):
    b = ctypes.c_void_p(begin.cuda_event) if begin is not None else None
    e = ctypes.c_void_p(end.cuda_event) if end is not None else None
    _raise(load().spec_profile_set_events(b, e), "spec_profile_set_events")


def bind_spec_verify_sample(logits, q, B, K, V, temperature, draft, uniforms, out_tokens, accept_len,
                            ws, diag=None, stream=None):
    """spec_verify_sample with its arguments checked and marshalled once: returns
    a function of no arguments that makes the same C call again.  For loops that
    issue the same call many times (the tensors must stay alive and in place)."""
    _check(q, torch.float32, B * K * V, "q")
    _check(draft, torch.int32, B * K, "draft")
    _check(uniforms, torch.float32, B * (K + 1), "uniforms")
    _check(out_tokens, torch.int32, B * (K + 1), "out_tokens")
    _check(accept_len, torch.int32, B, "accept_len")
    fn = load().spec_verify_sample
    args = (_ptr(logits), _dtype_code(logits), _ptr(q), B, K, V, float(temperature), _ptr(draft),
            _ptr(uniforms), _ptr(out_tokens), _ptr(accept_len), _ptr(diag), _ptr(ws), ws.numel(),
            _stream(stream))

    def call():
        st = fn(*args)
        if st != SV_OK:
            raise SpecVerifyError(st, "spec_verify_sample")

    return call


def bind_spec_profile_set_events(begin=None, end=None):
    """spec_profile_set_events with the event handles taken once (the events
    must already have been recorded once, so that they exist)."""
    fn = load().spec_profile_set_events
    b = ctypes.c_void_p(begin.cuda_event) if begin is not None else None
    e = ctypes.c_void_p(end.cuda_event) if end is not None else None

    def call():
        _raise(fn(b, e), "spec_profile_set_events")

    return call


def spec_set_wait_budget(cycles: int) -> int:
    """Device-side wait limit in SM cycles (0 restores the default); returns the
    previous value."""
    prev = int(load().spec_set_wait_budget(int(cycles)))
    if prev < 0:
        raise ValueError("cycles must be >= 0")
    return prev


def spec_set_small_kernel_limit(nbytes: int) -> int:
    """Largest per-request logits footprint (bytes) that runs on the
    request-per-CTA kernel; 0 sends every call to the streaming kernel.
    Returns the previous value."""
    return int(load().spec_set_small_kernel_limit(int(nbytes)))


def spec_set_cluster_kernel(enable: bool) -> bool:
    """Whether small batches of medium requests may run one cluster of CTAs
    per request.  Returns the previous setting."""
    return bool(load().spec_set_cluster_kernel(1 if enable else 0))


def _check_kv(block_table, seq_len, free_ids, free_count, status):
    _check(block_table, torch.int32, None, "block_table")
    _check(seq_len, torch.int32, block_table.shape[0], "seq_len")
    _check(free_ids, torch.int32, None, "free_ids")
    _check(free_count, torch.int32, 1, "free_count")
    if status is None or status.dtype not in (torch.int32, torch.uint32) or status.numel() < 1:
        raise TypeError("status: a device int32/uint32 word is required")
    if block_table.dim() != 2:
        raise ValueError("block_table: expected (B, max_blocks)")


def spec_kv_reserve(block_table, seq_len, free_ids, free_count, n_new, block_size, status, stream=None):
    _check_kv(block_table, seq_len, free_ids, free_count, status)
    B, max_blocks = block_table.shape
    _check(n_new, torch.int32, B, "n_new")
    st = load().spec_kv_reserve(_ptr(block_table), _ptr(seq_len), _ptr(free_ids), _ptr(free_count), _ptr(n_new),
                                B, max_blocks, int(block_size), _ptr(status), _stream(stream))
    _raise(st, "spec_kv_reserve")


def spec_kv_rollback(block_table, seq_len, free_ids, free_count, n_spec, accept_len, block_size, status,
                     stream=None):
    _check_kv(block_table, seq_len, free_ids, free_count, status)
    B, max_blocks = block_table.shape
    _check(n_spec, torch.int32, B, "n_spec")
    _check(accept_len, torch.int32, B, "accept_len")
    st = load().spec_kv_rollback(_ptr(block_table), _ptr(seq_len), _ptr(free_ids), _ptr(free_count), _ptr(n_spec),
                                 _ptr(accept_len), B, max_blocks, int(block_size), free_ids.numel(), _ptr(status),
                                 _stream(stream))
    _raise(st, "spec_kv_rollback")


def spec_draft_workspace_size(M: int, d: int, V: int) -> int:
    return int(load().spec_draft_workspace_size(M, d, V))


def spec_draft_sample(hidden, w_vocab_t, temperature, seed, offset, q_out, x_out, ws, u_out=None, stream=None):
    """Draft head + sampling: q_out (M, V) fp32 (sampling) and x_out (M,) int32."""
    _check(hidden, torch.bfloat16, None, "hidden")
    _check(w_vocab_t, torch.bfloat16, None, "w_vocab_t")
    M, d = hidden.shape
    V = w_vocab_t.shape[0]
    if w_vocab_t.shape[1] != d:
        raise ValueError("w_vocab_t: expected (V, d)")
    _check(x_out, torch.int32, M, "x_out")
    if temperature > 0:
        _check(q_out, torch.float32, M * V, "q_out")
    _check(u_out, torch.float32, M, "u_out")
    st = load().spec_draft_sample(_ptr(hidden), _ptr(w_vocab_t), d, M, V, float(temperature),
                                  int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _ptr(q_out), _ptr(x_out),
                                  _ptr(u_out), _ptr(ws), ws.numel(), _stream(stream))
    _raise(st, "spec_draft_sample")


def spec_lmhead_logits(hidden, w_vocab_t, logits, ws, stream=None):
    """logits (M x V fp32) = hidden (M x d bf16) . w_vocab_t (V x d bf16)^T on
    the LM-head GEMM; ws of spec_draft_workspace_size(M, d, V) bytes."""
    _check(hidden, torch.bfloat16, None, "hidden")
    _check(w_vocab_t, torch.bfloat16, None, "w_vocab_t")
    M, d = hidden.shape
    V = w_vocab_t.shape[0]
    _check(logits, torch.float32, M * V, "logits")
    st = load().spec_lmhead_logits(_ptr(hidden), _ptr(w_vocab_t), d, M, V, _ptr(logits), _ptr(ws), ws.numel(),
                                   _stream(stream))
    _raise(st, "spec_lmhead_logits")


def spec_ngram_draft(tokens, ctx_offsets, K, n_min, n_max, draft_out, k_out, stream=None):
    """Prompt-lookup drafts: draft_out (B, K) int32 (-1 padded), k_out (B,) int32."""
    _check(tokens, torch.int32, None, "tokens")
    _check(ctx_offsets, torch.int32, None, "ctx_offsets")
    B = ctx_offsets.numel() - 1
    _check(draft_out, torch.int32, B * K, "draft_out")
    _check(k_out, torch.int32, B, "k_out")
    st = load().spec_ngram_draft(_ptr(tokens), _ptr(ctx_offsets), B, K, n_min, n_max, _ptr(draft_out), _ptr(k_out),
                                 _stream(stream))
    _raise(st, "spec_ngram_draft")


def spec_dynk_update(accept_len, k_used, hist, count, policy, k_low, k_high, k_next, threshold=1.5, itl=None,
                     alpha_prior=0.5, row_offsets=None, stream=None):
    """Dynamic K after verification; hist (B, W, 2) int32 and count (B,) int32
    carry the state between calls."""
    B = accept_len.numel()
    _check(accept_len, torch.int32, B, "accept_len")
    _check(k_used, torch.int32, B, "k_used")
    _check(hist, torch.int32, None, "hist")
    _check(count, torch.int32, B, "count")
    _check(k_next, torch.int32, B, "k_next")
    _check(itl, torch.float32, None, "itl")
    _check(row_offsets, torch.int32, B + 1, "row_offsets")
    if hist.dim() != 3 or hist.shape[0] != B or hist.shape[2] != 2:
        raise ValueError("hist: expected (B, W, 2)")
    st = load().spec_dynk_update(_ptr(accept_len), _ptr(k_used), _ptr(hist), _ptr(count), B, hist.shape[1],
                                 int(policy), float(threshold), int(k_low), int(k_high), _ptr(itl), float(alpha_prior),
                                 _ptr(k_next), _ptr(row_offsets), _stream(stream))
    _raise(st, "spec_dynk_update")


def spec_last_launch_count() -> int:
    return int(load().spec_last_launch_count())


def spec_last_kernel() -> str:
    """The verification kernel the last verify call on this thread chose:
    "small", "cluster", "stream", "scalar" or "none"."""
    return load().spec_last_kernel().decode()


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A 256-byte aligned device buffer of nbytes (uint8) from torch's allocator."""
    t = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-t.data_ptr()) % 256
    return t[off:off + nbytes]
