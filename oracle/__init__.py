"""fp64 CPU oracle of the speculative-decoding verification step.

TEST INFRASTRUCTURE ONLY: the correctness reference for the CUDA library.
Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import it.  It shares no code with the CUDA path and never imports the
product package; inputs reach it as plain arrays.

Parity status of each function (what pins it is in ``tests/test_oracle_pins.py``):
  verify / verify_greedy   pinned: exact output law by enumeration on dyadic
                           cases, chi-square of the emitted token against p,
                           per-position acceptance against beta = sum min(p, q),
                           mean AL against the closed form, greedy against
                           plain argmax decoding, special cases.
  softmax_rows             pinned: closed forms.
  lmhead_logits            pinned: direct sum on small shapes.
  gemm_bound.*             pinned: simulated fp32 accumulations (round to
                           nearest and toward zero) stay inside the bound and
                           reach a stated fraction of it; perturbed logits
                           move p and the CDF inside the derived bands
                           (tests/test_oracle_pins_gemm_bound.py).
  speedup.*                pinned: the worked numbers printed on the pages.
  kv_blocks.*              pinned: token-by-token simulation, conservation of
                           block ids, reserve + full rejection = identity,
                           K - M evictions (tests/test_oracle_pins_kv.py).
  ngram.*                  pinned: str.rfind over an encoding of the tokens,
                           a periodic stream's closed form, special cases
                           (tests/test_oracle_pins_ngram.py).
  dynk.*                   pinned: closed form of E[N], the estimator's
                           convergence on simulated acceptance, the pages'
                           window rule, brute-force goodput argmax
                           (tests/test_oracle_pins_dynk.py).
  draft.*                  pinned: Philox4x32-10 known-answer vectors, exact
                           rational enumeration of the draw, chi-square of the
                           draws (tests/test_oracle_pins_draft.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "verify_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_verify_batch.argtypes = [P, ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int64,
                                                ctypes.c_double, ctypes.c_int, P, P, P, P, P, P, P,
                                                ctypes.c_double, P, P]
            lib.oracle_verify_batch.restype = ctypes.c_int
            lib.oracle_softmax_row.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_double, P]
            lib.oracle_softmax_row.restype = None
            lib.oracle_argmax_row.argtypes = [P, ctypes.c_int, ctypes.c_int64]
            lib.oracle_argmax_row.restype = ctypes.c_int64
            _lib = lib
    return _lib


def _as_numpy(x, dtype=None):
    """torch CPU tensor or array -> contiguous numpy array (bf16 as raw uint16)."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        t = x.detach()
        if t.device.type != "cpu":
            raise ValueError("oracle inputs must live on the host")
        if t.dtype == torch.bfloat16:
            return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16)), BF16
        x = t.contiguous().numpy()
    a = np.ascontiguousarray(x if dtype is None else x.astype(dtype, copy=False))
    return a, None


def _logits_code(arr: np.ndarray, tag) -> int:
    if tag == BF16:
        return BF16
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.float64:
        return F64
    raise TypeError(f"unsupported logits dtype {arr.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def verify(logits, q, draft, uniforms, row_offsets, temperature: float, greedy: bool = False,
           tie_band: float = 1e-6, p_rel_err=None, mass_err=None):
    """Run the oracle over a CSR batch.

    logits  (R, V) fp32 / bf16 / fp64;  q (R - B, V) fp32 (ignored if greedy);
    draft (R - B,) int32;  uniforms (R,) fp32 (ignored if greedy);
    row_offsets (B + 1,) int32.  p_rel_err (R - B,) and mass_err (R,) (fp64,
    optional) widen the near-tie tests by known error bounds of the compared
    side's p (see verify_oracle.c).  Returns a dict of numpy arrays:
      out_tokens (R,), accept_len (B,), p_draft (R - B,), residual_mass (B,),
      residual_prob (B,), near_tie_accept (B,), near_tie_sample (B,),
      zero_residual (B,), invalid (int).
    """
    lib = _load()
    z, ztag = _as_numpy(logits)
    zcode = _logits_code(z, ztag)
    R, V = z.shape
    ro, _ = _as_numpy(row_offsets, np.int32)
    ro = ro.astype(np.int32, copy=False)
    B = ro.shape[0] - 1
    x, _ = _as_numpy(draft, np.int32)
    x = x.astype(np.int32, copy=False)
    if greedy:
        qa, ua = None, None
    else:
        qa, _ = _as_numpy(q, np.float32)
        qa = qa.astype(np.float32, copy=False)
        ua, _ = _as_numpy(uniforms, np.float32)
        ua = ua.astype(np.float32, copy=False)
        if temperature <= 0:
            raise ValueError("sampling mode needs T > 0")
    if int(ro[-1]) != R:
        raise ValueError("row_offsets[-1] must equal the number of logits rows")
    out = np.full(R, -1, dtype=np.int32)
    al = np.zeros(B, dtype=np.int32)
    pd = np.full(max(R - B, 1), np.nan, dtype=np.float64)
    req = np.full(2 * B, np.nan, dtype=np.float64)
    flags = np.zeros(3 * B, dtype=np.int32)
    pre = me = None
    if p_rel_err is not None:
        pre = np.ascontiguousarray(np.asarray(p_rel_err, dtype=np.float64).reshape(-1))
        if pre.shape[0] != R - B:
            raise ValueError("p_rel_err needs one value per draft slot")
    if mass_err is not None:
        me = np.ascontiguousarray(np.asarray(mass_err, dtype=np.float64).reshape(-1))
        if me.shape[0] != R:
            raise ValueError("mass_err needs one value per logits row")
    rc = lib.oracle_verify_batch(_ptr(z), zcode, _ptr(qa), _ptr(ro), B, V,
                                 float(temperature if not greedy else 1.0), int(bool(greedy)),
                                 _ptr(x), _ptr(ua), _ptr(out), _ptr(al), _ptr(pd), _ptr(req),
                                 _ptr(flags), float(tie_band), _ptr(pre), _ptr(me))
    if rc < 0:
        raise ValueError("malformed row_offsets")
    flags = flags.reshape(B, 3)
    return {
        "out_tokens": out,
        "accept_len": al,
        "p_draft": pd[: R - B],
        "residual_mass": req[0::2].copy(),
        "residual_prob": req[1::2].copy(),
        "near_tie_accept": flags[:, 0].copy(),
        "near_tie_sample": flags[:, 1].copy(),
        "zero_residual": flags[:, 2].copy(),
        "invalid": int(rc),
    }


def verify_fixed(logits, q, draft, uniforms, B: int, K: int, temperature: float, greedy=False,
                 tie_band: float = 1e-6, p_rel_err=None, mass_err=None):
    ro = (np.arange(B + 1, dtype=np.int32) * (K + 1)).astype(np.int32)
    return verify(logits, q, draft, uniforms, ro, temperature, greedy, tie_band, p_rel_err, mass_err)


def softmax_rows(z, temperature: float) -> np.ndarray:
    """fp64 softmax(z / T) of each row (the oracle's own routine)."""
    lib = _load()
    a, tag = _as_numpy(z)
    code = _logits_code(a, tag)
    rows, V = a.shape
    out = np.empty((rows, V), dtype=np.float64)
    esize = a.dtype.itemsize
    for r in range(rows):
        lib.oracle_softmax_row(ctypes.c_void_p(a.ctypes.data + r * V * esize), code, V,
                               float(temperature), out[r].ctypes.data_as(ctypes.c_void_p))
    return out


def argmax_rows(z) -> np.ndarray:
    lib = _load()
    a, tag = _as_numpy(z)
    code = _logits_code(a, tag)
    rows, V = a.shape
    esize = a.dtype.itemsize
    return np.array([lib.oracle_argmax_row(ctypes.c_void_p(a.ctypes.data + r * V * esize), code, V)
                     for r in range(rows)], dtype=np.int64)


def lmhead_logits(hidden, w_vocab_t, v_chunk: int = 8192) -> np.ndarray:
    """z = hidden . W_vocab in fp64 from the bf16-decoded operands.

    hidden (M, d) bf16; w_vocab_t (V, d) bf16, i.e. W_vocab stored transposed
    (row v holds the d weights of vocabulary entry v).  The product is a
    library matmul in fp64, taken in
    column blocks of the vocabulary to bound host memory.
    """
    import torch
    h64 = hidden.to(torch.float64).numpy()
    V = w_vocab_t.shape[0]
    out = np.empty((h64.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, v_chunk):
        w64 = w_vocab_t[v0:v0 + v_chunk].to(torch.float64).numpy()
        out[:, v0:v0 + v_chunk] = h64 @ w64.T
    return out


def lmhead_verify(hidden, w_vocab_t, q, draft, uniforms, B: int, K: int, temperature: float,
                  tie_band: float = 1e-6, bands=None):
    """Fused front end + verification: fp64 GEMM, then the same steps as verify().
    Returns the verify() dict plus the fp64 logits under "logits".

    bands: None, or a gemm_bound.Bands of this batch (the fp64 logits, their
    accumulation bound and the induced p and mass error bounds, from
    gemm_bound.bands()); its logits are used and its bounds widen the near-tie
    tests.  In greedy mode the bands are not used here (see
    gemm_bound.greedy_flip_possible)."""
    z = lmhead_logits(hidden, w_vocab_t) if bands is None else bands.logits
    greedy = temperature == 0
    pre = me = None
    if bands is not None and not greedy:
        pre, me = bands.p_rel_err_at(draft, B, K), bands.mass_err
    res = verify_fixed(z, q, draft, uniforms, B, K, temperature if not greedy else 1.0, greedy, tie_band,
                       pre, me)
    res["logits"] = z
    return res
