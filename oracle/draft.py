"""Oracle of the draft side: q = softmax(h . W / T) and x ~ q by inverse CDF
with Philox4x32-10 uniforms drawn from (seed, counter).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  The GEMM is the oracle's
fp64 product of the bf16-decoded operands (oracle.lmhead_logits); softmax,
Philox and the draw are the C oracle's (verify_oracle.c).

What it follows: "Speculative Decoding in Large Language Models", section 2
(the draft proposes x ~ q; the verification's law assumes it), and
"Speculative Decoding in Production: Accelerating LLM Inference via Custom
Draft Models" (the draft model's distribution q over the vocabulary).
Readings: a draft head is one linear layer over the vocabulary (the pages'
draft models reduced to their last layer, with synthetic weights); T = 0
drafts greedily (argmax, lowest index on ties) and returns no q; draw r of a
call uses the uniform of index offset + r in Philox stream 1.

Parity: Philox is pinned by published known-answer vectors; the draw by exact
rational enumeration and a chi-square test (tests/test_oracle_pins_draft.py).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _load, lmhead_logits, softmax_rows, argmax_rows

DRAFT_STREAM = 1


def _lib():
    lib = _load()
    if not getattr(lib, "_draft_bound", False):
        P = ctypes.c_void_p
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_philox_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32]
        lib.oracle_philox_uniform.restype = ctypes.c_double
        lib.oracle_draw_inverse_cdf.argtypes = [P, ctypes.c_int64, ctypes.c_double, ctypes.c_double, P]
        lib.oracle_draw_inverse_cdf.restype = ctypes.c_int64
        lib._draft_bound = True
    return lib


def philox4x32_10(counter, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    _lib().oracle_philox4x32_10(c.ctypes.data_as(ctypes.c_void_p), k.ctypes.data_as(ctypes.c_void_p),
                                out.ctypes.data_as(ctypes.c_void_p))
    return out


def philox_uniform(seed: int, index: int, stream: int = DRAFT_STREAM) -> float:
    return float(_lib().oracle_philox_uniform(int(seed) & (2**64 - 1), int(index) & (2**64 - 1), int(stream)))


def draw_inverse_cdf(r, u: float, band: float = 1e-6):
    """(token, near_tie) of the inverse-CDF draw over weights r (fp64)."""
    a = np.ascontiguousarray(np.asarray(r, dtype=np.float64))
    nt = ctypes.c_int(0)
    v = _lib().oracle_draw_inverse_cdf(a.ctypes.data_as(ctypes.c_void_p), a.shape[0], float(u), float(band),
                                       ctypes.byref(nt))
    return int(v), bool(nt.value)


def draft_sample(hidden, w_vocab_t, temperature: float, seed: int, offset: int = 0, tie_band: float = 1e-6,
                 bands=None):
    """hidden (M, d) bf16, w_vocab_t (V, d) bf16.  Returns a dict: logits (fp64),
    q (M, V) fp64 or None (greedy), u (M,) (fp64, exactly representable in
    fp32), x (M,) int32, near_tie (M,) bool.

    bands: None, or the gemm_bound.Bands of these operands at this
    temperature: its logits are used, and row r's draw is a near tie when a
    CDF boundary lies within tie_band + 2 E_r / (1 - E_r) of u (E_r its bound
    on the error of the row's probability masses, whose total is 1)."""
    z = lmhead_logits(hidden, w_vocab_t) if bands is None else bands.logits
    M = z.shape[0]
    if temperature == 0:
        x = argmax_rows(z).astype(np.int32)
        return {"logits": z, "q": None, "u": None, "x": x, "near_tie": np.zeros(M, dtype=bool)}
    q = softmax_rows(z, temperature)
    u = np.array([philox_uniform(seed, offset + r) for r in range(M)], dtype=np.float64)
    x = np.zeros(M, dtype=np.int32)
    nt = np.zeros(M, dtype=bool)
    for r in range(M):
        band = tie_band
        if bands is not None:
            E = float(bands.mass_err[r])
            band = tie_band + 2.0 * E / (1.0 - E) if E < 1.0 else np.inf
        x[r], nt[r] = draw_inverse_cdf(q[r], u[r], band)
    return {"logits": z, "q": q, "u": u, "x": x, "near_tie": nt}
