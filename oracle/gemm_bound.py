"""Rounding-error bound of the LM-head GEMM's fp32 accumulation, the bands it
induces on the verification's decisions, and a model of the accumulation.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Nothing here reads a GPU
result: every bound is computed from the operands alone.

What is bounded.  The fused front end computes z = h . W with bf16 operands
and fp32 accumulation (the fused LM-head workload; "Co-Designing AI Models
Using Speculative Decoding for Faster LLM Inference", Guideline 1: the target's
LM-head GEMM).  The pages fix no more than "fp32 accumulate".  The reading
taken is the tensor core's block fused multiply-add: the hidden index k is
walked in ascending order in steps of g = 16 products (one MMA of kind::f16);
a bf16 x bf16 product has at most 16 significant bits and is exact; a step
adds its 16 products to the fp32 accumulator by aligning the 17 addends to
the largest one's exponent e, dropping every addend's bits below
2^(e - 23 - G) (G = 2 guard bits; rounding each addend toward zero), summing
the aligned addends exactly and rounding the sum to fp32.  This is the
behaviour the block-FMA literature describes for NVIDIA tensor cores (Fasi,
Higham, Mikaitis and Pranesh, "Numerical behavior of NVIDIA tensor cores",
PeerJ Computer Science, 2021); the number of guard bits, the rounding
directions and the exponent used for a product are this GPU's, and a GPU test
checks them on crafted operands and bit for bit on random ones
(tests/test_lmhead_logits_gpu.py; emulate() below is that model).

The bound.  Let S_j = B_1 + ... + B_j be the exact partial sums after step j
(B_j the exact sum of step j's products), m_j the largest |product| of step j,
Shat_j the accumulator, e_j = Shat_j - S_j (e_0 = 0).  Step j forms
T_j = Shat_{j-1} + B_j + t_j, where t_j, the addends' dropped bits, is below
16 2^(e - 25) <= 8u max(|Shat_{j-1}|, m_j) (at most 16 addends lose bits, each
less than 2^(e - 23 - G), and 2^e is at most the largest addend; u = 2^-24 is
the fp32 unit roundoff), then rounds: Shat_j = T_j (1 + d_j), |d_j| < 2u (to
nearest or toward zero).  Hence
    |e_j| <= 2u |S_j| + (1 + 2u) [(1 + 8u) |e_{j-1}| + 8u max(|S_{j-1}|, m_j)],
and with rho = (1 + 2u)(1 + 8u), n = d / g:
    |z_fp32 - z| <= beta = rho^n sum_{j=1..n} [2u |S_j| + 8u (1 + 2u) max(|S_{j-1}|, m_j)].
It follows the partial sums rather than the terms, so it is far tighter than
the textbook n u sum_k |h_k w_k| for operands of mixed sign.  The partial sums
are computed here in fp64 from the bf16-decoded operands (their own rounding,
below 2^-50 relative per step, is covered by a factor 1 + 2^-20); m_j is
bounded above by (max_k |h_k|)(max_k |w_k|) over the step.

Induced bands (temperature T; b_v = beta_v / T bounds the error of z_v / T):
  - log p_v = z_v / T - log sum_w exp(z_w / T).  The log-normaliser moves by
    at most L = log sum_w p_w exp(b_w) (Jensen's inequality bounds the move in
    both directions by it), so p_v moves by a relative error of at most
    exp(b_v + L) - 1.  The kernel then evaluates the softmax in fp32, which the
    logits-in parity rule bounds by REL = 1e-5 relative, so
        e_p(v) = exp(b_v + L) (1 + REL) - 1.
  - r = max(0, p - q) (or p itself) moves by at most e_p(v) p_v at every v:
    max(0, .) is 1-Lipschitz and q is an input, the same on both sides.  So
    every partial mass C(v) and the total R move by at most
        E = sum_w e_p(w) p_w.
    A CDF boundary compared with u in normalised units moves by at most
    2 E / (R - E) (the oracle's draw band, verify_oracle.c).
  - greedy: the computed argmax of a row can differ from the fp64 argmax v*
    only if some v != v* has z_v* - z_v <= beta_v* + beta_v.
"""
from __future__ import annotations

import dataclasses

import numpy as np

U32 = 2.0 ** -24   # fp32 unit roundoff
STEP = 16          # products per accumulation step (K of one MMA, bf16)
GUARD = 2          # guard bits kept below the fp32 significand when a step aligns its addends
REL = 1e-5         # relative error of the fp32 softmax evaluation (the logits-in rule)
_FP64_SLACK = 1.0 + 2.0 ** -20


def accumulation_bound(hidden, w_vocab_t, step: int = STEP, v_chunk: int = 512):
    """(z, beta): z = hidden . W in fp64 and beta, the bound above on
    |z_fp32 - z| per element.

    hidden (M, d) bf16 torch tensor; w_vocab_t (V, d) bf16 (row v = the d
    weights of token v).  d must be a multiple of `step`.  Both results are
    (M, V) fp64 numpy arrays."""
    import torch
    M, d = hidden.shape
    V = w_vocab_t.shape[0]
    if d % step:
        raise ValueError("d must be a multiple of the step")
    n = d // step
    u = U32
    rho_n = ((1.0 + 2 * u) * (1.0 + 8 * u)) ** n * _FP64_SLACK
    hb = hidden.to(torch.float64).reshape(M, n, step).permute(1, 0, 2).contiguous()   # (n, M, g)
    hmax = hb.abs().amax(dim=2)                                                       # (n, M)
    z = np.empty((M, V), dtype=np.float64)
    beta = np.empty((M, V), dtype=np.float64)
    for v0 in range(0, V, v_chunk):
        v1 = min(V, v0 + v_chunk)
        wb = w_vocab_t[v0:v1].to(torch.float64).reshape(v1 - v0, n, step).permute(1, 2, 0)  # (n, g, vc)
        S = torch.cumsum(torch.bmm(hb, wb), dim=0)          # S[j] = exact partial sum after step j + 1
        z[:, v0:v1] = S[-1].numpy()
        Sprev = torch.cat([torch.zeros_like(S[:1]), S[:-1]], dim=0).abs_()
        mj = hmax[:, :, None] * wb.abs().amax(dim=1)[:, None, :]   # >= the step's largest |product|
        c = S.abs_().mul_(2 * u) + torch.maximum(Sprev, mj).mul_(8 * u * (1 + 2 * u))
        beta[:, v0:v1] = (c.sum(dim=0) * rho_n).numpy()
    return z, beta


_NONE = -(1 << 30)  # exponent of zero (below every real one)


def _exponent(a: np.ndarray) -> np.ndarray:
    """floor(log2 |a|) per element of a float64 array of normal numbers or
    zeros (bf16 and fp32 values are normal in fp64), read from the bits;
    _NONE for zeros."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    e = ((a.view(np.int64) >> 52) & 0x7FF).astype(np.int64) - 1023
    return np.where(a != 0, e, _NONE)


def _round_toward_zero_f32(s: np.ndarray) -> np.ndarray:
    r = s.astype(np.float32)
    over = np.abs(r.astype(np.float64)) > np.abs(s)
    r[over] = np.nextafter(r[over], np.float32(0))
    return r.astype(np.float64)


def _step(acc, prods, ep, guard):
    """One step of the model: align the accumulator and the step's products
    to the largest exponent (a product's exponent being the sum of its
    operands'; a zero operand's sentinel keeps a zero product below every
    real exponent), keep each addend's bits down to 2^(e - 23 - guard) rounded
    toward zero, add exactly (the aligned addends are integers of at most 27
    bits, 17 of them), round toward zero to fp32."""
    emax = np.maximum(ep.max(axis=-1), _exponent(acc))
    shift = np.where(emax < _NONE // 2, 0, emax) - 23 - guard
    inv_q = np.ldexp(1.0, -shift)
    aligned = (prods * inv_q[..., None]).astype(np.int64).sum(axis=-1) + (acc * inv_q).astype(np.int64)
    return _round_toward_zero_f32(np.ldexp(aligned.astype(np.float64), shift))


def emulate(hidden, w_vocab_t, rows=None, cols=None, step: int = STEP, guard: int = GUARD,
            v_chunk: int = 2048) -> np.ndarray:
    """The accumulation model's fp32 logits (as fp64): all (M, V) of them, or
    the elements (rows[i], cols[i]) when both index arrays are given.  Pure
    numpy over every product: for small shapes and samples."""
    h = hidden.double().numpy()
    w = w_vocab_t.double().numpy()
    d = h.shape[1]
    if rows is not None:
        rows, cols = np.asarray(rows), np.asarray(cols)
        hp, wp = h[rows], w[cols]
        ehp, ewp = _exponent(hp), _exponent(wp)
        acc = np.zeros(rows.shape[0])
        for j in range(0, d, step):
            sl = slice(j, j + step)
            acc = _step(acc, hp[:, sl] * wp[:, sl], ehp[:, sl] + ewp[:, sl], guard)
        return acc
    eh, ew = _exponent(h), _exponent(w)
    M, V = h.shape[0], w.shape[0]
    out = np.empty((M, V))
    for v0 in range(0, V, v_chunk):
        v1 = min(V, v0 + v_chunk)
        acc = np.zeros((M, v1 - v0))
        for j in range(0, d, step):
            sl = slice(j, j + step)
            acc = _step(acc, h[:, None, sl] * w[None, v0:v1, sl], eh[:, None, sl] + ew[None, v0:v1, sl], guard)
        out[:, v0:v1] = acc
    return out


def softmax64(z: np.ndarray, T: float) -> np.ndarray:
    """Row-wise softmax(z / T) in fp64 (max-subtracted)."""
    a = z / T
    a = a - a.max(axis=1, keepdims=True)
    e = np.exp(a)
    return e / e.sum(axis=1, keepdims=True)


def p_error_bounds(z: np.ndarray, beta: np.ndarray, T: float, p: np.ndarray = None):
    """(e_p, E): per element the bound on the relative error of p = softmax(z/T)
    computed from logits within beta of z (and evaluated in fp32), and per row
    the bound on the absolute error of every probability mass of the row."""
    if p is None:
        p = softmax64(z, T)
    b = beta / T
    L = np.log(np.sum(p * np.exp(b), axis=1, keepdims=True))
    e_p = np.exp(b + L) * (1.0 + REL) - 1.0
    E = np.sum(e_p * p, axis=1)
    return e_p, E


def greedy_flip_possible(z: np.ndarray, beta: np.ndarray) -> np.ndarray:
    """Per row: can a computation within beta of z pick another argmax than the
    fp64 one (lowest index on ties)?"""
    vstar = np.argmax(z, axis=1)
    rows = np.arange(z.shape[0])
    zs = z[rows, vstar][:, None]
    bs = beta[rows, vstar][:, None]
    close = (zs - z) <= (bs + beta)
    close[rows, vstar] = False
    return close.any(axis=1)


@dataclasses.dataclass
class Bands:
    """The fp64 logits of a fused batch with their accumulation bound and the
    error bounds it induces at temperature T (None in greedy mode)."""
    logits: np.ndarray       # (M, V) fp64
    beta: np.ndarray         # (M, V) bound on |z_fp32 - z|
    T: float
    e_p: np.ndarray = None   # (M, V) relative error bound of p (sampling)
    mass_err: np.ndarray = None  # (M,) absolute error bound of the row's masses (sampling)

    def p_rel_err_at(self, draft, B: int, K: int) -> np.ndarray:
        """e_p at each draft slot (b, j): row b (K + 1) + j, token draft[b K + j]."""
        x = np.asarray(draft, dtype=np.int64).reshape(B, K)
        rows = (np.arange(B)[:, None] * (K + 1) + np.arange(K)[None, :])
        return self.e_p[rows, x].reshape(-1)


def bands(hidden, w_vocab_t, T: float) -> Bands:
    z, beta = accumulation_bound(hidden, w_vocab_t)
    if T == 0:
        return Bands(logits=z, beta=beta, T=0.0)
    e_p, E = p_error_bounds(z, beta, T)
    return Bands(logits=z, beta=beta, T=T, e_p=e_p, mass_err=E)
