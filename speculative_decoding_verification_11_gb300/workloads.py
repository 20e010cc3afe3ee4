"""Seeded synthetic inputs for the verification step.

This module is the only code shared by the CUDA path and the fp64 oracle.  It
builds the inputs the pages' statement of the problem names (target logits,
draft probabilities q, drafted token ids, uniforms) and holds none of the
verification arithmetic: no acceptance test, no residual, no scan.  It imports
nothing else from this package and touches no GPU.

Random numbers:
  * Gaussian logits and noise come from a seeded ``torch.Generator`` on the CPU.
  * Drafted tokens are drawn from q with ``torch.multinomial`` (the draft
    model's own sampling, which precedes verification).
  * The uniforms the verifier consumes come from Philox4x32-10, written here
    from its published definition (Salmon, Moraes, Dror and Shaw, "Parallel
    Random Numbers: As Easy as 1, 2, 3", SC'11): key = the 64-bit seed,
    counter = (element index, stream id, 0, 0); the first output word x gives
    u = ((x >> 9) + 0.5) * 2**-23, an fp32 value strictly inside (0, 1).

Workloads (shapes and value laws as the task's configurations state them):
  tiny      B=1 per step (1000 steps stacked), K=4, V=1024, fp32, T=1
  greedy    B=32, K=5, V=32000, bf16 logits, argmax-match
  sampling  B=64, K=4, V=128256, fp32, T=0.7, 32 boosted (+8) entries per row
  lmhead    B=16, K=7 (128 rows), d=8192, V=128256, bf16 GEMM front end, T=1
  ragged    B=256, K_i ~ U{0..8} (CSR offsets), V=151936, fp32, T=1
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

# ---------------------------------------------------------------------------
# Philox4x32-10 (SC'11 definition).  Round function on a 4-word counter with a
# 2-word key; the key is bumped by the Weyl constants between rounds.
# ---------------------------------------------------------------------------
_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = np.uint64(0x9E3779B9)
_PHILOX_W1 = np.uint64(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(counter: np.ndarray, key: np.ndarray) -> np.ndarray:
    """Apply Philox4x32 with 10 rounds.

    counter: (N, 4) uint32 array; key: (2,) uint32 array.  Returns (N, 4) uint32.
    """
    c = [counter[:, i].astype(np.uint64) for i in range(4)]
    k0 = np.uint64(key[0])
    k1 = np.uint64(key[1])
    for r in range(10):
        if r > 0:
            k0 = (k0 + _PHILOX_W0) & _MASK32
            k1 = (k1 + _PHILOX_W1) & _MASK32
        p0 = _PHILOX_M0 * c[0]
        p1 = _PHILOX_M1 * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return np.stack([x.astype(np.uint32) for x in c], axis=1)


def philox_uniforms(seed: int, n: int, stream: int = 0, offset: int = 0) -> np.ndarray:
    """n fp32 uniforms in (0, 1): element i uses counter (offset + i, stream, 0, 0)."""
    idx = np.arange(offset, offset + n, dtype=np.uint64)
    ctr = np.zeros((n, 4), dtype=np.uint32)
    ctr[:, 0] = (idx & _MASK32).astype(np.uint32)
    ctr[:, 1] = np.uint32(stream)
    ctr[:, 2] = ((idx >> np.uint64(32)) & _MASK32).astype(np.uint32)
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint32)
    x = philox4x32_10(ctr, key)[:, 0]
    u = ((x >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23
    return u.astype(np.float32)


# ---------------------------------------------------------------------------
# Batch container.  Row r of ``logits`` is position j = r - row_offsets[b] of
# request b (positions 0..K_b); q row / draft slot of that position is
# r - b for j < K_b.  Uniform r is u[b][j]: j < K_b accept draws, j = K_b the
# final draw.  Fixed-K batches use row_offsets[b] = b * (K + 1).
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Batch:
    name: str
    logits: Optional[torch.Tensor]      # (R, V) fp32 or bf16; None for lmhead
    q: Optional[torch.Tensor]           # (Nq, V) fp32; None in greedy mode
    draft: torch.Tensor                 # (Nq,) int32
    uniforms: Optional[torch.Tensor]    # (R,) fp32; None in greedy mode
    row_offsets: torch.Tensor           # (B+1,) int32
    B: int
    K: Optional[int]                    # fixed K, or None when ragged
    V: int
    temperature: float                  # 0 = greedy
    hidden: Optional[torch.Tensor] = None   # lmhead: (R, d) bf16
    w_vocab_t: Optional[torch.Tensor] = None  # lmhead: (V, d) bf16 (Linear weight layout)

    @property
    def rows(self) -> int:
        return int(self.row_offsets[-1])

    @property
    def n_draft(self) -> int:
        return self.rows - self.B


def fixed_offsets(B: int, K: int) -> torch.Tensor:
    return torch.arange(0, B + 1, dtype=torch.int32) * (K + 1)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _softmax_rows_f32(x: torch.Tensor, T: float) -> torch.Tensor:
    """Draft-model probabilities: softmax(x / T) taken in fp64, stored fp32."""
    return torch.softmax(x.to(torch.float64) / T, dim=-1).to(torch.float32)


def _draw_from(q: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    """Draft tokens x ~ q (one per row), via torch.multinomial in fp64."""
    out = torch.empty(q.shape[0], dtype=torch.int32)
    step = 256
    for i in range(0, q.shape[0], step):
        out[i:i + step] = torch.multinomial(q[i:i + step].to(torch.float64), 1,
                                            generator=g).squeeze(1).to(torch.int32)
    return out


def _draft_rows_index(row_offsets: torch.Tensor) -> torch.Tensor:
    """Indices of logits rows that carry a drafted token (positions j < K_b)."""
    ro = row_offsets.tolist()
    idx = []
    for b in range(len(ro) - 1):
        idx.extend(range(ro[b], ro[b + 1] - 1))
    return torch.tensor(idx, dtype=torch.int64)


def make_sampling_batch(name: str, seed: int, B: int, K: Optional[int], V: int, T: float,
                        logit_sigma: float, noise_sigma: float, boost: int = 0,
                        boost_value: float = 8.0, k_list: Optional[list] = None,
                        draft_noise_rows_only: bool = True) -> Batch:
    """Generic sampling-mode batch: target logits z ~ N(0, sigma^2) (+ boosted
    entries), draft logits = z + N(0, noise^2) on the drafted positions,
    q = softmax(draft / T), x ~ q, Philox uniforms."""
    g = _gen(seed)
    if k_list is None:
        row_offsets = fixed_offsets(B, K)
    else:
        ro = [0]
        for k in k_list:
            ro.append(ro[-1] + k + 1)
        row_offsets = torch.tensor(ro, dtype=torch.int32)
    R = int(row_offsets[-1])
    z = torch.randn(R, V, generator=g, dtype=torch.float32) * logit_sigma
    if boost:
        # `boost` distinct, uniformly placed indices per row, raised by boost_value
        keys = torch.rand(R, V, generator=g)
        pos = torch.topk(keys, boost, dim=1).indices
        z.scatter_add_(1, pos, torch.full((R, boost), boost_value))
        del keys
    draft_rows = _draft_rows_index(row_offsets)
    draft_logits = z[draft_rows] + torch.randn(len(draft_rows), V, generator=g) * noise_sigma
    q = _softmax_rows_f32(draft_logits, T)
    del draft_logits
    x = _draw_from(q, g)
    u = torch.from_numpy(philox_uniforms(seed, R, stream=0))
    return Batch(name=name, logits=z, q=q, draft=x, uniforms=u, row_offsets=row_offsets,
                 B=B, K=K, V=V, temperature=T)


def tiny(seed: int = 1000, steps: int = 1000) -> Batch:
    """B=1, K=4, V=1024 per step; `steps` independent steps stacked as requests.
    Target logits N(0, 2^2) over 5 positions; draft logits = target rows 0..3 +
    N(0, 0.5^2); q = softmax(draft); x ~ q; T = 1."""
    b = make_sampling_batch("tiny", seed, B=steps, K=4, V=1024, T=1.0,
                            logit_sigma=2.0, noise_sigma=0.5)
    return b


def greedy(seed: int = 1001, B: int = 32, K: int = 5, V: int = 32000) -> Batch:
    """B=32, K=5, V=32000; target logits bf16(N(0, 3^2)) over 6 positions;
    x_j = argmax(fp32(z_j) + N(0, 1.5^2)) for j < 5."""
    g = _gen(seed)
    row_offsets = fixed_offsets(B, K)
    R = B * (K + 1)
    z = (torch.randn(R, V, generator=g) * 3.0).to(torch.bfloat16)
    draft_rows = _draft_rows_index(row_offsets)
    noisy = z[draft_rows].to(torch.float32) + torch.randn(len(draft_rows), V, generator=g) * 1.5
    x = torch.argmax(noisy, dim=1).to(torch.int32)
    return Batch(name="greedy", logits=z, q=None, draft=x, uniforms=None,
                 row_offsets=row_offsets, B=B, K=K, V=V, temperature=0.0)


def sampling(seed: int = 1002, B: int = 64, K: int = 4, V: int = 128256) -> Batch:
    """B=64, K=4, V=128256; target logits N(0, 2^2) with 32 boosted (+8)
    entries per row; draft logits = target + N(0, 1); q = softmax(draft / T),
    T = 0.7; x ~ q."""
    return make_sampling_batch("sampling", seed, B=B, K=K, V=V, T=0.7,
                               logit_sigma=2.0, noise_sigma=1.0, boost=32)


def ragged(seed: int = 1004, B: int = 256, V: int = 151936, k_max: int = 8) -> Batch:
    """B=256, K_i ~ U{0..8} passed as CSR offsets, V=151936; target logits
    N(0, 2^2); draft logits = target + N(0, 0.8^2); q = softmax(draft); T=1."""
    g = _gen(seed + 77)
    k_list = torch.randint(0, k_max + 1, (B,), generator=g).tolist()
    return make_sampling_batch("ragged", seed, B=B, K=None, V=V, T=1.0,
                               logit_sigma=2.0, noise_sigma=0.8, k_list=k_list)


def lmhead(seed: int = 1003, B: int = 16, K: int = 7, d: int = 8192, V: int = 128256,
           d_draft: int = 2048, T: float = 1.0) -> Batch:
    """Fused LM-head workload: hidden bf16 (B(K+1)) x d ~ N(0, 1); W_vocab
    ~ N(0, 0.02^2) bf16, kept as its transpose (V x d, the layout of a Linear
    layer's weight); q from an independent draft head (hidden (B(K+1)) x 2048
    ~ N(0,1), W 2048 x V ~ N(0, 0.02^2), bf16, fp32 product) over rows
    0..K-1 of each request; x ~ q; T = 1."""
    g = _gen(seed)
    R = B * (K + 1)
    row_offsets = fixed_offsets(B, K)
    hidden = torch.randn(R, d, generator=g).to(torch.bfloat16)
    w_t = torch.empty(V, d, dtype=torch.bfloat16)
    step = 8192
    for i in range(0, V, step):
        w_t[i:i + step] = (torch.randn(min(step, V - i), d, generator=g) * 0.02).to(torch.bfloat16)
    h_d = torch.randn(R, d_draft, generator=g).to(torch.bfloat16)
    draft_rows = _draft_rows_index(row_offsets)
    qs = []
    for i in range(0, V, step):
        wd = (torch.randn(min(step, V - i), d_draft, generator=g) * 0.02).to(torch.bfloat16)
        qs.append(h_d[draft_rows].to(torch.float32) @ wd.to(torch.float32).T)
    draft_logits = torch.cat(qs, dim=1)
    q = _softmax_rows_f32(draft_logits, T)
    del draft_logits
    x = _draw_from(q, g) if q.shape[0] else torch.empty(0, dtype=torch.int32)
    u = torch.from_numpy(philox_uniforms(seed, R, stream=0))
    return Batch(name="lmhead", logits=None, q=q, draft=x, uniforms=u,
                 row_offsets=row_offsets, B=B, K=K, V=V, temperature=T,
                 hidden=hidden, w_vocab_t=w_t)


def lmhead_small(seed: int = 2003, B: int = 4, K: int = 3, d: int = 512, V: int = 4000,
                 T: float = 1.0) -> Batch:
    """A reduced LM-head batch with the same value laws (for oracle-speed parity)."""
    return lmhead(seed=seed, B=B, K=K, d=d, V=V, d_draft=256, T=T)


CONFIGS = {
    "tiny": tiny,
    "greedy": greedy,
    "sampling": sampling,
    "lmhead": lmhead,
    "ragged": ragged,
}


def nominal_bytes(batch: Batch) -> int:
    """Bytes of logits + q, each read once (the pages' roofline convention)."""
    esize = 2 if (batch.logits is not None and batch.logits.dtype == torch.bfloat16) else 4
    lb = batch.rows * batch.V * esize if batch.logits is not None else 0
    qb = batch.n_draft * batch.V * 4 if batch.q is not None else 0
    return lb + qb


def repetitive_streams(seed: int = 1006, B: int = 256, L: int = 8192, vocab: int = 32000,
                       copy_prob: float = 0.05, span=(8, 64)):
    """Synthetic token streams with repetition, the kind n-gram drafting is for
    (outputs that copy from their inputs).  Each stream starts with one random
    token; then, at every position, with probability copy_prob it copies a span
    of U{span} tokens from a uniformly chosen earlier position, else it emits a
    uniform random token.  Returns (tokens int32 concatenated, offsets (B+1,)
    int32)."""
    rng = np.random.default_rng(seed)
    out, offs = [], [0]
    for _ in range(B):
        s = [int(rng.integers(0, vocab))]
        while len(s) < L:
            if len(s) > 1 and rng.random() < copy_prob:
                n = int(rng.integers(span[0], span[1] + 1))
                src = int(rng.integers(0, len(s) - 1))
                for j in range(n):
                    s.append(s[src + j])
                    if len(s) >= L:
                        break
            else:
                s.append(int(rng.integers(0, vocab)))
        out.extend(s[:L])
        offs.append(offs[-1] + L)
    return np.asarray(out, dtype=np.int32), np.asarray(offs, dtype=np.int32)
