"""Convenience calls over the C ABI: allocate outputs and workspace with torch
(device memory is PyTorch's job here) and run one verification step on the
current stream.  Every step of the computation happens in libspecverify.so.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as _b


class Workspace:
    """Grow-only workspace cache keyed by nothing: reuse one per stream."""

    def __init__(self, device=None):
        self.device = device or torch.device("cuda")
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = _b.workspace(nbytes, self.device)
        return self.buf


_default_ws = {}


def _ws(device, nbytes, ws: Optional[Workspace]):
    if ws is None:
        key = (str(device), torch.cuda.current_stream(device).cuda_stream)
        ws = _default_ws.setdefault(key, Workspace(device))
    return ws.get(nbytes)


def verify_greedy(logits: torch.Tensor, draft: torch.Tensor, K: int, ws: Optional[Workspace] = None):
    rows, V = logits.shape
    B = rows // (K + 1)
    out = torch.empty(rows, dtype=torch.int32, device=logits.device)
    al = torch.empty(B, dtype=torch.int32, device=logits.device)
    w = _ws(logits.device, _b.spec_verify_workspace_size(B, rows, V), ws)
    _b.spec_verify_greedy(logits, draft, B, K, V, out, al, w)
    return out, al


def verify_sample(logits, q, draft, uniforms, K: int, temperature: float, diag: bool = False,
                  ws: Optional[Workspace] = None):
    rows, V = logits.shape
    B = rows // (K + 1)
    out = torch.empty(rows, dtype=torch.int32, device=logits.device)
    al = torch.empty(B, dtype=torch.int32, device=logits.device)
    dg = torch.full((rows - B + 2 * B,), float("nan"), dtype=torch.float32, device=logits.device) if diag else None
    w = _ws(logits.device, _b.spec_verify_workspace_size(B, rows, V), ws)
    _b.spec_verify_sample(logits, q, B, K, V, temperature, draft, uniforms, out, al, w, diag=dg)
    return out, al, dg


def verify_ragged(logits, q, row_offsets, draft, uniforms, temperature: float, diag: bool = False,
                  ws: Optional[Workspace] = None):
    rows, V = logits.shape
    B = row_offsets.numel() - 1
    out = torch.empty(rows, dtype=torch.int32, device=logits.device)
    al = torch.empty(B, dtype=torch.int32, device=logits.device)
    dg = torch.full((rows + B,), float("nan"), dtype=torch.float32, device=logits.device) if diag else None
    w = _ws(logits.device, _b.spec_verify_workspace_size(B, rows, V), ws)
    _b.spec_verify_ragged(logits, q, row_offsets, B, rows, V, temperature, draft, uniforms, out, al, w,
                          diag=dg)
    return out, al, dg


def lmhead_verify(hidden, w_vocab_t, q, draft, uniforms, K: int, temperature: float,
                  diag: bool = False, ws: Optional[Workspace] = None):
    M, d = hidden.shape
    V = w_vocab_t.shape[0]
    B = M // (K + 1)
    out = torch.empty(M, dtype=torch.int32, device=hidden.device)
    al = torch.empty(B, dtype=torch.int32, device=hidden.device)
    dg = torch.full((M + B,), float("nan"), dtype=torch.float32, device=hidden.device) if diag else None
    w = _ws(hidden.device, _b.spec_lmhead_workspace_size(B, K, d, V), ws)
    _b.spec_lmhead_verify(hidden, w_vocab_t, d, q, B, K, V, temperature, draft, uniforms, out, al, w,
                          diag=dg)
    return out, al, dg
