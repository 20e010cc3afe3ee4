"""The bench's algorithmic byte count for a verification call, checked on the
CPU against the scope table's per-step figure worked out by hand for the
headline workload (B=64, K=4, V=128256 fp32): every logit once (164,167,680 B),
16 B per draft for z[x], q[x], x and u (4,096 B), 4 B per output row and per
request (1,536 B), each request's selected logits row a second time
(32,833,536 B) and the q row of each request that rejected (56 of them on this
workload: 28,729,344 B).  The accepted lengths come from the oracle."""
from __future__ import annotations

import numpy as np
import torch

import bench
import oracle
from speculative_decoding_verification_11_gb300 import workloads as W


def test_headline_step_bytes_match_the_scope_table():
    b = W.sampling()
    res = oracle.verify(b.logits, b.q, b.draft, b.uniforms, b.row_offsets, b.temperature)
    al = torch.from_numpy(np.asarray(res["accept_len"], dtype=np.int32))
    rejected = int((al <= b.K).sum())
    assert rejected == 56
    V = b.V
    expected = b.rows * V * 4 + b.n_draft * 16 + (b.rows + b.B) * 4 + b.B * V * 4 + rejected * V * 4
    assert expected == 225_736_192
    assert bench._alg_bytes(b, al, b.rows) == expected


def test_greedy_calls_have_no_second_pass():
    b = W.greedy()
    al = torch.full((b.B,), 1, dtype=torch.int32)
    # bf16 logits once, the drafts' gathers, outputs; no selected-row re-read and no q rows
    assert bench._alg_bytes(b, al, b.rows) == b.rows * b.V * 2 + b.n_draft * 16 + (b.rows + b.B) * 4
