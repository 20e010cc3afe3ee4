"""Oracle of the paged KV-cache bookkeeping around the verification step.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): plain Python over numpy
arrays, one request at a time, in request order.

What it follows: "Speculative Decoding in Large Language Models: Architecture,
Mathematical Foundations, and Production Engineering", section 4 "Memory
Management: Contiguous vs. Segmented Allocation", subsection "Segmented Block
Allocation (PagedAttention)": the cache is cut into fixed-size blocks, the
allocator hands out block pointers for the speculative tokens, and a rejection
returns the pointers of the evicted positions to the global free list with no
copy; and "Speculative Decoding in Production: Accelerating LLM Inference via
Custom Draft Models", "Serving Architecture and KV Cache Syncing": with M of K
drafts accepted, K - M speculative slots are evicted, in the draft's cache and
in the target's.

Readings (the pages leave these open):
  - One cache is one block table (B x max_blocks, -1 = no block), one length
    per request (tokens with valid KV) and one free list, a stack of block ids
    whose top count is free_count.
  - reserve(n_new): request b gets the blocks that cover positions
    [0, seq_len_b + n_new_b); blocks are popped from the top of the stack,
    request 0 taking the lowest stack slots of the popped range, each
    request's blocks in logical order.  If the free list is short, nothing
    changes and the call reports it.
  - rollback(n_spec, accept_len): request b wrote n_spec_b speculative slots
    after its seq_len_b valid ones; of those, accept_len_b - 1 accepted drafts
    keep their KV (accept_len_b = 0, an invalid request, keeps none; the final
    emitted token gets its KV in the next step).  new_len = seq_len + kept.
    The blocks wholly beyond new_len, logical blocks ceil(new_len / bs) ..
    ceil((seq_len + n_spec) / bs) - 1, go back to the free list: pushed in
    request order, each request's blocks in logical order, the table entries
    set to -1.
  - Inputs that break a rule (a negative count, a length beyond the table, an
    accept length outside [0, n_spec + 1], a table entry that reserve would
    fill already holding a block, a table entry that rollback would free
    holding none, a free list that would overflow its capacity) leave
    everything unchanged and are reported.

Parity: exact (integer work); pinned by closed forms, conservation of block
ids and a token-by-token simulation in tests/test_oracle_pins_kv.py.
"""
from __future__ import annotations

import numpy as np

OK, OUT_OF_BLOCKS, BAD_INPUT = 0, 1, 2


def blocks_for(n_tokens: int, block_size: int) -> int:
    """Blocks that hold positions [0, n_tokens): ceil(n / bs)."""
    return -(-int(n_tokens) // int(block_size))


def reserve(block_table, seq_len, free_ids, free_count, n_new, block_size):
    """Returns (block_table, free_count, status) after the reservation; the
    arrays passed in are not modified."""
    bt = np.array(block_table, dtype=np.int32, copy=True)
    B, max_blocks = bt.shape
    fc = int(free_count)
    need = []
    for b in range(B):
        have = blocks_for(seq_len[b], block_size)
        want = blocks_for(int(seq_len[b]) + int(n_new[b]), block_size)
        if n_new[b] < 0 or seq_len[b] < 0 or want > max_blocks:
            return np.array(block_table, dtype=np.int32, copy=True), int(free_count), BAD_INPUT
        if any(bt[b, i] >= 0 for i in range(have, want)):  # would leak the block held there
            return np.array(block_table, dtype=np.int32, copy=True), int(free_count), BAD_INPUT
        need.append((have, want))
    total = sum(w - h for h, w in need)
    if total > fc:
        return np.array(block_table, dtype=np.int32, copy=True), int(free_count), OUT_OF_BLOCKS
    base = fc - total
    k = base
    for b, (have, want) in enumerate(need):
        for i in range(have, want):
            bt[b, i] = free_ids[k]
            k += 1
    return bt, base, OK


def rollback(block_table, seq_len, free_ids, free_count, n_spec, accept_len, block_size):
    """Returns (block_table, seq_len, free_ids, free_count, status) after the
    rollback; the arrays passed in are not modified."""
    bt = np.array(block_table, dtype=np.int32, copy=True)
    sl = np.array(seq_len, dtype=np.int32, copy=True)
    fl = np.array(free_ids, dtype=np.int32, copy=True)
    B, max_blocks = bt.shape
    fc = int(free_count)
    plan = []
    for b in range(B):
        al = int(accept_len[b])
        end = int(seq_len[b]) + int(n_spec[b])
        if n_spec[b] < 0 or seq_len[b] < 0 or al < 0 or al > int(n_spec[b]) + 1 or \
                blocks_for(end, block_size) > max_blocks:
            return (np.array(block_table, dtype=np.int32, copy=True), np.array(seq_len, dtype=np.int32, copy=True),
                    np.array(free_ids, dtype=np.int32, copy=True), int(free_count), BAD_INPUT)
        kept = max(al - 1, 0)
        new_len = int(seq_len[b]) + kept
        lo, hi = blocks_for(new_len, block_size), blocks_for(end, block_size)
        if any(bt[b, i] < 0 for i in range(lo, hi)):
            return (np.array(block_table, dtype=np.int32, copy=True), np.array(seq_len, dtype=np.int32, copy=True),
                    np.array(free_ids, dtype=np.int32, copy=True), int(free_count), BAD_INPUT)
        plan.append((new_len, lo, hi))
    total = sum(hi - lo for _, lo, hi in plan)
    if fc + total > len(fl):
        return (np.array(block_table, dtype=np.int32, copy=True), np.array(seq_len, dtype=np.int32, copy=True),
                np.array(free_ids, dtype=np.int32, copy=True), int(free_count), BAD_INPUT)
    k = fc
    for b, (new_len, lo, hi) in enumerate(plan):
        for i in range(lo, hi):
            fl[k] = bt[b, i]
            bt[b, i] = -1
            k += 1
        sl[b] = new_len
    return bt, sl, fl, k, OK
