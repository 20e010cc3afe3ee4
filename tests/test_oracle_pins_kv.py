"""Pins of the paged KV-cache oracle (oracle/kv_blocks.py) against facts that do
not come from its own code: a token-by-token simulation of the cache, the
conservation of block ids, the identity of a reservation followed by a full
rejection, the pages' statement that K - M slots are evicted when M of K
drafts are accepted, and the error cases.
"""
from __future__ import annotations

import numpy as np
import pytest

from oracle import kv_blocks as kv


def _state(rng, B, max_blocks, bs, n_ids=None, fill=0.5):
    """A consistent random cache: every request holds the blocks of its length,
    the remaining ids are on the free stack in a random order."""
    n_ids = n_ids or B * max_blocks + 7
    ids = rng.permutation(n_ids).astype(np.int32)
    bt = np.full((B, max_blocks), -1, dtype=np.int32)
    seq = np.zeros(B, dtype=np.int32)
    k = 0
    for b in range(B):
        seq[b] = rng.integers(0, int(max_blocks * bs * fill) + 1)
        for i in range(kv.blocks_for(seq[b], bs)):
            bt[b, i] = ids[k]
            k += 1
    free = np.full(n_ids, -1, dtype=np.int32)
    rest = ids[k:]
    free[:len(rest)] = rest
    return bt, seq, free, len(rest)


def _ids_in_use(bt, free, fc):
    return np.sort(np.concatenate([bt[bt >= 0], free[:fc]]))


def _simulate_blocks(seq_len, n_add, n_remove, bs):
    """Token-level model: positions are appended one at a time, a position that
    starts a block (p % bs == 0) takes a new block; then positions are removed
    from the end one at a time, and removing the first position of a block
    frees it.  Returns (blocks taken, blocks freed)."""
    pos = list(range(seq_len))
    taken = freed = 0
    for _ in range(n_add):
        p = len(pos)
        if p % bs == 0:
            taken += 1
        pos.append(p)
    for _ in range(n_remove):
        p = pos.pop()
        if p % bs == 0:
            freed += 1
    return taken, freed


@pytest.mark.parametrize("bs", [1, 3, 16])
def test_counts_match_token_by_token_simulation(bs):
    rng = np.random.default_rng(bs)
    B, max_blocks = 40, 12
    bt, seq, free, fc = _state(rng, B, max_blocks, bs, fill=0.6)
    K = rng.integers(0, 7, size=B).astype(np.int32)
    K = np.minimum(K, max_blocks * bs - seq).astype(np.int32)
    al = np.array([rng.integers(0, k + 2) for k in K], dtype=np.int32)
    bt1, fc1, st = kv.reserve(bt, seq, free, fc, K, bs)
    assert st == kv.OK
    bt2, seq2, free2, fc2, st = kv.rollback(bt1, seq, free, fc1, K, al, bs)
    assert st == kv.OK
    for b in range(B):
        kept = max(int(al[b]) - 1, 0)
        taken, freed = _simulate_blocks(int(seq[b]), int(K[b]), int(K[b]) - kept, bs)
        assert int((bt1[b] >= 0).sum() - (bt[b] >= 0).sum()) == taken
        assert int((bt1[b] >= 0).sum() - (bt2[b] >= 0).sum()) == freed
        assert seq2[b] == seq[b] + kept
        # the table holds exactly the blocks of the new length, as a prefix
        n = int((bt2[b] >= 0).sum())
        assert np.all(bt2[b, :n] >= 0) and np.all(bt2[b, n:] < 0)
        assert (n - 1) * bs < max(int(seq2[b]), 1) <= n * bs or (n == 0 and seq2[b] == 0)
    assert fc1 == fc - int((bt1 >= 0).sum() - (bt >= 0).sum())
    assert fc2 == fc1 + int((bt1 >= 0).sum() - (bt2 >= 0).sum())


def test_block_ids_are_conserved():
    rng = np.random.default_rng(5)
    bs, B, max_blocks = 4, 30, 10
    bt, seq, free, fc = _state(rng, B, max_blocks, bs)
    before = _ids_in_use(bt, free, fc)
    for step in range(6):
        K = np.minimum(rng.integers(0, 9, size=B), max_blocks * bs - seq).astype(np.int32)
        bt, fc, st = kv.reserve(bt, seq, free, fc, K, bs)
        assert st == kv.OK
        al = np.array([rng.integers(0, k + 2) for k in K], dtype=np.int32)
        bt, seq, free, fc, st = kv.rollback(bt, seq, free, fc, K, al, bs)
        assert st == kv.OK
        after = _ids_in_use(bt, free, fc)
        assert np.array_equal(after, before), step


@pytest.mark.parametrize("bs", [3, 8])
def test_reserve_then_full_rejection_is_the_identity(bs):
    """accept_len = 1 keeps no draft: every block the reservation took goes back,
    in the order it left, and the cache is as before (spans of several blocks)."""
    rng = np.random.default_rng(11)
    bt, seq, free, fc = _state(rng, 25, 9, bs)
    K = np.minimum(rng.integers(1, 3 * bs + 2, size=25), 9 * bs - seq).astype(np.int32)
    bt1, fc1, _ = kv.reserve(bt, seq, free, fc, K, bs)
    bt2, seq2, free2, fc2, st = kv.rollback(bt1, seq, free, fc1, K, np.ones(25, np.int32), bs)
    assert st == kv.OK
    assert np.array_equal(bt2, bt) and np.array_equal(seq2, seq) and fc2 == fc
    assert np.array_equal(free2[:fc2], free[:fc])


def test_full_acceptance_keeps_every_speculative_block():
    rng = np.random.default_rng(12)
    bs = 5
    bt, seq, free, fc = _state(rng, 20, 8, bs)
    K = np.minimum(rng.integers(0, 9, size=20), 8 * bs - seq).astype(np.int32)
    bt1, fc1, _ = kv.reserve(bt, seq, free, fc, K, bs)
    bt2, seq2, _, fc2, st = kv.rollback(bt1, seq, free, fc1, K, K + 1, bs)
    assert st == kv.OK and fc2 == fc1 and np.array_equal(bt2, bt1)
    assert np.array_equal(seq2, seq + K)


def test_block_size_one_evicts_k_minus_m_slots():
    """One token per block: with M of K drafts accepted, K - M slots (blocks)
    are evicted, as the pages state."""
    rng = np.random.default_rng(13)
    bt, seq, free, fc = _state(rng, 16, 40, 1, fill=0.5)
    K = np.minimum(rng.integers(0, 9, size=16), 40 - seq).astype(np.int32)
    bt1, fc1, _ = kv.reserve(bt, seq, free, fc, K, 1)
    M = np.array([rng.integers(0, k + 1) for k in K], dtype=np.int32)
    _, _, _, fc2, st = kv.rollback(bt1, seq, free, fc1, K, M + 1, 1)
    assert st == kv.OK
    assert fc2 - fc1 == int((K - M).sum())


def test_invalid_request_keeps_nothing():
    bs = 4
    bt = np.array([[7, 3, -1, -1]], dtype=np.int32)
    seq = np.array([5], dtype=np.int32)
    free = np.array([9, 8, 6, -1, -1, -1], dtype=np.int32)
    bt1, fc1, st = kv.reserve(bt, seq, free, 3, np.array([6]), bs)   # 11 tokens: 3 blocks
    assert st == kv.OK and fc1 == 2 and list(bt1[0]) == [7, 3, 6, -1]
    bt2, seq2, free2, fc2, st = kv.rollback(bt1, seq, free, fc1, np.array([6]), np.array([0]), bs)
    assert st == kv.OK and seq2[0] == 5 and list(bt2[0]) == [7, 3, -1, -1]
    assert fc2 == 3 and list(free2[:3]) == [9, 8, 6]


def test_out_of_blocks_and_bad_inputs_change_nothing():
    bs = 4
    bt = np.array([[1, -1], [2, -1]], dtype=np.int32)
    seq = np.array([3, 4], dtype=np.int32)
    free = np.array([5, -1, -1, -1], dtype=np.int32)
    out = kv.reserve(bt, seq, free, 1, np.array([2, 2]), bs)  # needs 2 blocks, 1 free
    assert out[2] == kv.OUT_OF_BLOCKS and np.array_equal(out[0], bt) and out[1] == 1
    out = kv.reserve(bt, seq, free, 1, np.array([9, 0]), bs)  # beyond the table
    assert out[2] == kv.BAD_INPUT and np.array_equal(out[0], bt)
    leak = np.array([[1, 4], [2, -1]], dtype=np.int32)       # entry to fill already holds a block
    assert kv.reserve(leak, seq, free, 1, np.array([2, 0]), bs)[2] == kv.BAD_INPUT
    r = kv.rollback(bt, seq, free, 1, np.array([1, 0]), np.array([3, 1]), bs)  # AL > K + 1
    assert r[4] == kv.BAD_INPUT and np.array_equal(r[0], bt) and np.array_equal(r[1], seq)
    hole = np.array([[1, -1], [2, -1]], dtype=np.int32)      # a block to free is missing
    r = kv.rollback(hole, seq, free, 1, np.array([3, 0]), np.array([1, 1]), bs)
    assert r[4] == kv.BAD_INPUT


def test_exactly_enough_free_blocks():
    """The free list holding exactly the blocks a reservation needs is enough
    (the stack empties); one block fewer is not.  The rollback that follows
    fills the stack back to its capacity, and one slot less of capacity is
    refused."""
    bs = 4
    bt = np.array([[1, -1, -1], [2, -1, -1]], dtype=np.int32)
    seq = np.array([4, 3], dtype=np.int32)
    free = np.array([7, 5, 6], dtype=np.int32)
    # request 0 needs blocks 1 and 2 (4 + 6 tokens), request 1 block 1 (3 + 3): 3 blocks, 3 free
    bt1, fc1, st = kv.reserve(bt, seq, free, 3, np.array([6, 3]), bs)
    assert st == kv.OK and fc1 == 0
    assert list(bt1[0]) == [1, 7, 5] and list(bt1[1]) == [2, 6, -1]
    out = kv.reserve(bt, seq, free[:2], 2, np.array([6, 3]), bs)
    assert out[2] == kv.OUT_OF_BLOCKS and np.array_equal(out[0], bt) and out[1] == 2
    bt2, seq2, free2, fc2, st = kv.rollback(bt1, seq, free, fc1, np.array([6, 3]), np.array([1, 1]), bs)
    assert st == kv.OK and fc2 == 3 and list(free2) == [7, 5, 6]
    assert np.array_equal(bt2, bt) and np.array_equal(seq2, seq)
    r = kv.rollback(bt1, seq, free[:2], fc1, np.array([6, 3]), np.array([1, 1]), bs)
    assert r[4] == kv.BAD_INPUT and np.array_equal(r[0], bt1)

