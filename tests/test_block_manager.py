"""Host tests of the block manager: allocation, sharing, copy-on-write, reclamation."""
import json
import os

import numpy as np
import pytest

from paged_kv_cache_242_gb300.block_manager import BlockManager, OutOfBlocks


def _invariants(m: BlockManager):
    refs = np.zeros(m.num_blocks, dtype=np.int64)
    for table in m.tables.values():
        for b in table:
            refs[b] += 1
    assert np.array_equal(refs, m.refcount), "refcount must equal the number of table references"
    free = list(m._free)
    assert len(free) == len(set(free)), "a block is twice on the free list"
    assert all(m.refcount[b] == 0 for b in free), "a referenced block is on the free list"
    assert len(free) + int((m.refcount > 0).sum()) == m.num_blocks, "a block leaked"
    for s, table in m.tables.items():
        assert len(table) == -(-m.lengths[s] // m.block_size)


def test_seven_token_example(golden_dir):
    with open(os.path.join(golden_dir, "seven_token_example.json")) as f:
        g = json.load(f)
    m = BlockManager(8, g["block_size"])
    m.add_sequence(0, g["prefill_tokens"])
    assert len(m.tables[0]) == g["blocks_after_prefill"]
    m.append_slot(0)  # token 8 fills the spare slot
    assert len(m.tables[0]) == g["blocks_after_token_8"]
    m.append_slot(0)  # token 9: the previous block is full
    assert len(m.tables[0]) == g["blocks_after_token_9"]
    _invariants(m)


def test_slots_follow_the_block_table():
    m = BlockManager(50, 16, free_order=np.random.default_rng(0).permutation(50))
    slots = m.add_sequence(7, 37)
    for _ in range(30):
        slots.append(m.append_slot(7)[0])
    table = m.tables[7]
    for pos, slot in enumerate(slots):
        assert slot // 16 == table[pos // 16] and slot % 16 == pos % 16
    _invariants(m)


def test_fork_copy_on_write_and_isolation():
    m = BlockManager(10, 4)
    m.add_sequence(0, 6)  # blocks: full + partial (2 of 4)
    m.fork(0, 1)
    shared_last = m.tables[0][-1]
    assert m.refcount[shared_last] == 2
    slot, cow = m.append_slot(1)  # child writes into the shared partial block
    assert cow is not None and cow[0] == shared_last
    assert m.tables[1][-1] == cow[1] != shared_last
    assert slot == cow[1] * 4 + 2
    assert m.refcount[shared_last] == 1 and m.refcount[cow[1]] == 1
    assert m.tables[1][0] == m.tables[0][0] and m.refcount[m.tables[0][0]] == 2
    slot0, cow0 = m.append_slot(0)  # the parent is now sole owner: writes in place
    assert cow0 is None and slot0 == shared_last * 4 + 2
    _invariants(m)


def test_last_writer_writes_in_place():
    """With k sharers of a partial block, k - 1 copies happen and the last writes in place."""
    m = BlockManager(40, 32)
    m.add_sequence(0, 1040)  # 32 full blocks + one block of 16
    for j in range(1, 8):
        m.fork(0, j)
    pairs = [m.append_slot(s)[1] for s in range(8)]
    copies = [p for p in pairs if p is not None]
    assert len(copies) == 7 and len({p[1] for p in copies}) == 7
    assert all(p[0] == copies[0][0] for p in copies)
    assert pairs[7] is None
    _invariants(m)


def test_no_copy_when_prompt_fills_whole_blocks():
    m = BlockManager(300, 32)
    m.add_sequence(0, 1024)
    for j in range(1, 8):
        m.fork(0, j)
    assert all(m.append_slot(s)[1] is None for s in range(8))
    _invariants(m)


def test_free_releases_only_at_zero():
    m = BlockManager(6, 4)
    m.add_sequence(0, 8)
    m.fork(0, 1)
    m.append_slot(1)  # new private block for the child
    before = m.num_free
    m.free(0)  # shared blocks stay: the child still maps them
    assert m.num_free == before
    assert all(m.refcount[b] == 1 for b in m.tables[1])
    m.free(1)
    assert m.num_free == 6
    _invariants(m)


def test_out_of_blocks_and_no_reuse_of_live_blocks():
    m = BlockManager(3, 2)
    m.add_sequence(0, 5)
    live = set(m.tables[0])
    with pytest.raises(OutOfBlocks):
        m.add_sequence(1, 3)
    assert 1 not in m.tables
    m.append_slot(0)  # position 5 fits in the third block
    with pytest.raises(OutOfBlocks):
        m.append_slot(0)
    assert set(m.tables[0]) == live
    m.free(0)
    m.add_sequence(2, 6)
    _invariants(m)


def test_random_fork_append_free_keeps_invariants():
    """Beam-search-like churn: forks, appends, frees in random order."""
    rng = np.random.default_rng(3)
    m = BlockManager(400, 4, free_order=rng.permutation(400))
    m.add_sequence(0, 9)
    alive, next_id = [0], 1
    for _ in range(2000):
        op = rng.integers(3)
        if op == 0 and len(alive) < 12:
            parent = alive[rng.integers(len(alive))]
            m.fork(parent, next_id)
            alive.append(next_id)
            next_id += 1
        elif op == 1:
            s = alive[rng.integers(len(alive))]
            try:
                before = list(m.tables[s])
                slot, cow = m.append_slot(s)
                if cow is not None:
                    assert cow[0] == before[-1]
            except OutOfBlocks:
                pass
        elif len(alive) > 1:
            s = alive.pop(rng.integers(len(alive)))
            m.free(s)
        _invariants(m)


def test_block_table_array_and_lengths():
    m = BlockManager(10, 4, free_order=[9, 8, 7, 6, 5, 4, 3, 2, 1, 0])
    m.add_sequence(0, 5)
    m.add_sequence(1, 0)
    bt = m.block_table_array([0, 1], pad=-1)
    assert bt.dtype == np.int32 and bt.tolist() == [[9, 8], [-1, -1]]
    assert m.seq_lens_array([0, 1]).tolist() == [5, 0]
    with pytest.raises(ValueError):
        m.block_table_array([0], max_blocks=1)
