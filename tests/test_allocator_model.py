"""Pins for the allocator model in the oracle, against the pages.

The model restates the BlockManager of "LLM推理优化：vLLM PagedAttention深度
解析与工程实践" section 3.2 (free list taken from the front, returned to the
back in table order, all-or-nothing allocate) and the BlockSpaceManager of
"vLLM 深度拆解：当大模型推理学会「分页注意力」" section 3.3 (append_slot,
free, copy-on-write sharing).  These tests pin each rule to its page and check
the invariants the pages state (no fragment larger than one block per
sequence; freed blocks reusable by anyone; forks copy only the table).
"""
import os
import random

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_free_list_front_and_back_order(oracle_mod):
    m = oracle_mod.BlockManagerModel(8, 16)
    m.allocate(1, 20)                       # ceil(20/16) = 2 blocks from the front
    m.allocate(2, 16)
    assert m.allocated[1] == [0, 1] and m.allocated[2] == [2]
    m.free(1)                               # back of the list, in table order
    assert list(m.free_blocks) == [3, 4, 5, 6, 7, 0, 1]
    m.allocate(3, 40)
    assert m.allocated[3] == [3, 4, 5]


def test_allocate_guard_and_incremental_growth(oracle_mod):
    m = oracle_mod.BlockManagerModel(8, 16)
    m.allocate(1, 20)
    m.allocate(1, 10)                       # already holds 32 slots >= 10: no change
    assert m.allocated[1] == [0, 1] and m.lens[1] == 20
    m.allocate(1, 33)                       # needs ceil((33 - 32) / 16) = 1 more
    assert m.allocated[1] == [0, 1, 2] and m.lens[1] == 33


def test_oom_is_all_or_nothing(oracle_mod):
    m = oracle_mod.BlockManagerModel(4, 16)
    m.allocate(1, 48)
    before = (list(m.free_blocks), {k: list(v) for k, v in m.allocated.items()}, list(m.ref))
    with pytest.raises(oracle_mod.OracleOOM):
        m.allocate(2, 32)
    assert (list(m.free_blocks), {k: list(v) for k, v in m.allocated.items()}, list(m.ref)) == before
    assert 2 not in m.allocated


def test_pages_worked_table_next_slot(oracle_mod):
    rows, meta = [], {}
    with open(os.path.join(GOLDEN, "block_table_example.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                p = line.split()
                (rows.append([int(x) for x in p]) if p[0].isdigit() else meta.update({p[0]: int(p[1])}))
    phys = [r[1] for r in rows]
    N = 96
    order = phys + [b for b in range(N) if b not in phys]
    m = oracle_mod.BlockManagerModel(N, meta["block_size"], order)
    m.allocate(0, meta["context_len"])
    tbl, lens = m.export([0])
    assert tbl[0].tolist() == phys and lens[0] == 40
    slot, cow = m.append_slot(0)
    assert slot == meta["next_slot"] == 1432 and cow is None
    # internal fragmentation stays under one block
    assert len(m.allocated[0]) * 16 - m.lens[0] < 16


def test_pages_diagram_slots(oracle_mod):
    N = 32
    order = [7, 3, 21] + [b for b in range(N) if b not in (7, 3, 21)]
    m = oracle_mod.BlockManagerModel(N, 16, order)
    m.allocate(0, 48)
    assert m.allocated[0] == [7, 3, 21]
    assert [m.slot_of(0, t) for t in (0, 15, 16, 31, 32, 47)] == [112, 127, 48, 63, 336, 351]


def test_append_slot_fills_then_takes_new_block(oracle_mod):
    m = oracle_mod.BlockManagerModel(4, 4)
    m.allocate(0, 0)
    slots = [m.append_slot(0)[0] for _ in range(9)]
    assert slots == [0, 1, 2, 3, 4, 5, 6, 7, 8]
    assert m.allocated[0] == [0, 1, 2]


def test_fork_shares_and_cow_copies_on_write(oracle_mod):
    m = oracle_mod.BlockManagerModel(8, 16)
    m.allocate(0, 20)                       # blocks 0 (full), 1 (4 slots)
    m.fork(0, 1)
    assert m.allocated[1] == [0, 1] and m.ref[0] == 2 and m.ref[1] == 2
    slot, cow = m.append_slot(1)            # child writes into shared block 1 -> copy
    assert cow == (1, 2) and slot == 2 * 16 + 4 and m.allocated[1] == [0, 2]
    assert m.ref[1] == 1 and m.ref[2] == 1 and m.ref[0] == 2
    slot, cow = m.append_slot(0)            # parent is now the only holder: in place
    assert cow is None and slot == 1 * 16 + 4
    m.free(0)
    assert m.ref[0] == 1 and 1 in m.free_blocks and 0 not in m.free_blocks
    m.free(1)
    assert sorted(m.free_blocks) == list(range(8))


def test_prefix_sharing_copy_counts(oracle_mod):
    """256 sharers of a block-aligned prefix append without copies; with a
    1000-token prefix (62 full blocks + 8 slots) the first 255 appenders copy
    the partial block and the last writes in place."""
    for prefix, expected in ((1024, 0), (1000, 255)):
        m = oracle_mod.BlockManagerModel(400, 16)
        m.allocate(0, prefix)
        for s in range(1, 256):
            m.fork(0, s)
        shared = m.stats()["shared_blocks"]
        assert shared == (prefix + 15) // 16
        slots, pairs = m.append_batch(range(256))
        assert len(pairs) == expected
        assert len(set(slots)) == 256
        if expected:
            src = {p[0] for p in pairs}
            assert len(src) == 1 and m.ref[next(iter(src))] == 1


def test_batch_oom_is_all_or_nothing(oracle_mod):
    m = oracle_mod.BlockManagerModel(3, 4)
    m.allocate(0, 4)
    m.allocate(1, 4)
    m.allocate(2, 3)
    with pytest.raises(oracle_mod.OracleOOM):
        m.append_batch([2, 0, 1])           # 0 and 1 need new blocks; none free
    assert m.lens == {0: 4, 1: 4, 2: 3}


def _check_invariants(m):
    N, bs = m.num_blocks, m.block_size
    counts = [0] * N
    for s, t in m.allocated.items():
        assert len(t) == (m.lens[s] + bs - 1) // bs        # fragment < one block
        for b in t:
            counts[b] += 1
    assert counts == m.ref
    used = sum(1 for r in m.ref if r > 0)
    assert used + len(m.free_blocks) == N
    assert all(m.ref[b] == 0 for b in m.free_blocks)
    assert len(set(m.free_blocks)) == len(m.free_blocks)


def test_random_operation_sequences_keep_invariants(oracle_mod):
    rnd = random.Random(11)
    for trial in range(20):
        bs = rnd.choice([4, 8, 16])
        m = oracle_mod.BlockManagerModel(64, bs, np.random.default_rng(trial).permutation(64))
        nxt = 0
        for _ in range(400):
            live = list(m.allocated)
            op = rnd.random()
            try:
                if op < 0.25 or not live:
                    m.allocate(nxt, rnd.randint(0, 40))
                    nxt += 1
                elif op < 0.6:
                    m.append_slot(rnd.choice(live))
                elif op < 0.7:
                    m.fork(rnd.choice(live), nxt)
                    nxt += 1
                elif op < 0.85:
                    m.free(rnd.choice(live))
                else:
                    s = rnd.choice(live)
                    m.allocate(s, m.lens[s] + rnd.randint(0, 20))
            except (oracle_mod.OracleOOM, oracle_mod.OracleInvalid):
                pass
            _check_invariants(m)
