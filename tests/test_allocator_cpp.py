"""The C++ allocator behind the C ABI against the oracle's allocator model:
the same operations give bit-identical tables, lengths, slots, copy pairs,
reference counts and free lists, and the same errors."""
import random

import numpy as np
import pytest

from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import build as pa_build


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()


ERR = {binding.PaError: None}


def _same_state(cpp, model, live):
    assert cpp.free_list() == list(model.free_blocks)
    for b in range(model.num_blocks):
        assert cpp.block_ref(b) == model.ref[b]
    if live:
        w = max(len(model.allocated[s]) for s in live) + 1
        t1, l1 = cpp.export(live, w)
        t2, l2 = model.export(live, w)
        assert np.array_equal(t1, t2) and np.array_equal(l1, l2)
    st = cpp.stats()
    ms = model.stats()
    for k in ("num_blocks", "free_blocks", "used_blocks", "shared_blocks", "num_seqs",
              "num_tokens"):
        assert st[k] == ms[k], k


def _apply(fn_cpp, fn_model, oracle_mod):
    """Runs both; both must succeed with equal results or fail the same way."""
    try:
        r2 = fn_model()
        e2 = None
    except oracle_mod.OracleOOM:
        r2, e2 = None, 2
    except oracle_mod.OracleInvalid:
        r2, e2 = None, "invalid"
    try:
        r1 = fn_cpp()
        e1 = None
    except binding.PaError as e:
        r1, e1 = None, e.status
    if e2 is None:
        assert e1 is None, e1
    elif e2 == 2:
        assert e1 == 2
    else:
        assert e1 in (1, 3)
    return r1, r2


@pytest.mark.parametrize("trial", range(12))
def test_random_operations_match_the_model(oracle_mod, trial):
    rnd = random.Random(100 + trial)
    N = rnd.choice([16, 48, 97])
    bs = rnd.choice([4, 8, 16, 32])
    order = np.random.default_rng(trial).permutation(N).astype(np.int32)
    cpp = binding.Allocator(N, bs, order)
    model = oracle_mod.BlockManagerModel(N, bs, order)
    nxt = 0
    for step in range(300):
        live = sorted(model.allocated)
        op = rnd.random()
        if op < 0.2 or not live:
            sid, n = nxt, rnd.randint(0, 3 * bs)
            nxt += 1
            _apply(lambda: cpp.alloc(sid, n), lambda: model.allocate(sid, n), oracle_mod)
        elif op < 0.45:
            sid = rnd.choice(live)
            r1, r2 = _apply(lambda: cpp.append_slot(sid), lambda: model.append_slot(sid),
                            oracle_mod)
            assert r1 == r2
        elif op < 0.6:
            batch = rnd.sample(live, rnd.randint(1, len(live)))
            r1, r2 = _apply(lambda: cpp.append_batch(batch), lambda: model.append_batch(batch),
                            oracle_mod)
            if r2 is not None:
                assert r1[0].tolist() == r2[0]
                assert [tuple(p) for p in r1[1].tolist()] == [tuple(p) for p in r2[1]]
        elif op < 0.72:
            parent = rnd.choice(live)
            child = nxt
            nxt += 1
            _apply(lambda: cpp.fork(parent, child), lambda: model.fork(parent, child), oracle_mod)
        elif op < 0.85:
            sid = rnd.choice(live)
            _apply(lambda: cpp.free(sid), lambda: model.free(sid), oracle_mod)
        else:
            sid = rnd.choice(live)
            n = model.lens[sid] + rnd.randint(0, 2 * bs)
            _apply(lambda: cpp.alloc(sid, n), lambda: model.allocate(sid, n), oracle_mod)
        _same_state(cpp, model, sorted(model.allocated))
    # slots of every live sequence's positions agree
    for sid in sorted(model.allocated):
        n = model.lens[sid]
        assert cpp.seq_slots(sid, 0, n).tolist() == [model.slot_of(sid, t) for t in range(n)]
    cpp.close()


def test_errors_leave_state_unchanged(oracle_mod):
    cpp = binding.Allocator(4, 16)
    cpp.alloc(1, 48)
    before = (cpp.free_list(), cpp.export([1], 4))
    with pytest.raises(binding.PaError) as e:
        cpp.alloc(2, 32)
    assert e.value.status == 2
    with pytest.raises(binding.PaError) as e:
        cpp.free(7)
    assert e.value.status == 3
    with pytest.raises(binding.PaError) as e:
        cpp.fork(1, 1)
    assert e.value.status == 1
    with pytest.raises(binding.PaError) as e:
        cpp.append_batch([1, 1])
    assert e.value.status == 1
    after = (cpp.free_list(), cpp.export([1], 4))
    assert before[0] == after[0] and np.array_equal(before[1][0], after[1][0])
    with pytest.raises(binding.PaError):
        binding.Allocator(4, 16, [0, 1, 1, 2])          # not a permutation


def test_pages_worked_table_through_the_abi():
    phys = [47, 23, 89]
    order = phys + [b for b in range(96) if b not in phys]
    a = binding.Allocator(96, 16, order)
    a.alloc(0, 40)
    tbl, lens = a.export([0], 3)
    assert tbl[0].tolist() == phys and lens[0] == 40
    assert a.append_slot(0) == (1432, None)


def test_prefix_share_cow_counts_through_the_abi():
    for prefix, expected in ((1024, 0), (1000, 255)):
        a = binding.Allocator(400, 16)
        a.alloc(0, prefix)
        for s in range(1, 256):
            a.fork(0, s)
        slots, pairs = a.append_batch(list(range(256)))
        assert len(pairs) == expected and len(set(slots.tolist())) == 256
