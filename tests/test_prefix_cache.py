"""Automatic prefix caching in the allocator: the oracle's model pinned to the
pages' rules and to a brute-force definition, and the C++ allocator behind the
C ABI bit-identical to the model under random operation sequences.

Pages: the untitled Qwen2.5-7B deployment page (mhpq.cn/news/468822), section
3.2 (blocks of block_size tokens are cached by their token ids; a hit needs a
token-exact prefix aligned to block boundaries; a change in the first block
invalidates every later one); "LLM推理优化：vLLM PagedAttention深度解析与工程实践",
section 4.2 (reuse across requests, the worked two-request example).
"""
import os
import random

import numpy as np
import pytest

from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import build as pa_build

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "prefix_cache_example.txt")


def _golden():
    reqs, cases = {}, []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        f = line.split()
        if f[0].startswith("request_"):
            reqs[f[0]] = [int(x) for x in f[1:]]
        else:
            cases.append((int(f[0]), int(f[1])))
    return reqs, cases


# ---------------------------------------------------------------- model pins
def test_worked_example_from_the_page(oracle_mod):
    reqs, cases = _golden()
    assert len(cases) == 5
    for bs, expect in cases:
        m = oracle_mod.BlockManagerModel(64, bs)
        assert m.allocate_prompt(1, reqs["request_a"]) == 0
        assert m.allocate_prompt(2, reqs["request_b"]) == expect
        # the shared blocks are the same physical blocks, counted twice
        k = expect // bs
        assert m.allocated[1][:k] == m.allocated[2][:k]
        assert all(m.ref[b] == 2 for b in m.allocated[1][:k])
        assert not set(m.allocated[1][k:]) & set(m.allocated[2][k:])


def test_hit_rules(oracle_mod):
    bs = 4
    m = oracle_mod.BlockManagerModel(64, bs)
    base = list(range(100, 122))                     # 5 full blocks + 2 tokens
    assert m.allocate_prompt(0, base) == 0
    # identical prompt: every full block, never the partial last block
    assert m.allocate_prompt(1, base) == 20
    assert m.allocated[1][:5] == m.allocated[0][:5] and m.allocated[1][5] != m.allocated[0][5]
    # a varying token in front (a timestamp, a request id) breaks every block
    assert m.allocate_prompt(2, [7] + base) == 0
    # a change inside block k keeps exactly blocks 0..k-1
    for k in range(5):
        p = list(base)
        p[k * bs + 1] += 1000
        assert m.allocate_prompt(10 + k, p) == k * bs
    # a shared prefix of 2.5 blocks keeps 2 blocks
    assert m.allocate_prompt(20, base[:10] + [5, 5, 5, 5]) == 8
    # a prompt shorter than a block caches nothing
    assert m.allocate_prompt(21, base[:3]) == 0


def test_reuse_after_free_and_eviction(oracle_mod):
    bs, N = 4, 12
    m = oracle_mod.BlockManagerModel(N, bs)
    p = list(range(12))                              # 3 full blocks
    m.allocate_prompt(0, p)
    blocks = list(m.allocated[0])
    m.free(0)
    assert list(m.free_blocks)[-3:] == blocks        # freed, still cached
    assert m.prefix_stats()["cached_free"] == 3
    assert m.allocate_prompt(1, p) == 12             # revived from the free list
    assert m.allocated[1] == blocks and not set(blocks) & set(m.free_blocks)
    assert all(m.ref[b] == 1 for b in blocks)
    m.free(1)
    # hand out every free block once: the oldest freed go last, but all go
    m.allocate(2, (N - 0) * bs)
    st = m.prefix_stats()
    assert st["evicted"] == 3 and st["entries"] == 0
    m.free(2)
    assert m.allocate_prompt(3, p) == 0


def test_generated_tokens_are_cached_when_their_block_fills(oracle_mod):
    bs = 4
    m = oracle_mod.BlockManagerModel(32, bs)
    prompt = [1, 2, 3, 4, 5, 6]
    m.allocate_prompt(0, prompt)
    reply = [7, 8, 9, 10, 11]
    for t in reply:
        m.append_token(0, t)
    turn2 = prompt + reply + [12, 13, 14]
    # 11 tokens known: blocks [1..4], [5..8] and [9..11]+... -> two full blocks cached
    assert m.allocate_prompt(1, turn2) == 8
    assert m.allocated[1][:2] == m.allocated[0][:2]
    # an untracked append (token unknown) stops registering
    m.allocate_prompt(5, [50, 51, 52])
    m.append_slot(5)
    # registered: [1..4] and [5..8] by sequence 0, [9..12] by sequence 1, nothing by 5
    assert m.prefix_stats()["registered"] == 3


def _cached_prefixes_brute(history, bs):
    """Every block-aligned prefix whose tokens some live-or-freed sequence ever
    held in full blocks (no eviction happens in the calling test)."""
    out = set()
    for toks in history:
        for k in range(1, len(toks) // bs + 1):
            out.add(tuple(toks[: k * bs]))
    return out


@pytest.mark.parametrize("seed", range(6))
def test_hits_equal_the_longest_cached_block_prefix(oracle_mod, seed):
    rng = random.Random(seed)
    bs = rng.choice([2, 4, 8])
    m = oracle_mod.BlockManagerModel(4000, bs)       # large pool: no eviction
    stems = [[rng.randrange(4) for _ in range(rng.randrange(0, 40))] for _ in range(5)]
    history = []
    live = []
    for sid in range(60):
        stem = rng.choice(stems)
        p = stem[: rng.randrange(0, len(stem) + 1)] + [rng.randrange(4) for _ in range(rng.randrange(0, 12))]
        cached = _cached_prefixes_brute(history, bs)
        expect = max([k * bs for k in range(0, len(p) // bs + 1) if k == 0 or tuple(p[: k * bs]) in cached])
        assert m.allocate_prompt(sid, p) == expect
        toks = list(p)
        for _ in range(rng.randrange(0, 9)):
            t = rng.randrange(4)
            m.append_token(sid, t)
            toks.append(t)
        history.append(toks)
        live.append(sid)
        if live and rng.random() < 0.4:
            m.free(live.pop(rng.randrange(len(live))))
    # conservation and counts
    used = {b for s in m.allocated.values() for b in s}
    assert len(used) + len(m.free_blocks) == m.num_blocks
    for b in range(m.num_blocks):
        assert m.ref[b] == sum(t.count(b) for t in m.allocated.values())


# ----------------------------------------------------------- C++ vs the model
@pytest.fixture(scope="module")
def _built():
    pa_build.build()


def _same(cpp, model):
    assert cpp.free_list() == list(model.free_blocks)
    for b in range(model.num_blocks):
        assert cpp.block_ref(b) == model.ref[b]
    live = sorted(model.allocated)
    if live:
        w = max(len(model.allocated[s]) for s in live) + 1
        t1, l1 = cpp.export(live, w)
        t2, l2 = model.export(live, w)
        assert np.array_equal(t1, t2) and np.array_equal(l1, l2)
    assert cpp.prefix_stats() == model.prefix_stats()


def _both(fc, fm, oracle_mod):
    try:
        rm, em = fm(), None
    except oracle_mod.OracleOOM:
        rm, em = None, 2
    except oracle_mod.OracleInvalid:
        rm, em = None, 1
    try:
        rc, ec = fc(), None
    except binding.PaError as e:
        rc, ec = None, e.status
    if em is None:
        assert ec is None, ec
    elif em == 2:
        assert ec == 2
    else:
        assert ec in (1, 3)
    return rc, rm


@pytest.mark.parametrize("trial", range(10))
def test_cpp_allocator_matches_model_with_prefix_caching(_built, oracle_mod, trial):
    rng = random.Random(100 + trial)
    bs = rng.choice([2, 4, 8, 16])
    N = rng.randrange(8, 80)
    order = list(range(N))
    rng.shuffle(order)
    cpp = binding.Allocator(N, bs, np.asarray(order, np.int32))
    model = oracle_mod.BlockManagerModel(N, bs, order)
    stems = [[rng.randrange(3) for _ in range(rng.randrange(0, 5 * bs))] for _ in range(4)]
    next_id = 0
    for step in range(300):
        live = sorted(model.allocated)
        op = rng.random()
        if op < 0.3 or not live:
            stem = rng.choice(stems)
            p = stem[: rng.randrange(0, len(stem) + 1)] + [rng.randrange(3) for _ in range(rng.randrange(0, 2 * bs))]
            sid = next_id
            next_id += 1
            rc, rm = _both(lambda: cpp.alloc_prompt(sid, p), lambda: model.allocate_prompt(sid, p), oracle_mod)
            assert rc == rm
        elif op < 0.55:
            s = rng.choice(live)
            t = rng.randrange(3)
            rc, rm = _both(lambda: cpp.append_token(s, t), lambda: model.append_token(s, t), oracle_mod)
            assert rc == rm
        elif op < 0.65:
            ids = rng.sample(live, rng.randrange(1, len(live) + 1))
            toks = [rng.randrange(3) for _ in ids]
            rc, rm = _both(lambda: cpp.append_batch(ids, tokens=toks),
                           lambda: model.append_batch(ids, toks), oracle_mod)
            if rc is not None:
                assert rc[0].tolist() == list(rm[0])
                assert [tuple(x) for x in rc[1].tolist()] == list(rm[1])
        elif op < 0.7:
            s = rng.choice(live)
            rc, rm = _both(lambda: cpp.append_slot(s), lambda: model.append_slot(s), oracle_mod)
            assert rc == rm
        elif op < 0.75:
            s = rng.choice(live)
            n = model.lens[s] + rng.randrange(0, 2 * bs)
            _both(lambda: cpp.alloc(s, n), lambda: model.allocate(s, n), oracle_mod)
        elif op < 0.82:
            s = rng.choice(live)
            c = next_id
            next_id += 1
            _both(lambda: cpp.fork(s, c), lambda: model.fork(s, c), oracle_mod)
        else:
            s = rng.choice(live)
            _both(lambda: cpp.free(s), lambda: model.free(s), oracle_mod)
        _same(cpp, model)
    cpp.close()


def test_cpp_rejects_bad_prompt_calls(_built):
    a = binding.Allocator(8, 4)
    a.alloc_prompt(1, [1, 2, 3])
    with pytest.raises(binding.PaError):
        a.alloc_prompt(1, [1, 2, 3])                 # sequence exists
    with pytest.raises(binding.PaError) as e:
        a.alloc_prompt(2, list(range(100)))          # does not fit
    assert e.value.status == 2
    assert a.stats()["num_seqs"] == 1 and a.prefix_stats()["lookups"] == 0
    assert a.alloc_prompt(3, []) == 0
    a.close()
