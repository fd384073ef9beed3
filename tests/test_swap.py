"""Swap space in the allocator: the oracle's model pinned to its rules and to
data preservation through plain copies, and the C++ allocator bit-identical
to the model under random operation sequences that include swaps.

Pages: "LLM推理优化：vLLM PagedAttention深度解析与工程实践", section 3.2 (an
allocation that finds too few free blocks calls for swap or preemption);
"vLLM推理加速深度解析：从PagedAttention原理到生产部署实战", section 4 (swap space
moves KV cache to CPU memory).
"""
import random

import numpy as np
import pytest
import torch

from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import build as pa_build
from paged_kv_cache_103_gb300 import workloads as wl


def test_swap_rules(oracle_mod):
    m = oracle_mod.BlockManagerModel(8, 4, [3, 1, 4, 0, 5, 2, 7, 6])
    m.set_swap_pool(5)
    m.allocate(0, 9)                                  # blocks 3 1 4
    m.allocate(1, 3)                                  # block 0
    pairs = m.swap_out(0)
    assert pairs == [(3, 0), (1, 1), (4, 2)]
    assert list(m.free_blocks) == [5, 2, 7, 6, 3, 1, 4]
    assert list(m.host_free) == [3, 4]
    with pytest.raises(oracle_mod.OracleInvalid):
        m.append_slot(0)                              # swapped: no appends
    with pytest.raises(oracle_mod.OracleInvalid):
        m.export([0])
    with pytest.raises(oracle_mod.OracleOOM):
        m.allocate(2, 4 * 7 + 1)                      # needs 8 > 7 free
    m.allocate(2, 4 * 6)                              # 6 of 7 free blocks
    with pytest.raises(oracle_mod.OracleOOM):
        m.swap_in(0)                                  # needs 3, one free
    assert 0 in m.swapped and list(m.host_free) == [3, 4]   # unchanged
    m.free(2)
    back = m.swap_in(0)
    assert [h for h, _ in back] == [0, 1, 2]
    assert m.allocated[0] == [d for _, d in back] and m.lens[0] == 9
    assert list(m.host_free) == [3, 4, 0, 1, 2]
    # a freed swapped sequence returns its host blocks
    m.swap_out(1)
    m.free(1)
    assert list(m.host_free) == [4, 0, 1, 2, 3]


def test_swap_out_of_a_shared_block(oracle_mod):
    m = oracle_mod.BlockManagerModel(10, 4)
    m.set_swap_pool(10)
    m.allocate(0, 6)
    m.fork(0, 1)
    shared = list(m.allocated[0])
    m.swap_out(1)
    assert all(m.ref[b] == 1 for b in shared)          # the sharer keeps them
    assert not set(shared) & set(m.free_blocks)
    m.swap_in(1)
    assert not set(m.allocated[1]) & set(shared)       # private after swap-in
    m.append_slot(1)                                   # no copy-on-write needed now
    assert m.ref[m.allocated[1][-1]] == 1


def test_swap_preserves_what_decode_reads(oracle_mod):
    """Blocks swapped out, the device blocks reused and overwritten, then
    swapped in: the decode through the new table equals the decode before,
    bit for bit (plain copies only)."""
    bs, N, Hkv, d, H = 8, 40, 2, 64, 4
    m = oracle_mod.BlockManagerModel(N, bs, np.random.default_rng(0).permutation(N))
    m.set_swap_pool(30)
    lens = [21, 40, 9]
    for i, n in enumerate(lens):
        m.allocate(i, n)
    kc = wl.normal_tensor((N, bs, Hkv, d), torch.float16, 1)
    vc = wl.normal_tensor((N, bs, Hkv, d), torch.float16, 2)
    q = wl.normal_tensor((3, H, d), torch.float16, 3)
    tbl, ln = m.export(range(3))
    before = oracle_mod.decode(wl.bits(q), wl.bits(kc), wl.bits(vc), tbl, ln, 0.125,
                               oracle_mod.DTYPE_F16)
    hk = torch.zeros(30, bs, Hkv, d, dtype=torch.float16)
    hv = torch.zeros_like(hk)
    for s in (0, 2):
        oracle_mod.swap_blocks([kc, vc], [hk, hv], m.swap_out(s))
    m.allocate(7, N * bs // 2)                         # reuse the freed blocks ...
    for b in m.allocated[7]:
        kc[b] = float("nan")                           # ... and overwrite them
        vc[b] = float("nan")
    m.free(7)
    for s in (2, 0):
        oracle_mod.swap_blocks([hk, hv], [kc, vc], m.swap_in(s))
    tbl2, ln2 = m.export(range(3))
    assert not np.array_equal(tbl2, tbl)
    after = oracle_mod.decode(wl.bits(q), wl.bits(kc), wl.bits(vc), tbl2, ln2, 0.125,
                              oracle_mod.DTYPE_F16)
    assert np.array_equal(before, after)


# ----------------------------------------------------------- C++ vs the model
@pytest.fixture(scope="module")
def _built():
    pa_build.build()


def _same(cpp, model):
    assert cpp.free_list() == list(model.free_blocks)
    assert cpp.host_free_list() == list(model.host_free)
    for b in range(model.num_blocks):
        assert cpp.block_ref(b) == model.ref[b]
    live = sorted(s for s in model.allocated if s not in model.swapped)
    if live:
        w = max(len(model.allocated[s]) for s in live) + 1
        t1, l1 = cpp.export(live, w)
        t2, l2 = model.export(live, w)
        assert np.array_equal(t1, t2) and np.array_equal(l1, l2)
    st = cpp.swap_stats()
    assert st["swapped_seqs"] == len(model.swapped) and st["host_free"] == len(model.host_free)
    assert cpp.stats()["num_tokens"] == model.stats()["num_tokens"]


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
def test_cpp_allocator_matches_model_with_swaps(_built, oracle_mod, trial):
    rng = random.Random(300 + trial)
    bs = rng.choice([4, 8, 16])
    N = rng.randrange(8, 60)
    H = rng.randrange(0, 50)
    order = list(range(N))
    rng.shuffle(order)
    cpp = binding.Allocator(N, bs, np.asarray(order, np.int32))
    model = oracle_mod.BlockManagerModel(N, bs, order)
    cpp.set_swap_pool(H)
    model.set_swap_pool(H)
    nxt = 0
    for _ in range(300):
        seqs = sorted(model.allocated)
        op = rng.random()
        if op < 0.2 or not seqs:
            n = rng.randrange(0, 4 * bs)
            s, nxt = nxt, nxt + 1
            _both(lambda: cpp.alloc(s, n), lambda: model.allocate(s, n), oracle_mod)
        elif op < 0.4:
            s = rng.choice(seqs)
            rc, rm = _both(lambda: cpp.append_slot(s), lambda: model.append_slot(s), oracle_mod)
            assert rc == rm
        elif op < 0.55:
            s = rng.choice(seqs)
            rc, rm = _both(lambda: cpp.swap_out(s), lambda: model.swap_out(s), oracle_mod)
            if rm is not None:
                assert [tuple(p) for p in rc.tolist()] == rm
        elif op < 0.7:
            s = rng.choice(seqs)
            rc, rm = _both(lambda: cpp.swap_in(s), lambda: model.swap_in(s), oracle_mod)
            if rm is not None:
                assert [tuple(p) for p in rc.tolist()] == rm
        elif op < 0.8:
            s = rng.choice(seqs)
            c, nxt = nxt, nxt + 1
            _both(lambda: cpp.fork(s, c), lambda: model.fork(s, c), oracle_mod)
        elif op < 0.85:
            ids = rng.sample(seqs, rng.randrange(1, len(seqs) + 1))
            rc, rm = _both(lambda: cpp.append_batch(ids), lambda: model.append_batch(ids),
                           oracle_mod)
            if rm is not None:
                assert rc[0].tolist() == list(rm[0])
        else:
            s = rng.choice(seqs)
            _both(lambda: cpp.free(s), lambda: model.free(s), oracle_mod)
        _same(cpp, model)
    cpp.close()
