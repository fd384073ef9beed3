"""Pins for the fp64 decode oracle, against facts that do not come from it.

Each test checks the oracle against something independent: exact element
conversions from numpy / torch, closed forms of softmax attention, a library
attention routine on contiguous K/V, the worked block tables printed on the
pages, and invariants of paging (placement, sharing).  A plausible mistake in
the oracle -- a dropped or wrong scale, a wrong head mapping, a wrong table
index, a missing max-subtraction or normalisation -- fails at least one.
"""
import math
import os

import numpy as np
import pytest
import torch

from paged_kv_cache_103_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F16, BF16 = 0, 1


def _bits(t):
    return wl.bits(t)


def _table_from_blocks(blocks_per_seq, width):
    tbl = np.full((len(blocks_per_seq), width), -1, dtype=np.int32)
    for i, b in enumerate(blocks_per_seq):
        tbl[i, : len(b)] = b
    return tbl


def _contiguous_reference(q, K, V, scale, G):
    """torch SDPA (fp64, CPU) on contiguous K/V for one sequence.

    q: [H, d], K/V: [n, Hkv, d] (float64).  Query head h reads KV head h // G.
    """
    qt = torch.from_numpy(q)[:, None, :]                                  # [H, 1, d]
    Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [H, n, d]
    Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0)
    out = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    return out[:, 0, :].numpy()


# ---------------------------------------------------------------- conversions
def test_fp16_conversion_matches_numpy_for_every_pattern(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.to_double(pats, F16)
    ref = pats.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_bf16_conversion_matches_torch_for_every_pattern(oracle_mod):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.to_double(pats, BF16)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_known_patterns(oracle_mod):
    assert oracle_mod.to_double(np.array([0x3C00, 0xC000, 0x0001, 0x7BFF], np.uint16),
                                F16).tolist() == [1.0, -2.0, 2.0 ** -24, 65504.0]
    assert oracle_mod.to_double(np.array([0x3F80, 0x4049, 0x0001], np.uint16),
                                BF16).tolist() == [1.0, 3.140625, 2.0 ** -133]


# ---------------------------------------------------------------- closed forms
def _single_seq_case(n, H=4, Hkv=2, d=64, bs=16, dtype=torch.float16, seed=0):
    nb = (n + bs - 1) // bs
    N = nb + 3
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(1, H, d, generator=g).to(dtype)
    kc = torch.randn(N, bs, Hkv, d, generator=g).to(dtype)
    vc = torch.randn(N, bs, Hkv, d, generator=g).to(dtype)
    blocks = list(np.random.default_rng(seed).permutation(N)[:nb])
    tbl = _table_from_blocks([blocks], nb)
    return q, kc, vc, tbl, blocks


def test_single_token_returns_v0_exactly(oracle_mod):
    q, kc, vc, tbl, blocks = _single_seq_case(1)
    out = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), tbl, np.array([1]), 0.125, F16)
    v0 = vc[blocks[0], 0].double().numpy()                       # [Hkv, d]
    for h in range(4):
        assert np.array_equal(out[0, h], v0[h // 2])


def test_equal_keys_give_mean_of_v(oracle_mod):
    n = 37
    q, kc, vc, tbl, blocks = _single_seq_case(n, seed=1)
    kc[:] = kc[blocks[0], 0]                                      # every key row identical
    out = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), tbl, np.array([n]), 0.125, F16)
    rows = [vc[blocks[j // 16], j % 16].double().numpy() for j in range(n)]
    mean = np.mean(np.stack(rows), axis=0)                        # [Hkv, d]
    for h in range(4):
        np.testing.assert_allclose(out[0, h], mean[h // 2], rtol=0, atol=1e-14)


def test_two_tokens_logistic_closed_form(oracle_mod):
    """q = a e0, k_j = b_j e0 -> logits scale*a*b_j; w0 = 1 / (1 + exp(s1 - s0))."""
    d, bs = 64, 16
    scale = 1.0 / math.sqrt(d)
    a, b0, b1 = 1.5, 2.0, -0.75
    q = torch.zeros(1, 1, d, dtype=torch.float16)
    q[0, 0, 0] = a
    kc = torch.zeros(1, bs, 1, d, dtype=torch.float16)
    kc[0, 0, 0, 0], kc[0, 1, 0, 0] = b0, b1
    vc = torch.zeros(1, bs, 1, d, dtype=torch.float16)
    vc[0, 0, 0, :] = 1.0
    vc[0, 1, 0, :] = -3.0
    out = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), np.array([[0]], np.int32),
                            np.array([2]), scale, F16)
    w0 = 1.0 / (1.0 + math.exp(scale * a * (b1 - b0)))
    np.testing.assert_allclose(out[0, 0], w0 * 1.0 + (1.0 - w0) * -3.0, rtol=1e-15)


def test_one_dominant_logit_selects_its_row(oracle_mod):
    """A logit 60 above the rest gives that row within exp(-60)."""
    d, bs, n = 64, 16, 20
    q = torch.zeros(1, 1, d, dtype=torch.bfloat16)
    q[0, 0, 3] = 8.0
    kc = torch.zeros(2, bs, 1, d, dtype=torch.bfloat16)
    kc[1, 2, 0, 3] = 60.0                                          # token 16 + 2 = 18
    g = torch.Generator().manual_seed(3)
    vc = torch.randn(2, bs, 1, d, generator=g).to(torch.bfloat16)
    out = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), np.array([[0, 1]], np.int32),
                            np.array([n]), 1.0 / 8.0, BF16)
    np.testing.assert_allclose(out[0, 0], vc[1, 2, 0].double().numpy(), atol=1e-20)


def test_gqa_head_mapping_is_contiguous_groups(oracle_mod):
    """KV head g holds the constant value g+1 in V, so out[h] = h // G + 1."""
    H, Hkv, d, bs, n = 8, 4, 64, 16, 19
    g = torch.Generator().manual_seed(4)
    q = torch.randn(1, H, d, generator=g).to(torch.float16)
    kc = torch.randn(2, bs, Hkv, d, generator=g).to(torch.float16)
    vc = torch.empty(2, bs, Hkv, d, dtype=torch.float16)
    for kv in range(Hkv):
        vc[:, :, kv, :] = kv + 1
    out = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), np.array([[1, 0]], np.int32),
                            np.array([n]), 0.125, F16)
    for h in range(H):
        np.testing.assert_allclose(out[0, h], h // (H // Hkv) + 1, rtol=1e-15)


def test_softmax_weights_sum_to_one_and_ones_in_ones_out(oracle_mod):
    n = 150
    q, kc, vc, tbl, blocks = _single_seq_case(n, seed=5)
    for h in range(4):
        w = oracle_mod.weights(_bits(q), _bits(kc), tbl, np.array([n]), 0.125, F16, 0, h)
        assert abs(w.sum() - 1.0) < 1e-12 and (w > 0).all()
    ones = torch.ones_like(vc)
    out = oracle_mod.decode(_bits(q), _bits(kc), _bits(ones), tbl, np.array([n]), 0.125, F16)
    np.testing.assert_allclose(out, 1.0, rtol=1e-14)


def test_large_logits_need_max_subtraction(oracle_mod):
    """Logits near 1000 overflow exp() unless the max is subtracted first."""
    d, bs = 64, 16
    q = torch.zeros(1, 1, d, dtype=torch.bfloat16)
    q[0, 0, 0] = 256.0
    kc = torch.zeros(1, bs, 1, d, dtype=torch.bfloat16)
    kc[0, 0, 0, 0], kc[0, 1, 0, 0] = 32.0, 31.5                   # logits 1024, 1008
    vc = torch.zeros(1, bs, 1, d, dtype=torch.bfloat16)
    vc[0, 0, 0, :], vc[0, 1, 0, :] = 1.0, 0.0
    out = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), np.array([[0]], np.int32),
                            np.array([2]), 1.0 / 8.0, BF16)
    w0 = 1.0 / (1.0 + math.exp(-16.0))
    np.testing.assert_allclose(out[0, 0], w0, rtol=1e-15)


def test_empty_context_gives_zeros(oracle_mod):
    q, kc, vc, tbl, _ = _single_seq_case(5)
    out = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), tbl, np.array([0]), 0.125, F16)
    assert np.array_equal(out, np.zeros_like(out))


def test_rejects_out_of_pool_block(oracle_mod):
    q, kc, vc, tbl, _ = _single_seq_case(5)
    bad = tbl.copy()
    bad[0, 0] = kc.shape[0]
    with pytest.raises(ValueError):
        oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), bad, np.array([5]), 0.125, F16)


# ------------------------------------------------- library routine on contiguous K/V
@pytest.mark.parametrize("H,Hkv,d,bs,dtype", [(4, 2, 64, 16, torch.float16),
                                              (8, 8, 128, 8, torch.float16),
                                              (28, 4, 128, 32, torch.bfloat16),
                                              (32, 8, 128, 16, torch.bfloat16)])
def test_matches_sdpa_on_gathered_contiguous_kv(oracle_mod, H, Hkv, d, bs, dtype):
    rng = np.random.default_rng(H * 1000 + bs)
    B = 3
    lens = rng.integers(1, 5 * bs + 3, size=B).astype(np.int32)
    nbs = [(int(n) + bs - 1) // bs for n in lens]
    N = sum(nbs) + 4
    perm = rng.permutation(N)
    blocks, off = [], 0
    for nb in nbs:
        blocks.append(list(perm[off: off + nb]))
        off += nb
    tbl = _table_from_blocks(blocks, max(nbs))
    g = torch.Generator().manual_seed(int(H + d + bs))
    q = torch.randn(B, H, d, generator=g).to(dtype)
    kc = torch.randn(N, bs, Hkv, d, generator=g).to(dtype)
    vc = torch.randn(N, bs, Hkv, d, generator=g).to(dtype)
    scale = 1.0 / math.sqrt(d)
    code = F16 if dtype == torch.float16 else BF16
    out = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), tbl, lens, scale, code, num_threads=2)
    for i in range(B):
        n = int(lens[i])
        K = np.stack([kc[blocks[i][j // bs], j % bs].double().numpy() for j in range(n)])
        V = np.stack([vc[blocks[i][j // bs], j % bs].double().numpy() for j in range(n)])
        ref = _contiguous_reference(q[i].double().numpy(), K, V, scale, H // Hkv)
        np.testing.assert_allclose(out[i], ref, rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------ paging invariants
def _place(logical_k, logical_v, blocks, N, bs):
    """Write a sequence's logical rows [n, Hkv, d] into a pool through ``blocks``."""
    n, Hkv, d = logical_k.shape
    kc = torch.zeros(N, bs, Hkv, d, dtype=logical_k.dtype)
    vc = torch.zeros_like(kc)
    for j in range(n):
        kc[blocks[j // bs], j % bs] = logical_k[j]
        vc[blocks[j // bs], j % bs] = logical_v[j]
    return kc, vc


def test_permuting_physical_blocks_is_bit_identical(oracle_mod):
    bs, n, N = 16, 77, 12
    g = torch.Generator().manual_seed(7)
    K = torch.randn(n, 2, 64, generator=g).to(torch.float16)
    V = torch.randn(n, 2, 64, generator=g).to(torch.float16)
    q = torch.randn(1, 4, 64, generator=g).to(torch.float16)
    outs = []
    for seed in range(3):
        blocks = list(np.random.default_rng(seed).permutation(N)[:5])
        kc, vc = _place(K, V, blocks, N, bs)
        outs.append(oracle_mod.decode(_bits(q), _bits(kc), _bits(vc),
                                      _table_from_blocks([blocks], 5), np.array([n]), 0.125, F16))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_shared_prefix_equals_private_copies(oracle_mod):
    bs, N = 16, 20
    g = torch.Generator().manual_seed(8)
    kc = torch.randn(N, bs, 2, 64, generator=g).to(torch.bfloat16)
    vc = torch.randn(N, bs, 2, 64, generator=g).to(torch.bfloat16)
    q = torch.randn(2, 4, 64, generator=g).to(torch.bfloat16)
    shared = [[0, 1, 2, 5], [0, 1, 2, 6]]                          # blocks 0..2 shared
    kc2, vc2 = kc.clone(), vc.clone()
    for src, dst in [(0, 10), (1, 11), (2, 12)]:
        kc2[dst], vc2[dst] = kc[src], vc[src]
    copied = [[0, 1, 2, 5], [10, 11, 12, 6]]
    lens = np.array([60, 55], np.int32)
    a = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), _table_from_blocks(shared, 4), lens,
                          0.125, BF16)
    b = oracle_mod.decode(_bits(q), _bits(kc2), _bits(vc2), _table_from_blocks(copied, 4), lens,
                          0.125, BF16)
    assert np.array_equal(a, b)


def _read_golden_table(name):
    rows, meta = [], {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0].isdigit():
                rows.append([int(x) for x in parts])
            else:
                meta[parts[0]] = int(parts[1])
    return rows, meta


def test_pages_block_table_example_and_diagram(oracle_mod):
    """The worked table (47, 23, 89; 8 slots in the last) and the diagram
    (7, 3, 21) placing the same logical tokens give the contiguous result, and
    the two placements agree bit for bit."""
    ex_rows, ex_meta = _read_golden_table("block_table_example.txt")
    dg_rows, dg_meta = _read_golden_table("block_table_diagram.txt")
    bs = ex_meta["block_size"]
    n = sum(r[2] for r in ex_rows)
    assert n == ex_meta["context_len"] == 40
    N = 96
    g = torch.Generator().manual_seed(9)
    K = torch.randn(n, 2, 64, generator=g).to(torch.float16)
    V = torch.randn(n, 2, 64, generator=g).to(torch.float16)
    q = torch.randn(1, 4, 64, generator=g).to(torch.float16)
    outs = []
    for rows in (ex_rows, dg_rows):
        blocks = [r[1] for r in rows]
        kc, vc = _place(K, V, blocks, N, bs)
        outs.append(oracle_mod.decode(_bits(q), _bits(kc), _bits(vc),
                                      _table_from_blocks([blocks], 3), np.array([n]), 0.125, F16))
    assert np.array_equal(outs[0], outs[1])
    ref = _contiguous_reference(q[0].double().numpy(), K.double().numpy(), V.double().numpy(),
                                0.125, 2)
    np.testing.assert_allclose(outs[0][0], ref, rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------ KV-size closed forms
def test_kv_sizes_printed_on_the_pages(oracle_mod):
    with open(os.path.join(GOLDEN, "kv_sizes.txt"), encoding="utf-8") as f:
        lines = [l.split("#")[0].split() for l in f if l.split("#")[0].strip()]
    assert len(lines) == 7
    for layers, kvh, hd, seq, batch, eb, expected in ([int(x) for x in l] for l in lines):
        assert oracle_mod.kv_cache_bytes(layers, kvh, hd, seq, batch, eb) == expected


def test_kv_concurrency_printed_on_the_page(oracle_mod):
    with open(os.path.join(GOLDEN, "kv_concurrency.txt"), encoding="utf-8") as f:
        lines = [l.split("#")[0].split() for l in f if l.split("#")[0].strip()]
    assert len(lines) == 3
    per_tok = oracle_mod.kv_bytes_per_token(28, 4, 128, 2)
    for budget, tok_bytes, max_len, expected in ([int(x) for x in l] for l in lines):
        assert tok_bytes == per_tok
        assert budget // (per_tok * max_len) == expected


# ------------------------------------------------------- append and copy-on-write
def test_scatter_at_allocator_slots_then_table_walk_is_contiguous(oracle_mod):
    """K/V written with the oracle's scatter at the allocator's slots, read back
    through the allocator's table, give SDPA on the contiguous rows."""
    bs, N, n, Hkv, d = 16, 40, 37, 2, 64
    order = np.random.default_rng(21).permutation(N)
    m = oracle_mod.BlockManagerModel(N, bs, order)
    m.allocate(0, 0)
    slots = [m.append_slot(0)[0] for _ in range(n)]
    g = torch.Generator().manual_seed(22)
    K = torch.randn(n, Hkv, d, generator=g).to(torch.float16)
    V = torch.randn(n, Hkv, d, generator=g).to(torch.float16)
    q = torch.randn(1, 4, d, generator=g).to(torch.float16)
    kc = torch.full((N, bs, Hkv, d), float("nan"), dtype=torch.float16)
    vc = kc.clone()
    oracle_mod.reshape_and_cache(K, V, np.array(slots), kc, vc)
    tbl, lens = m.export([0])
    out = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), tbl, lens, 0.125, F16)
    ref = _contiguous_reference(q[0].double().numpy(), K.double().numpy(), V.double().numpy(),
                                0.125, 2)
    np.testing.assert_allclose(out[0], ref, rtol=1e-11, atol=1e-13)
    # padding slots are skipped
    kc2 = kc.clone()
    oracle_mod.reshape_and_cache(K[:1] + 1, V[:1] + 1, np.array([-1]), kc2, vc)
    assert torch.equal(kc2.view(torch.int16), kc.view(torch.int16))


def test_cow_copy_read_through_the_copy_equals_the_original(oracle_mod):
    """After a fork and an append into the shared partial block, the copied
    block holds the shared rows, so both sequences still see the same prefix."""
    bs, N, Hkv, d = 16, 12, 2, 64
    m = oracle_mod.BlockManagerModel(N, bs, np.random.default_rng(23).permutation(N))
    m.allocate(0, 20)
    m.fork(0, 1)
    g = torch.Generator().manual_seed(24)
    kc = torch.randn(N, bs, Hkv, d, generator=g).to(torch.bfloat16)
    vc = torch.randn(N, bs, Hkv, d, generator=g).to(torch.bfloat16)
    q = torch.randn(2, 4, d, generator=g).to(torch.bfloat16)
    tbl0, lens0 = m.export([0, 1], 2)
    before = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), tbl0, lens0, 0.125, BF16)
    slot, cow = m.append_slot(1)
    assert cow is not None
    oracle_mod.copy_blocks([kc], [vc], [cow])
    tbl1, _ = m.export([0, 1], 2)
    assert tbl1[1, 1] == cow[1] and tbl1[0, 1] == cow[0]
    after = oracle_mod.decode(_bits(q), _bits(kc), _bits(vc), tbl1, lens0, 0.125, BF16)
    assert np.array_equal(before, after)
