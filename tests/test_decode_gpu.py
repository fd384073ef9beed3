"""GPU parity: pa_reshape_and_cache + pa_decode through the C ABI against the
fp64 oracle on the same seeded inputs, on every workload shape at full size.

Attention outputs must satisfy |gpu - ref| <= 2e-3 + 1e-2 |ref| per element;
cache contents must match bit for bit.  Unused slots of every last block hold
NaN, so a kernel that lets rows past a context leak in fails.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import workloads as wl

from _harness import (GpuRun, assert_close, bit_equal, build_tables, nan_tails,
                      oracle_decode)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_103_gb300 import build
    build.build()
    binding.load()


def _append_then_decode(w, nan=True):
    host = wl.qkv(w)
    m, slots = build_tables(w)
    if nan:
        nan_tails(m, host["k_cache"], host["v_cache"])
    tbl, lens = m.export(range(w.B))
    run = GpuRun(w, host)
    run.append(host["k_new"], host["v_new"], slots)
    out = run.decode(tbl, lens)
    flags = binding.pa_check_device_errors()
    assert flags == 0
    # oracle: same append on host copies, then fp64 attention
    kc, vc = host["k_cache"].clone(), host["v_cache"].clone()
    oracle.reshape_and_cache(host["k_new"], host["v_new"], slots, kc, vc)
    assert bit_equal(run.k_cache, kc) and bit_equal(run.v_cache, vc)
    ref = oracle_decode(w, host["q"], kc, vc, tbl, lens)
    return assert_close(out.cpu(), ref, w.name), run, (tbl, lens, ref)


@pytest.mark.parametrize("seed", [1001, 7, 8, 9, 10])
def test_tiny(seed):
    _append_then_decode(wl.tiny(seed))


def test_llama13b_mha_full_size():
    _append_then_decode(wl.llama13b())


@pytest.mark.parametrize("B,n", [(1, 1024), (8, 4096), (8, 8192), (16, 32768)])
def test_gqa7b_full_size(B, n):
    _append_then_decode(wl.gqa7b(B, n))


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_qwen_longtail_full_size(bs):
    _append_then_decode(wl.qwen_longtail(bs))


@pytest.mark.parametrize("with_suffix,copies", [(True, 0), (False, 255)])
def test_prefix_share_decode_then_append_with_cow(with_suffix, copies):
    """Decode over shared prefix blocks, then one append each: copy-on-write
    of the shared partial block (255 copies for the 1000-token prefix, none
    for the block-aligned 1024), the writes, and a second decode."""
    w = wl.prefix_share(with_suffix=with_suffix, prefix_len=1024 if with_suffix else 1000)
    host = wl.qkv(w)
    m, _ = build_tables(w)
    nan_tails(m, host["k_cache"], host["v_cache"])
    tbl, lens = m.export(range(w.B))
    run = GpuRun(w, host)
    out = run.decode(tbl, lens)
    kc, vc = host["k_cache"].clone(), host["v_cache"].clone()
    assert_close(out.cpu(), oracle_decode(w, host["q"], kc, vc, tbl, lens), w.name)

    slots, pairs = m.append_batch(range(w.B))
    assert len(pairs) == copies
    if pairs:
        pd = torch.tensor(pairs, dtype=torch.int32).cuda()
        binding.pa_copy_blocks([run.k_cache], [run.v_cache], pd)
        oracle.copy_blocks([kc], [vc], pairs)
    run.append(host["k_new"], host["v_new"], slots)
    oracle.reshape_and_cache(host["k_new"], host["v_new"], slots, kc, vc)
    assert binding.pa_check_device_errors() == 0
    assert bit_equal(run.k_cache, kc) and bit_equal(run.v_cache, vc)
    tbl2, lens2 = m.export(range(w.B))
    out2 = run.decode(tbl2, lens2)
    assert_close(out2.cpu(), oracle_decode(w, host["q"], kc, vc, tbl2, lens2), w.name + "+1")
    assert binding.pa_check_device_errors() == 0


def test_repeated_calls_reuse_workspace_and_are_deterministic():
    """Split pairs leave their tickets at zero, so calls can repeat on one
    workspace; results are bit-identical."""
    _, run, (tbl, lens, ref) = _append_then_decode(wl.gqa7b(1, 1024))
    first = run.out.clone()
    for _ in range(3):
        out = run.decode(tbl, lens)
        assert torch.equal(out, first)
    # a different shape on the same workspace size class
    w2 = wl.gqa7b(2, 3000, seed=5)
    _append_then_decode(w2)


def _custom(B, H, Hkv, d, bs, lens, dtype=torch.bfloat16, seed=0, extra_blocks=3):
    lens = np.asarray(lens, np.int32)
    N = int(sum((int(n) + bs - 1) // bs for n in lens)) + extra_blocks
    w = wl.Workload("custom", B, H, Hkv, d, bs, "bf16" if dtype == torch.bfloat16 else "f16",
                    lens, N, np.random.default_rng(seed).permutation(N).astype(np.int32), seed)
    host = wl.qkv(w, with_new=False)
    m = oracle.BlockManagerModel(N, bs, w.free_order)
    for i, n in enumerate(lens):
        m.allocate(i, int(n))
    nan_tails(m, host["k_cache"], host["v_cache"])
    tbl, lens_ = m.export(range(B), max(1, max(len(m.allocated[i]) for i in range(B))))
    return w, host, tbl, lens_


@pytest.mark.parametrize("case", [
    dict(B=5, H=8, Hkv=8, d=64, bs=16, lens=[1, 0, 33, 0, 64], dtype=torch.float16),
    dict(B=3, H=32, Hkv=2, d=128, bs=8, lens=[100, 1, 257]),            # G = 16
    dict(B=4, H=28, Hkv=4, d=128, bs=32, lens=[32, 64, 31, 65]),         # chunk edges
    dict(B=2, H=14, Hkv=2, d=64, bs=16, lens=[5000, 17], dtype=torch.bfloat16),
    dict(B=1, H=4, Hkv=1, d=128, bs=16, lens=[100000]),                  # one pair on every CTA
    dict(B=300, H=8, Hkv=2, d=128, bs=16, lens=list(range(1, 301))),
    # many short bf16 rows: a few keys whose V terms cancel need more than the
    # 8 bits of a bf16 P
    dict(B=512, H=28, Hkv=4, d=128, bs=8, lens=[1 + (7 * i) % 12 for i in range(512)]),
])
def test_edge_shapes(case):
    dtype = case.pop("dtype", torch.bfloat16)
    w, host, tbl, lens = _custom(dtype=dtype, **case)
    run = GpuRun(w, host)
    out = run.decode(tbl, lens)
    assert binding.pa_check_device_errors() == 0
    ref = oracle_decode(w, host["q"], host["k_cache"], host["v_cache"], tbl, lens)
    assert_close(out.cpu(), ref, "edge")
    zero_rows = np.where(lens == 0)[0]
    assert torch.count_nonzero(out[zero_rows]).item() == 0 if len(zero_rows) else True


def test_all_empty_batch_gives_zeros():
    w, host, tbl, lens = _custom(3, 4, 2, 64, 16, [0, 0, 0], extra_blocks=4)
    run = GpuRun(w, host)
    run.out.fill_(1.0)
    out = run.decode(np.zeros((3, 1), np.int32), lens)
    assert binding.pa_check_device_errors() == 0
    assert torch.count_nonzero(out).item() == 0


def test_pages_block_table_placements_on_gpu():
    """The worked table (47, 23, 89 with 8 slots used) and the diagram
    placement (7, 3, 21) of the same 40 tokens give bit-identical outputs."""
    bs, N, n = 16, 96, 40
    g = torch.Generator().manual_seed(3)
    K = torch.randn(n, 2, 64, generator=g).to(torch.float16)
    V = torch.randn(n, 2, 64, generator=g).to(torch.float16)
    q = torch.randn(1, 4, 64, generator=g).to(torch.float16)
    outs = []
    for blocks in ([47, 23, 89], [7, 3, 21]):
        kc = torch.full((N, bs, 2, 64), float("nan"), dtype=torch.float16)
        vc = kc.clone()
        for j in range(n):
            kc[blocks[j // bs], j % bs] = K[j]
            vc[blocks[j // bs], j % bs] = V[j]
        w = wl.Workload("pages", 1, 4, 2, 64, bs, "f16", np.array([n], np.int32), N,
                        np.arange(N, dtype=np.int32), 0)
        run = GpuRun(w, {"q": q, "k_cache": kc, "v_cache": vc})
        tbl = np.array([blocks], np.int32)
        outs.append(run.decode(tbl, np.array([n], np.int32)).cpu())
        ref = oracle_decode(w, q, kc, vc, tbl, np.array([n], np.int32))
        assert_close(outs[-1], ref, "pages")
    assert torch.equal(outs[0], outs[1])


def test_bad_table_entries_are_flagged_not_followed():
    w, host, tbl, lens = _custom(2, 8, 2, 128, 16, [40, 20])
    run = GpuRun(w, host)
    bad = tbl.copy()
    bad[0, 1] = w.num_blocks + 1000           # outside the pool
    bad[1, 0] = -7
    run.decode(bad, lens)
    flags = binding.pa_check_device_errors()
    assert flags & binding.DEVERR["BLOCK_ID"]
    # a context longer than its table row
    run.decode(tbl[:, :1], np.array([40, 20], np.int32))
    assert binding.pa_check_device_errors() & binding.DEVERR["TABLE_WIDTH"]
    # afterwards a good call is clean and correct
    out = run.decode(tbl, lens)
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), oracle_decode(w, host["q"], host["k_cache"], host["v_cache"], tbl,
                                          lens), "after-bad")


def test_single_long_pair_split_over_every_cta_d64():
    """One sequence, one KV head, head_dim 64: the pair is cut into as many
    partials as there are CTAs, more than the merge can stage at once."""
    w, host, tbl, lens = _custom(1, 2, 1, 64, 16, [200000], dtype=torch.bfloat16)
    run = GpuRun(w, host)
    out = run.decode(tbl, lens)
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), oracle_decode(w, host["q"], host["k_cache"], host["v_cache"], tbl,
                                          lens), "long-d64")


@pytest.mark.parametrize("H,Hkv,d,dtype", [(32, 2, 128, torch.bfloat16), (8, 8, 64, torch.float16)])
def test_max_batch(H, Hkv, d, dtype):
    """The largest batch one call takes: 4096 short sequences, empty ones
    among them, G = 16 and G = 1."""
    B = 4096
    lens = np.random.default_rng(H + d).integers(0, 48, size=B)
    w, host, tbl, lens = _custom(B, H, Hkv, d, 16, lens, dtype=dtype, seed=H + d)
    run = GpuRun(w, host)
    out = run.decode(tbl, lens)
    assert binding.pa_check_device_errors() == 0
    ref = oracle_decode(w, host["q"], host["k_cache"], host["v_cache"], tbl, lens)
    assert_close(out.cpu(), ref, "B=4096 G=%d" % (H // Hkv))
    assert torch.count_nonzero(out[np.where(lens == 0)[0]]).item() == 0


def test_batch_above_the_limit_is_refused():
    w, host, tbl, lens = _custom(4097, 4, 4, 64, 16, np.ones(4097, np.int32), seed=3)
    run = GpuRun(w, host)
    run.out.fill_(7.0)
    with pytest.raises(binding.PaError) as e:
        run.decode(tbl, lens)
    assert binding.STATUS_NAMES[e.value.status] == "PA_ERR_UNSUPPORTED"
    torch.cuda.synchronize()
    assert bool((run.out == 7.0).all())                    # nothing was launched
    assert binding.pa_check_device_errors() == 0


@pytest.mark.parametrize("H,Hkv,d,bs,dtype", [(32, 1, 128, 16, torch.bfloat16),
                                              (96, 2, 64, 8, torch.float16),
                                              (64, 1, 128, 32, torch.float16)])
def test_groups_wider_than_16(H, Hkv, d, bs, dtype):
    """Multi-query attention and other groups of 32 .. 64 query heads per KV
    head: each KV head's heads are processed 16 at a time."""
    lens = [1, 0, 31, 33, 700, 5000, 64, 257]
    w, host, tbl, lens = _custom(len(lens), H, Hkv, d, bs, lens, dtype=dtype, seed=H + d)
    run = GpuRun(w, host)
    out = run.decode(tbl, lens)
    assert binding.pa_check_device_errors() == 0
    ref = oracle_decode(w, host["q"], host["k_cache"], host["v_cache"], tbl, lens)
    assert_close(out.cpu(), ref, "G=%d" % (H // Hkv))


def test_group_above_16_not_a_multiple_is_refused():
    w, host, tbl, lens = _custom(2, 24, 1, 64, 16, [10, 20], seed=4)
    run = GpuRun(w, host)
    with pytest.raises(binding.PaError) as e:
        run.decode(tbl, lens)
    assert binding.STATUS_NAMES[e.value.status] == "PA_ERR_UNSUPPORTED"
