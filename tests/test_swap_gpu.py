"""GPU parity of swapping (pa_swap_blocks between the device pools and a
pinned host pool): the host pool holds bit copies of the swapped blocks, the
blocks swapped back in are bit copies of the originals even after their old
device blocks were reused and overwritten, and the decode after swap-in is
bit-identical to the decode before swap-out and within tolerance of the
oracle.  Three layers' K and V (six pools) move in one launch per direction."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import workloads as wl

from _harness import THREADS, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_103_gb300 import build
    build.build()
    binding.load()


def _pairs(p, where):
    t = torch.from_numpy(np.ascontiguousarray(p, np.int32))
    return t.cuda() if where == "device" else t.pin_memory()


@pytest.mark.parametrize("pairs_in", ["device", "pinned"])
def test_swap_round_trip_bit_exact_and_decode(pairs_in):
    L, bs, Hkv, d, H, N, HB = 3, 16, 4, 128, 28, 800, 300
    dt = torch.bfloat16
    a = binding.Allocator(N, bs, np.random.default_rng(1).permutation(N).astype(np.int32))
    a.set_swap_pool(HB)
    lens = np.random.default_rng(2).integers(100, 1500, 8)
    for i, n in enumerate(lens):
        a.alloc(i, int(n))
    pools = [wl.normal_tensor((N, bs, Hkv, d), dt, 10 + j).cuda() for j in range(2 * L)]
    host = [torch.zeros(HB, bs, Hkv, d, dtype=dt).pin_memory() for _ in range(2 * L)]
    orig = [p.clone() for p in pools]
    B = len(lens)
    tbl, ln = a.export(list(range(B)), 128)
    q = wl.normal_tensor((B, H, d), dt, 5).cuda()
    ws = torch.empty(binding.pa_decode_workspace_size(B, H, d), dtype=torch.uint8, device="cuda")
    binding.pa_decode_workspace_init(ws)

    def decode(tb, l, layer):
        out = torch.empty_like(q)
        binding.pa_decode(q, pools[2 * layer], pools[2 * layer + 1],
                          torch.from_numpy(tb).cuda(), torch.from_numpy(l).cuda(),
                          int(l.max()), 1 / math.sqrt(d), out, ws)
        return out

    before = [decode(tbl, ln, layer).cpu() for layer in range(L)]
    out_pairs = {}
    for s in (1, 4, 6):
        p = a.swap_out(s)
        out_pairs[s] = p
        binding.pa_swap_blocks(pools, host, _pairs(p, pairs_in))
    torch.cuda.synchronize()
    for s, p in out_pairs.items():
        for j in range(2 * L):
            assert torch.equal(host[j][torch.from_numpy(p[:, 1]).long()].view(torch.int16),
                               orig[j][torch.from_numpy(p[:, 0]).long().cuda()].cpu().view(torch.int16))
    # reuse the freed device blocks and overwrite them
    a.alloc(100, int(a.stats()["free_blocks"]) * bs)
    tb100, _ = a.export([100], N)
    used = torch.from_numpy(tb100[0][tb100[0] >= 0]).long().cuda()
    for pl in pools:
        pl[used] = float("nan")
    a.free(100)
    in_pairs = {}
    for s in (6, 1, 4):
        p = a.swap_in(s)
        in_pairs[s] = p
        binding.pa_swap_blocks(host, pools, _pairs(p, pairs_in))
    assert binding.pa_check_device_errors() == 0
    # swapped-in blocks are bit copies of the originals
    for s in (1, 4, 6):
        src_dev = torch.from_numpy(out_pairs[s][:, 0]).long().cuda()
        hosts = {h: dblk for h, dblk in in_pairs[s]}
        new_dev = torch.from_numpy(np.array([hosts[h] for h in out_pairs[s][:, 1]])).long().cuda()
        for j in range(2 * L):
            assert torch.equal(pools[j][new_dev].view(torch.int16), orig[j][src_dev].view(torch.int16))
    tbl2, ln2 = a.export(list(range(B)), 128)
    for layer in range(L):
        after = decode(tbl2, ln2, layer).cpu()
        assert torch.equal(after.view(torch.int16), before[layer].view(torch.int16))
        ref = oracle.decode(wl.bits(q.cpu()), wl.bits(orig[2 * layer].cpu()),
                            wl.bits(orig[2 * layer + 1].cpu()), tbl, ln, 1 / math.sqrt(d),
                            oracle.DTYPE_BF16, num_threads=THREADS)
        assert_close(after, ref, "decode after swap-in, layer %d" % layer)


def test_swap_blocks_flags_bad_pairs():
    src = torch.ones(4, 16, 2, 64, dtype=torch.float16, device="cuda")
    dst = torch.zeros(4, 16, 2, 64, dtype=torch.float16).pin_memory()
    pairs = torch.tensor([[1, 2], [4, 0], [0, 9]], dtype=torch.int32, device="cuda")
    binding.pa_swap_blocks([src], [dst], pairs)
    assert binding.pa_check_device_errors() & binding.DEVERR["PAIR"]
    assert torch.count_nonzero(dst).item() == dst[2].numel()      # only block 2 written


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_swap_round_trip_of_an_8bit_cache(fmt):
    """An 8-bit cache swaps as two pool pairs moved with the same block pairs:
    the codes [N, bs, Hkv, 128] and the scales [N, Hkv, bs].  After swap-out,
    reuse and overwrite of the freed device blocks (NaN codes and scales) and
    swap-in, the blocks are bit copies and the 8-bit decode is bit-identical
    to the one before, and within tolerance of the oracle."""
    bs, Hkv, d, H, N, HB = 16, 4, 128, 28, 700, 300
    a = binding.Allocator(N, bs, np.random.default_rng(3).permutation(N).astype(np.int32))
    a.set_swap_pool(HB)
    lens = np.random.default_rng(4).integers(100, 1500, 6).astype(np.int32)
    for i, n in enumerate(lens):
        a.alloc(i, int(n))
    w = wl.Workload("swap8", len(lens), H, Hkv, d, bs, "bf16", lens, N,
                    np.arange(N, dtype=np.int32), 41)
    c = wl.fp8_cache(w) if fmt == "fp8" else wl.int8_cache(w)
    codes = [c["k_codes"].cuda(), c["v_codes"].cuda()]
    scales = [c["k_scale"].cuda(), c["v_scale"].cuda()]
    hcodes = [torch.zeros(HB, bs, Hkv, d, dtype=torch.uint8).pin_memory() for _ in range(2)]
    hscales = [torch.zeros(HB, Hkv, bs, dtype=torch.float32).pin_memory() for _ in range(2)]
    B = len(lens)
    tbl, ln = a.export(list(range(B)), 128)
    q = wl.normal_tensor((B, H, d), torch.bfloat16, 6).cuda()
    ws = torch.empty(binding.pa_decode_workspace_size(B, H, d), dtype=torch.uint8, device="cuda")
    binding.pa_decode_workspace_init(ws)
    decode8 = getattr(binding, "pa_decode_" + fmt)

    def decode(tb, l):
        out = torch.empty_like(q)
        decode8(q, codes[0], codes[1], scales[0], scales[1], torch.from_numpy(tb).cuda(),
                torch.from_numpy(l).cuda(), int(l.max()), 1 / math.sqrt(d), out, ws)
        return out.cpu()

    before = decode(tbl, ln)
    out_pairs = {}
    for s in (0, 3, 5):
        p = a.swap_out(s)
        out_pairs[s] = p
        pt = _pairs(p, "device")
        binding.pa_swap_blocks(codes, hcodes, pt)
        binding.pa_swap_blocks(scales, hscales, pt)
    torch.cuda.synchronize()
    a.alloc(100, int(a.stats()["free_blocks"]) * bs)
    tb100, _ = a.export([100], N)
    used = torch.from_numpy(tb100[0][tb100[0] >= 0]).long().cuda()
    for pl in codes:
        pl[used] = 0x7F
    for pl in scales:
        pl[used] = float("nan")
    a.free(100)
    in_pairs = {}
    for s in (5, 0, 3):
        p = a.swap_in(s)
        in_pairs[s] = p
        pt = _pairs(p, "pinned")
        binding.pa_swap_blocks(hcodes, codes, pt)
        binding.pa_swap_blocks(hscales, scales, pt)
    assert binding.pa_check_device_errors() == 0
    for s in (0, 3, 5):
        src = torch.from_numpy(out_pairs[s][:, 0]).long()
        hosts = {h: dblk for h, dblk in in_pairs[s]}
        new = torch.from_numpy(np.array([hosts[h] for h in out_pairs[s][:, 1]])).long().cuda()
        for j, name in enumerate(("k", "v")):
            assert torch.equal(codes[j][new].cpu(), c[name + "_codes"][src])
            assert torch.equal(scales[j][new].cpu().view(torch.int32),
                               c[name + "_scale"][src].view(torch.int32))
    tbl2, ln2 = a.export(list(range(B)), 128)
    after = decode(tbl2, ln2)
    assert torch.equal(after.view(torch.int16), before.view(torch.int16))
    ref = getattr(oracle, "decode_" + fmt)(wl.bits(q.cpu()), oracle.DTYPE_BF16,
                                           c["k_codes"].numpy(), c["v_codes"].numpy(),
                                           c["k_scale"].numpy(), c["v_scale"].numpy(), tbl, ln,
                                           1 / math.sqrt(d))
    assert_close(after, ref, "%s decode after swap-in" % fmt)
