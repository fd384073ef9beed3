"""GPU parity of the INT8 KV cache: pa_reshape_and_cache_int8 against the
oracle's quantiser (codes and scales bit for bit) and pa_decode_int8 against
the oracle's fp64 attention over the dequantised rows (|gpu - ref| <= 2e-3 +
1e-2 |ref| per element).  Full-size caches take seeded random codes and
scales; small and mid-size ones are written through the quantising append on
both sides.  Unused slots of every last block hold NaN scales."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import workloads as wl

from _harness import assert_close, build_tables
from test_fp8_gpu import _special_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_103_gb300 import build
    build.build()
    binding.load()


def _code(dtype):
    return oracle.DTYPE_F16 if dtype == torch.float16 else oracle.DTYPE_BF16


class Int8Run:
    """Device copies of an INT8 cache plus the decode buffers."""

    def __init__(self, q, c, B, H, d):
        self.q = q.cuda()
        self.kc, self.vc = c["k_codes"].cuda(), c["v_codes"].cuda()
        self.ks, self.vs = c["k_scale"].cuda(), c["v_scale"].cuda()
        self.out = torch.empty_like(self.q)
        self.ws = torch.empty(binding.pa_decode_workspace_size(B, H, d), dtype=torch.uint8,
                              device="cuda")
        binding.pa_decode_workspace_init(self.ws)

    def append(self, k_new, v_new, slots):
        binding.pa_reshape_and_cache_int8(k_new.cuda(), v_new.cuda(),
                                          torch.from_numpy(np.asarray(slots, np.int64)).cuda(),
                                          self.kc, self.vc, self.ks, self.vs)

    def decode(self, tbl, lens, scale):
        t = torch.from_numpy(np.ascontiguousarray(tbl, np.int32)).cuda()
        n = torch.from_numpy(np.ascontiguousarray(lens, np.int32)).cuda()
        binding.pa_decode_int8(self.q, self.kc, self.vc, self.ks, self.vs, t, n,
                               int(np.max(lens)) if len(lens) else 0, scale, self.out, self.ws)
        return self.out


def _same_cache(run, c):
    assert torch.equal(run.kc.cpu(), c["k_codes"]) and torch.equal(run.vc.cpu(), c["v_codes"])
    for dev, host in ((run.ks, c["k_scale"]), (run.vs, c["v_scale"])):
        assert torch.equal(dev.cpu().view(torch.int32), host.view(torch.int32))


def _oracle_decode(q, c, tbl, lens, scale):
    return oracle.decode_int8(wl.bits(q), _code(q.dtype), c["k_codes"].numpy(),
                              c["v_codes"].numpy(), c["k_scale"].numpy(), c["v_scale"].numpy(),
                              tbl, lens, scale)


def _nan_tails(m, c):
    bs = m.block_size
    for s, table in m.allocated.items():
        for pos in range(m.lens[s], len(table) * bs):
            b, r = table[pos // bs], pos % bs
            c["k_codes"][b, r] = 0x7F
            c["v_codes"][b, r] = 0x81
            c["k_scale"][b, :, r] = float("nan")
            c["v_scale"][b, :, r] = float("nan")


@pytest.mark.parametrize("T,N,bs,Hkv,dtype", [(4, 64, 16, 2, torch.float16),
                                              (256, 400, 16, 4, torch.bfloat16),
                                              (1000, 3000, 8, 8, torch.bfloat16),
                                              (77, 50, 32, 40, torch.float16)])
def test_reshape_and_cache_int8_bit_exact(T, N, bs, Hkv, dtype):
    d = 128
    rng = np.random.default_rng(T + 29)
    slots = rng.choice(N * bs, size=T, replace=False).astype(np.int64)
    slots[5::7] = -1                                  # padding tokens are skipped
    kn = wl.normal_tensor((T, Hkv, d), dtype, 5)
    vn = wl.normal_tensor((T, Hkv, d), dtype, 6)
    _special_rows(kn)
    _special_rows(vn)
    w = wl.Workload("append", 1, Hkv, Hkv, d, bs, "f16", np.ones(1, np.int32), N,
                    np.arange(N, dtype=np.int32), T)
    c = wl.int8_cache(w)
    run = Int8Run(torch.zeros(1, Hkv, d, dtype=dtype), c, 1, Hkv, d)
    run.append(kn, vn, slots)
    assert binding.pa_check_device_errors() == 0
    oracle.reshape_and_cache_int8(kn, vn, slots, c["k_codes"].numpy(), c["v_codes"].numpy(),
                                  c["k_scale"].numpy(), c["v_scale"].numpy())
    _same_cache(run, c)


def test_reshape_and_cache_int8_flags_out_of_range_slot():
    N, bs, Hkv, d = 8, 16, 2, 128
    kc = torch.zeros(N, bs, Hkv, d, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros(N, Hkv, bs, dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    kn = -torch.ones(2, Hkv, d, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([N * bs, 3], dtype=torch.int64, device="cuda")
    binding.pa_reshape_and_cache_int8(kn, kn, slots, kc, vc, ks, vs)
    assert binding.pa_check_device_errors() & binding.DEVERR["SLOT"]
    assert torch.count_nonzero(kc).item() == Hkv * d          # only slot 3 written
    assert (kc[0, 3] == 0x81).all()                            # -1 / (1 / 127) -> -127
    assert torch.equal(ks[0, :, 3].cpu(), torch.full((Hkv,), np.float32(1.0) / np.float32(127)))


def _quantised_through_append(B, H, Hkv, bs, dtype, lens, seed):
    d = 128
    N = int(math.ceil(1.25 * sum((int(n) + bs - 1) // bs for n in lens))) + 2
    w = wl.Workload("int8_small", B, H, Hkv, d, bs, "f16" if dtype == torch.float16 else "bf16",
                    np.asarray(lens, np.int32), N, wl._perm(N, seed + 1), seed)
    m = oracle.BlockManagerModel(N, bs, w.free_order)
    slots = []
    for i in range(B):
        m.allocate(i, 0)
        slots += [m.append_slot(i)[0] for _ in range(int(lens[i]))]
    slots = np.asarray(slots, np.int64)
    T = len(slots)
    kn = wl.normal_tensor((max(T, 1), Hkv, d), dtype, seed * 8 + 1)[:T]
    vn = wl.normal_tensor((max(T, 1), Hkv, d), dtype, seed * 8 + 2)[:T]
    q = wl.normal_tensor((B, H, d), dtype, seed * 8 + 3)
    c = wl.int8_cache(w)
    _nan_tails(m, c)
    run = Int8Run(q, c, B, H, d)
    if T:
        run.append(kn, vn, slots)
        oracle.reshape_and_cache_int8(kn, vn, slots, c["k_codes"].numpy(), c["v_codes"].numpy(),
                                      c["k_scale"].numpy(), c["v_scale"].numpy())
    tbl, out_lens = m.export(range(B))
    return q, c, run, tbl, out_lens


@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 4), (28, 4), (32, 2), (32, 1)])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_decode_int8_small(H, Hkv, bs, dtype):
    rng = np.random.default_rng(H * 100 + Hkv * 10 + bs + 3)
    lens = rng.integers(1, 300, size=5)
    lens[2] = 32 * 4 + 1                              # a chunk boundary plus one
    q, c, run, tbl, n = _quantised_through_append(5, H, Hkv, bs, dtype, lens, 60 + bs)
    scale = 1.0 / math.sqrt(128)
    out = run.decode(tbl, n, scale)
    assert binding.pa_check_device_errors() == 0
    _same_cache(run, c)
    assert_close(out.cpu(), _oracle_decode(q, c, tbl, n, scale),
                 "int8 G=%d bs=%d" % (H // Hkv, bs))


def test_decode_int8_mid_size_quantised_cache():
    q, c, run, tbl, n = _quantised_through_append(8, 32, 8, 16, torch.bfloat16,
                                                  np.full(8, 4096), 79)
    _same_cache(run, c)
    out = run.decode(tbl, n, 1.0 / math.sqrt(128))
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _oracle_decode(q, c, tbl, n, 1.0 / math.sqrt(128)), "int8 8x4096")


def _append_then_decode_int8(w):
    m, slots = build_tables(w)
    c = wl.int8_cache(w)
    _nan_tails(m, c)
    dt = w.torch_dtype
    q = wl.normal_tensor((w.B, w.H, w.d), dt, w.seed * 16 + 1)
    kn = wl.normal_tensor((w.B, w.Hkv, w.d), dt, w.seed * 16 + 4)
    vn = wl.normal_tensor((w.B, w.Hkv, w.d), dt, w.seed * 16 + 5)
    tbl, lens = m.export(range(w.B))
    run = Int8Run(q, c, w.B, w.H, w.d)
    run.append(kn, vn, slots)
    out = run.decode(tbl, lens, w.scale)
    assert binding.pa_check_device_errors() == 0
    oracle.reshape_and_cache_int8(kn, vn, slots, c["k_codes"].numpy(), c["v_codes"].numpy(),
                                  c["k_scale"].numpy(), c["v_scale"].numpy())
    _same_cache(run, c)
    assert_close(out.cpu(), _oracle_decode(q, c, tbl, lens, w.scale), w.name + " int8")


def test_decode_int8_llama13b_full_size():
    _append_then_decode_int8(wl.llama13b())


def test_decode_int8_qwen_longtail_full_size():
    _append_then_decode_int8(wl.qwen_longtail(16))


def test_decode_int8_zero_lengths_and_bad_block():
    lens = np.array([0, 40, 0, 17])
    q, c, run, tbl, n = _quantised_through_append(4, 8, 2, 16, torch.float16, lens, 7)
    scale = 1.0 / math.sqrt(128)
    out = run.decode(tbl, n, scale)
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _oracle_decode(q, c, tbl, n, scale), "int8 zero lengths")
    assert not out[0].any() and not out[2].any()
    bad = tbl.copy()
    bad[1, 1] = c["k_codes"].shape[0] + 5
    run.decode(bad, n, scale)
    assert binding.pa_check_device_errors() & binding.DEVERR["BLOCK_ID"]
    assert torch.isfinite(run.out).all()
