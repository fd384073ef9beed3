"""Seeded random shapes through the C ABI against the fp64 oracle: head dim,
block size, GQA group, batch, dtype and the length mix (empty, one token,
chunk and block edges, long) drawn per case, so combinations the hand-picked
tests do not name are covered.  Tolerance |gpu - ref| <= 2e-3 + 1e-2 |ref|;
unused slots of every last block hold NaN (16-bit) or NaN codes and scales
(FP8)."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import workloads as wl

from _harness import THREADS, assert_close, nan_tails

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_103_gb300 import build
    build.build()
    binding.load()


def _shape(rng, d=None, max_b=32, max_len=9000):
    """(d, block size, Hkv, G, B, lengths, dtype); lengths mix empty and 1-2
    token contexts, 32-token chunk edges (+-1), short and long ones."""
    d = int(d or rng.choice([64, 128]))
    bs = int(rng.choice([8, 16, 32]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 12, 16, 32]))
    B = int(rng.integers(1, max_b + 1))
    kind = rng.integers(0, 4, size=B)
    lens = np.where(kind == 0, rng.integers(0, 3, size=B),
           np.where(kind == 1, 32 * rng.integers(1, 9, size=B) + rng.integers(-1, 2, size=B),
           np.where(kind == 2, rng.integers(3, 700, size=B),
                    rng.integers(2000, max_len, size=B)))).astype(np.int64)
    lens = np.maximum(lens, 0)
    dtype = torch.float16 if rng.random() < 0.5 else torch.bfloat16
    return d, bs, Hkv, G, B, lens, dtype


def _pool(lens, bs, seed):
    N = int(math.ceil(1.25 * sum(math.ceil(int(n) / bs) for n in lens))) + 3
    m = oracle.BlockManagerModel(N, bs, np.random.default_rng(seed).permutation(N))
    for i, n in enumerate(lens):
        m.allocate(i, int(n))
    return N, m


def _code(dtype):
    return oracle.DTYPE_F16 if dtype == torch.float16 else oracle.DTYPE_BF16


@pytest.mark.parametrize("seed", range(48))
def test_decode(seed):
    rng = np.random.default_rng(7000 + seed)
    d, bs, Hkv, G, B, lens, dtype = _shape(rng)
    H = Hkv * G
    N, m = _pool(lens, bs, seed)
    kc = wl.normal_tensor((N, bs, Hkv, d), dtype, seed * 4 + 1)
    vc = wl.normal_tensor((N, bs, Hkv, d), dtype, seed * 4 + 2)
    nan_tails(m, kc, vc)
    q = wl.normal_tensor((B, H, d), dtype, seed * 4 + 3)
    tbl, ln = m.export(range(B), max(1, max(len(m.allocated[i]) for i in range(B))))
    scale = float(rng.uniform(0.5, 1.5)) / math.sqrt(d)
    out = torch.full_like(q, float("nan")).cuda()
    ws = torch.empty(binding.pa_decode_workspace_size(B, H, d), dtype=torch.uint8, device="cuda")
    binding.pa_decode_workspace_init(ws)
    binding.pa_decode(q.cuda(), kc.cuda(), vc.cuda(), torch.from_numpy(tbl).cuda(),
                      torch.from_numpy(ln).cuda(), int(ln.max()), scale, out, ws)
    assert binding.pa_check_device_errors() == 0
    ref = oracle.decode(wl.bits(q), wl.bits(kc), wl.bits(vc), tbl, ln, scale, _code(dtype),
                        num_threads=THREADS)
    what = "d=%d bs=%d Hkv=%d G=%d B=%d %s" % (d, bs, Hkv, G, B, dtype)
    assert_close(out.cpu(), ref, what)


@pytest.mark.parametrize("seed", range(24))
def test_decode_fp8(seed):
    rng = np.random.default_rng(8000 + seed)
    d, bs, Hkv, G, B, lens, dtype = _shape(rng, d=128, max_b=12, max_len=4000)
    H = Hkv * G
    N, m = _pool(lens, bs, seed)
    w = wl.Workload("random", B, H, Hkv, d, bs, "f16" if dtype == torch.float16 else "bf16",
                    lens.astype(np.int32), N, np.arange(N, dtype=np.int32), 9000 + seed)
    c = wl.fp8_cache(w)
    for s, table in m.allocated.items():           # unused slots: NaN codes and scales
        for pos in range(m.lens[s], len(table) * bs):
            b, r = table[pos // bs], pos % bs
            c["k_codes"][b, r] = 0x7F
            c["v_codes"][b, r] = 0x7F
            c["k_scale"][b, :, r] = float("nan")
            c["v_scale"][b, :, r] = float("nan")
    q = wl.normal_tensor((B, H, d), dtype, seed * 4 + 3)
    tbl, ln = m.export(range(B), max(1, max(len(m.allocated[i]) for i in range(B))))
    scale = 1 / math.sqrt(d)
    dev = {k: v.cuda() for k, v in c.items()}
    out = torch.full_like(q, float("nan")).cuda()
    ws = torch.empty(binding.pa_decode_workspace_size(B, H, d), dtype=torch.uint8, device="cuda")
    binding.pa_decode_workspace_init(ws)
    binding.pa_decode_fp8(q.cuda(), dev["k_codes"], dev["v_codes"], dev["k_scale"],
                          dev["v_scale"], torch.from_numpy(tbl).cuda(),
                          torch.from_numpy(ln).cuda(), int(ln.max()), scale, out, ws)
    assert binding.pa_check_device_errors() == 0
    ref = oracle.decode_fp8(wl.bits(q), _code(dtype), c["k_codes"].numpy(), c["v_codes"].numpy(),
                            c["k_scale"].numpy(), c["v_scale"].numpy(), tbl, ln, scale)
    what = "fp8 bs=%d Hkv=%d G=%d B=%d %s" % (bs, Hkv, G, B, dtype)
    assert_close(out.cpu(), ref, what)


@pytest.mark.parametrize("seed", range(36))
def test_multi_query(seed):
    rng = np.random.default_rng(9500 + seed)
    d, bs, Hkv, G, B, lens, dtype = _shape(rng, max_b=12, max_len=4000)
    H = Hkv * G
    lens = np.maximum(lens, 1)
    cap = int(rng.choice([1, 3, 6, 17, 64]))
    qlens = np.minimum(lens, rng.integers(0, cap + 1, size=B))
    N, m = _pool(lens, bs, seed)
    kc = wl.normal_tensor((N, bs, Hkv, d), dtype, seed * 4 + 1)
    vc = wl.normal_tensor((N, bs, Hkv, d), dtype, seed * 4 + 2)
    nan_tails(m, kc, vc)
    q_start = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = wl.normal_tensor((max(int(q_start[-1]), 1), H, d), dtype, seed * 4 + 3)[: int(q_start[-1])]
    tbl, ln = m.export(range(B), max(1, max(len(m.allocated[i]) for i in range(B))))
    scale = 1 / math.sqrt(d)
    mq = int(qlens.max())
    out = torch.full(q.shape, float("nan"), dtype=dtype, device="cuda")
    ws = torch.empty(binding.pa_multi_query_workspace_size(B, H, Hkv, d, mq), dtype=torch.uint8,
                     device="cuda")
    binding.pa_decode_workspace_init(ws)
    binding.pa_multi_query(q.cuda(), torch.from_numpy(q_start).cuda(), kc.cuda(), vc.cuda(),
                           torch.from_numpy(tbl).cuda(), torch.from_numpy(ln).cuda(), mq, scale,
                           out, ws)
    assert binding.pa_check_device_errors() == 0
    ref = oracle.multi_query(wl.bits(q), q_start, wl.bits(kc), wl.bits(vc), tbl, ln, scale,
                             _code(dtype), num_threads=THREADS)
    what = "mq d=%d bs=%d Hkv=%d G=%d B=%d max_q %d %s" % (d, bs, Hkv, G, B, mq, dtype)
    assert_close(out.cpu(), ref, what)
