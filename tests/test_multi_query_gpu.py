"""GPU parity of pa_multi_query (several causal query tokens per sequence over
the paged cache: chunked prefill, speculative verification) against the fp64
oracle, |gpu - ref| <= 2e-3 + 1e-2 |ref| per element.  Unused slots of every
last block hold NaN, so keys past a context must contribute nothing."""
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


def _setup(lens, qlens, H, Hkv, d, bs, dtype, seed):
    N = int(math.ceil(1.25 * sum(math.ceil(n / bs) for n in lens))) + 2
    m = oracle.BlockManagerModel(N, bs, np.random.default_rng(seed).permutation(N))
    for i, n in enumerate(lens):
        m.allocate(i, int(n))
    kc = wl.normal_tensor((N, bs, Hkv, d), dtype, seed * 3 + 1)
    vc = wl.normal_tensor((N, bs, Hkv, d), dtype, seed * 3 + 2)
    nan_tails(m, kc, vc)
    tbl, ln = m.export(range(len(lens)))
    q_start = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = wl.normal_tensor((int(q_start[-1]), H, d), dtype, seed * 3 + 3)
    return kc, vc, tbl, ln, q_start, q


def _workspace(B, H, Hkv, d, mq):
    ws = torch.empty(binding.pa_multi_query_workspace_size(B, H, Hkv, d, mq), dtype=torch.uint8,
                     device="cuda")
    binding.pa_decode_workspace_init(ws)
    return ws


def _gpu(kc, vc, tbl, ln, q_start, q, scale, max_q_len=None, ws=None):
    out = torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda")
    mq = int(max_q_len if max_q_len is not None else np.diff(q_start).max(initial=0))
    H, d = q.shape[1], q.shape[2]
    if ws is None:
        ws = _workspace(len(ln), H, kc.shape[2], d, mq)
    binding.pa_multi_query(q.cuda(), torch.from_numpy(q_start).cuda(), kc.cuda(), vc.cuda(),
                           torch.from_numpy(tbl).cuda(), torch.from_numpy(ln).cuda(), mq, scale,
                           out, ws)
    return out


def _ref(kc, vc, tbl, ln, q_start, q, scale):
    code = oracle.DTYPE_F16 if q.dtype == torch.float16 else oracle.DTYPE_BF16
    return oracle.multi_query(wl.bits(q), q_start, wl.bits(kc), wl.bits(vc), tbl, ln, scale, code,
                              num_threads=THREADS)


@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 2), (28, 4), (32, 4), (32, 2)])
@pytest.mark.parametrize("d,bs,dtype", [(64, 16, torch.float16), (128, 8, torch.bfloat16),
                                        (128, 32, torch.float16)])
def test_mixed_query_lengths(H, Hkv, d, bs, dtype):
    lens = [1, 37, 200, 130, 64, 71, 5]
    qlens = [1, 6, 200, 65, 1, 0, 5]          # decode, speculative, whole prompt, chunk, none
    kc, vc, tbl, ln, qs, q = _setup(lens, qlens, H, Hkv, d, bs, dtype, H + d + bs)
    scale = 1 / math.sqrt(d)
    out = _gpu(kc, vc, tbl, ln, qs, q, scale)
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, scale), "multi-query G=%d" % (H // Hkv))


def test_speculative_verification_full_size():
    """128 sequences of the Qwen long-tail shape verifying 6 tokens each (a
    draft of 5 plus the last accepted token)."""
    w = wl.qwen_longtail(16)
    lens = np.asarray(w.context_lens, np.int64) + 6
    qlens = [6] * w.B
    kc, vc, tbl, ln, qs, q = _setup(lens, qlens, w.H, w.Hkv, w.d, w.block_size, torch.bfloat16, 21)
    out = _gpu(kc, vc, tbl, ln, qs, q, w.scale)
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, w.scale), "speculative 128 x 6")


def test_chunked_prefill_chunk_of_512():
    """Two sequences each prefilling a 512-token chunk on top of 3584 cached
    tokens (GQA 32 / 8, bf16)."""
    lens = [4096, 4096]
    qlens = [512, 512]
    kc, vc, tbl, ln, qs, q = _setup(lens, qlens, 32, 8, 128, 16, torch.bfloat16, 22)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128))
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128)), "chunk 512")


def test_chunked_prefill_chunk_of_2048_whole_tiles():
    """A 2048-token chunk on top of 6144 cached tokens (GQA 32 / 8, bf16).  A
    64-row tile is 16 tokens x the 4 heads of a KV head; whole tiles (every
    head of 16 consecutive tokens) are checked every 64 tokens across the
    chunk, including its first and last tiles: token t attends to 6144 + t + 1
    keys."""
    n, qlen, H, Hkv, d = 8192, 2048, 32, 8, 128
    kc, vc, tbl, ln, qs, q = _setup([n], [qlen], H, Hkv, d, 16, torch.bfloat16, 23)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(d)).cpu()
    assert binding.pa_check_device_errors() == 0
    for t0 in list(range(0, qlen, 64)) + [qlen - 16]:
        ref = oracle.multi_query(wl.bits(q[t0:t0 + 16]), [0, 16], wl.bits(kc), wl.bits(vc), tbl,
                                 [n - qlen + t0 + 16], 1 / math.sqrt(d), oracle.DTYPE_BF16,
                                 num_threads=THREADS)
        assert_close(out[t0:t0 + 16], ref, "chunk 2048 tokens %d.." % t0)


def test_single_query_matches_decode_reference():
    lens = [300, 1, 1000, 64]
    kc, vc, tbl, ln, qs, q = _setup(lens, [1, 1, 1, 1], 8, 2, 128, 16, torch.float16, 24)
    out = _gpu(kc, vc, tbl, ln, qs, q, 0.1)
    ref = oracle.decode(wl.bits(q), wl.bits(kc), wl.bits(vc), tbl, ln, 0.1, oracle.DTYPE_F16,
                        num_threads=THREADS)
    assert_close(out.cpu(), ref, "single query")


def test_repeat_reuses_workspace_and_is_deterministic():
    """Long contexts with few tiles make the items split between CTAs; a
    reused workspace must come back with every ticket at zero."""
    kc, vc, tbl, ln, qs, q = _setup([20000, 333, 9000], [6, 17, 6], 28, 4, 128, 16,
                                    torch.bfloat16, 25)
    ws = _workspace(3, 28, 4, 128, 17)
    a = _gpu(kc, vc, tbl, ln, qs, q, 0.09, ws=ws)
    for _ in range(3):
        b = _gpu(kc, vc, tbl, ln, qs, q, 0.09, ws=ws)
        assert torch.equal(a, b)
    assert binding.pa_check_device_errors() == 0
    assert_close(a.cpu(), _ref(kc, vc, tbl, ln, qs, q, 0.09), "split items")


@pytest.mark.parametrize("H,Hkv,d,dtype", [(8, 1, 64, torch.float16), (32, 2, 128, torch.float16),
                                           (16, 16, 64, torch.bfloat16)])
def test_split_items_every_instantiation(H, Hkv, d, dtype):
    """Few tiles over long contexts: each tile is shared by several CTAs and
    merged from partials, for head dims 64 / 128, f16 / bf16, G = 1 .. 16."""
    lens = [30000, 12000, 7]
    qlens = [3, 9, 7]
    kc, vc, tbl, ln, qs, q = _setup(lens, qlens, H, Hkv, d, 32, dtype, 27 + H)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(d))
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(d)), "split items")


def test_more_queries_than_context_is_flagged_and_skipped():
    kc, vc, tbl, ln, qs, q = _setup([10, 20], [3, 5], 4, 2, 64, 16, torch.float16, 26)
    ln_bad = ln.copy()
    ln_bad[0] = 2                                # 3 queries, 2 cached tokens
    out = _gpu(kc, vc, tbl, ln_bad, qs, q, 0.125)
    assert binding.pa_check_device_errors() & binding.DEVERR["CONTEXT"]
    assert torch.isnan(out[:3].float()).all()     # sequence 0 untouched
    ref = _ref(kc, vc, tbl, ln, qs, q, 0.125)
    assert_close(out[3:].cpu(), ref[3:], "the valid sequence")


def test_max_batch():
    """4096 sequences (the largest batch one call takes), each verifying 0 to
    3 tokens over a short context."""
    B = 4096
    rng = np.random.default_rng(31)
    lens = rng.integers(1, 60, size=B)
    qlens = np.minimum(lens, rng.integers(0, 4, size=B))
    kc, vc, tbl, ln, qs, q = _setup(lens, qlens, 8, 2, 128, 16, torch.bfloat16, 31)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128))
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128)), "B=4096")


def test_batch_above_the_limit_is_refused():
    lens = [2] * 4097
    kc, vc, tbl, ln, qs, q = _setup(lens, [1] * 4097, 4, 2, 64, 16, torch.float16, 32)
    with pytest.raises(binding.PaError) as e:
        _gpu(kc, vc, tbl, ln, qs, q, 0.125)
    assert binding.STATUS_NAMES[e.value.status] == "PA_ERR_UNSUPPORTED"
    assert binding.pa_check_device_errors() == 0


@pytest.mark.parametrize("H,Hkv,d,dtype,qlens", [(8, 1, 64, torch.float16, [6, 1, 5]),
                                                 (16, 2, 128, torch.bfloat16, [6, 3, 6]),
                                                 (28, 4, 128, torch.float16, [6, 6, 2]),
                                                 (4, 4, 64, torch.bfloat16, [12, 1, 7])])
def test_three_warp_shape_every_instantiation(H, Hkv, d, dtype, qlens):
    """Items of at most 48 rows (max_q_len x G <= 48) run three consumer warps
    and three CTAs per SM; long contexts split them between CTAs."""
    assert max(qlens) * (H // Hkv) <= 48
    lens = [25000, 9000, 7]
    kc, vc, tbl, ln, qs, q = _setup(lens, qlens, H, Hkv, d, 16, dtype, 40 + H + d)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(d))
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(d)), "three warps")
