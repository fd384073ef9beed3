"""GPU parity of pa_multi_query_tc (several causal query tokens per sequence
over the paged cache on the tcgen05 tensor cores) against the fp64 oracle,
|gpu - ref| <= 2e-3 + 1e-2 |ref| per element, in both of its modes: pairs of
128-row query tiles sharing each key tile (prefill chunks) and one query tile
per (sequence, KV head) with the key tiles split evenly over the CTAs
(max_q_len * G <= 128: speculative verification, decode-like batches).
Unused slots of every last block hold NaN, so keys past a context must
contribute nothing.  The first case is the smallest one the kernel runs: one
128-row tile over one key tile."""
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


def _workspace(B, H, Hkv):
    ws = torch.empty(binding.pa_multi_query_tc_workspace_size(B, H, Hkv, 128), dtype=torch.uint8,
                     device="cuda")
    binding.pa_decode_workspace_init(ws)
    return ws


def _gpu(kc, vc, tbl, ln, q_start, q, scale, ws=None, max_q_len=None):
    out = torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda")
    mq = int(max_q_len if max_q_len is not None else np.diff(q_start).max(initial=0))
    if ws is None:
        ws = _workspace(len(ln), q.shape[1], kc.shape[2])
    binding.pa_multi_query_tc(q.cuda(), torch.from_numpy(q_start).cuda(), kc.cuda(), vc.cuda(),
                              torch.from_numpy(tbl).cuda(), torch.from_numpy(ln).cuda(), mq, scale,
                              out, ws)
    return out


def _ref(kc, vc, tbl, ln, q_start, q, scale):
    code = oracle.DTYPE_F16 if q.dtype == torch.float16 else oracle.DTYPE_BF16
    return oracle.multi_query(wl.bits(q), q_start, wl.bits(kc), wl.bits(vc), tbl, ln, scale, code,
                              num_threads=THREADS)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_bringup_one_tile(dtype):
    """One sequence, one KV head of 4 query heads, the last 32 of 64 cached
    tokens as queries: a single 128-row tile over a single key tile."""
    kc, vc, tbl, ln, qs, q = _setup([64], [32], 4, 1, 128, 16, dtype, 3)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128))
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128)), "one tile")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_whole_prompts(dtype):
    """Whole prompts (qlen = n): the first rows see one key; several query and
    key tiles with the causal edge inside them; a bf16 P adds its residual."""
    lens = [200, 130, 37, 300]
    kc, vc, tbl, ln, qs, q = _setup(lens, lens, 8, 2, 128, 16, dtype, 5)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128))
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128)), "whole prompts")


@pytest.mark.parametrize("H,Hkv", [(4, 4), (8, 4), (32, 8), (32, 4), (16, 2), (16, 1), (128, 1)])
@pytest.mark.parametrize("bs,dtype", [(16, torch.bfloat16), (8, torch.float16),
                                      (32, torch.bfloat16)])
def test_mixed_query_lengths(H, Hkv, bs, dtype):
    """Every power-of-two grouping G = 1 .. 128, every block size: decode rows,
    a few draft tokens, whole prompts, a chunk, an empty query list."""
    lens = [1, 37, 200, 390, 64, 71, 5, 1000]
    qlens = [1, 6, 200, 130, 1, 0, 5, 300]
    kc, vc, tbl, ln, qs, q = _setup(lens, qlens, H, Hkv, 128, bs, dtype, H + bs)
    scale = 1 / math.sqrt(128)
    out = _gpu(kc, vc, tbl, ln, qs, q, scale)
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, scale), "G=%d bs=%d" % (H // Hkv, bs))


def test_chunk_of_512():
    """Two sequences each prefilling a 512-token chunk on top of 3584 cached
    tokens (GQA 32 / 8, bf16), every row checked."""
    kc, vc, tbl, ln, qs, q = _setup([4096, 4096], [512, 512], 32, 8, 128, 16, torch.bfloat16, 22)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128))
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128)), "chunk 512")


def test_chunk_of_2048_whole_tiles():
    """The benchmark's shape, one sequence: a 2048-token chunk on 6144 cached
    tokens (GQA 32 / 8, bf16).  A tile is 32 tokens x the 4 heads of a KV head;
    whole tiles are checked at the chunk's start, at tile edges inside it and
    at its end (every head of every token of each): tokens t attend to
    6144 + t + 1 keys."""
    n, qlen, H, Hkv, d = 8192, 2048, 32, 8, 128
    kc, vc, tbl, ln, qs, q = _setup([n], [qlen], H, Hkv, d, 16, torch.bfloat16, 23)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(d)).cpu()
    assert binding.pa_check_device_errors() == 0
    for t0 in list(range(0, qlen, 128)) + [32, 2016]:
        ref = oracle.multi_query(wl.bits(q[t0:t0 + 32]), [0, 32], wl.bits(kc), wl.bits(vc), tbl,
                                 [n - qlen + t0 + 32], 1 / math.sqrt(d), oracle.DTYPE_BF16,
                                 num_threads=THREADS)
        assert_close(out[t0:t0 + 32], ref, "chunk 2048 tokens %d.." % t0)


def test_matches_the_mma_sync_kernel():
    """The same prefill through pa_multi_query (the mma.sync kernel) and
    pa_multi_query_tc: both within tolerance of the oracle and of each other."""
    kc, vc, tbl, ln, qs, q = _setup([700, 1500], [300, 256], 16, 4, 128, 16, torch.float16, 9)
    scale = 1 / math.sqrt(128)
    a = _gpu(kc, vc, tbl, ln, qs, q, scale)
    ws = torch.empty(binding.pa_multi_query_workspace_size(2, 16, 4, 128, 300), dtype=torch.uint8,
                     device="cuda")
    binding.pa_decode_workspace_init(ws)
    b = torch.empty_like(a)
    binding.pa_multi_query(q.cuda(), torch.from_numpy(qs).cuda(), kc.cuda(), vc.cuda(),
                           torch.from_numpy(tbl).cuda(), torch.from_numpy(ln).cuda(), 300, scale,
                           b, ws)
    assert binding.pa_check_device_errors() == 0
    ref = _ref(kc, vc, tbl, ln, qs, q, scale)
    assert_close(a.cpu(), ref, "tcgen05")
    assert_close(b.cpu(), ref, "mma.sync")


def test_repeat_is_deterministic():
    kc, vc, tbl, ln, qs, q = _setup([3000, 333], [600, 200], 32, 8, 128, 32, torch.bfloat16, 12)
    a = _gpu(kc, vc, tbl, ln, qs, q, 0.09)
    for _ in range(3):
        assert torch.equal(a, _gpu(kc, vc, tbl, ln, qs, q, 0.09))
    assert binding.pa_check_device_errors() == 0


def test_many_sequences():
    """300 sequences of short prompts prefilled whole (more items than CTAs,
    items of different lengths dealt over the CTAs)."""
    rng = np.random.default_rng(41)
    lens = rng.integers(1, 400, size=300)
    kc, vc, tbl, ln, qs, q = _setup(lens, lens, 8, 1, 128, 16, torch.bfloat16, 41)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128))
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128)), "300 prompts")


def test_bad_inputs_are_flagged_and_skipped():
    """A sequence with more queries than cached tokens is skipped and flagged;
    a table entry outside the pool reads zeros and is flagged."""
    kc, vc, tbl, ln, qs, q = _setup([10, 200], [3, 150], 8, 2, 128, 16, torch.float16, 26)
    ln_bad = ln.copy()
    ln_bad[0] = 2
    out = _gpu(kc, vc, tbl, ln_bad, qs, q, 0.125)
    assert binding.pa_check_device_errors() & binding.DEVERR["CONTEXT"]
    assert torch.isnan(out[:3].float()).all()
    assert_close(out[3:].cpu(), _ref(kc, vc, tbl, ln, qs, q, 0.125)[3:], "the valid sequence")
    tbl_bad = tbl.copy()
    tbl_bad[1, 2] = kc.shape[0] + 5
    _gpu(kc, vc, tbl_bad, ln, qs, q, 0.125)
    assert binding.pa_check_device_errors() & binding.DEVERR["BLOCK_ID"]


@pytest.mark.parametrize("H,Hkv,d,qlen", [(28, 4, 128, 40), (8, 2, 64, 8)])
def test_unsupported_shapes_are_refused(H, Hkv, d, qlen):
    """Head dim 64; a grouping that is not a power of two with more rows per
    sequence than one tile holds (40 tokens x 7 heads)."""
    kc, vc, tbl, ln, qs, q = _setup([60], [qlen], H, Hkv, d, 16, torch.float16, 27)
    with pytest.raises(binding.PaError) as e:
        _gpu(kc, vc, tbl, ln, qs, q, 0.1)
    assert binding.STATUS_NAMES[e.value.status] == "PA_ERR_UNSUPPORTED"
    assert binding.pa_check_device_errors() == 0


# ---- the split mode: one query tile per (sequence, KV head) ---------------------


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_speculative_verification_full_size(dtype):
    """128 sequences of the Qwen long-tail shape (28 / 4 heads: G = 7, 42 rows
    a tile) verifying 6 tokens each; the long contexts are split over CTAs."""
    w = wl.qwen_longtail(16)
    lens = np.asarray(w.context_lens, np.int64) + 6
    kc, vc, tbl, ln, qs, q = _setup(lens, [6] * w.B, w.H, w.Hkv, w.d, 16, dtype, 21)
    out = _gpu(kc, vc, tbl, ln, qs, q, w.scale)
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, w.scale), "speculative 128 x 6")


@pytest.mark.parametrize("H,Hkv", [(28, 4), (12, 4), (4, 4), (40, 8), (96, 1), (8, 1)])
@pytest.mark.parametrize("bs,dtype", [(16, torch.bfloat16), (8, torch.float16),
                                      (32, torch.bfloat16)])
def test_split_mode_mixed(H, Hkv, bs, dtype):
    """Groupings 1 .. 96 (powers of two and not), every block size: decode rows,
    a few draft tokens, one-token contexts, empty query lists, long contexts
    split between CTAs."""
    G = H // Hkv
    mq = max(1, min(6, 128 // G))
    lens = [1, 37, 6000, 300, 64, 71, 5, 1000, 17000]
    qlens = [1, min(mq, 6), mq, 1, 0, mq, min(5, mq), mq, 2 if mq >= 2 else 1]
    kc, vc, tbl, ln, qs, q = _setup(lens, qlens, H, Hkv, 128, bs, dtype, H + bs + 7)
    scale = 1 / math.sqrt(128)
    out = _gpu(kc, vc, tbl, ln, qs, q, scale)
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, scale), "split G=%d bs=%d" % (G, bs))


def test_split_mode_one_tile_rows():
    """Rows filling a whole tile in the split mode: 32 tokens x 4 heads over
    long contexts, two sequences (both split over many CTAs)."""
    kc, vc, tbl, ln, qs, q = _setup([30000, 9000], [32, 32], 16, 4, 128, 16, torch.bfloat16, 61)
    out = _gpu(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128))
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), _ref(kc, vc, tbl, ln, qs, q, 1 / math.sqrt(128)), "32 x 4 rows")


def test_split_mode_reuses_its_workspace():
    """Few sequences over long contexts (every pair split between CTAs): a
    reused workspace must come back with every ticket at zero, and repeats are
    bit-identical."""
    kc, vc, tbl, ln, qs, q = _setup([20000, 333, 9000], [6, 1, 6], 28, 4, 128, 16,
                                    torch.bfloat16, 25)
    ws = _workspace(3, 28, 4)
    a = _gpu(kc, vc, tbl, ln, qs, q, 0.09, ws=ws)
    for _ in range(3):
        assert torch.equal(a, _gpu(kc, vc, tbl, ln, qs, q, 0.09, ws=ws))
    assert binding.pa_check_device_errors() == 0
    assert_close(a.cpu(), _ref(kc, vc, tbl, ln, qs, q, 0.09), "split pairs")


def test_split_mode_matches_the_decode():
    """One query token per sequence is the decode: the split mode equals the
    oracle's decode of the same batch."""
    lens = [300, 1, 1000, 64, 5000]
    kc, vc, tbl, ln, qs, q = _setup(lens, [1] * 5, 8, 2, 128, 16, torch.float16, 24)
    out = _gpu(kc, vc, tbl, ln, qs, q, 0.1)
    assert binding.pa_check_device_errors() == 0
    ref = oracle.decode(wl.bits(q), wl.bits(kc), wl.bits(vc), tbl, ln, 0.1, oracle.DTYPE_F16,
                        num_threads=THREADS)
    assert_close(out.cpu(), ref, "decode rows")


def test_split_mode_flags_bad_inputs():
    """More queries than max_q_len promised, or than cached tokens: skipped
    and flagged; the other sequences are right."""
    kc, vc, tbl, ln, qs, q = _setup([10, 200, 50], [3, 6, 4], 28, 4, 128, 16, torch.float16, 28)
    ln_bad = ln.copy()
    ln_bad[0] = 2
    out = _gpu(kc, vc, tbl, ln_bad, qs, q, 0.125, max_q_len=6)
    assert binding.pa_check_device_errors() & binding.DEVERR["CONTEXT"]
    assert torch.isnan(out[:3].float()).all()
    assert_close(out[3:].cpu(), _ref(kc, vc, tbl, ln, qs, q, 0.125)[3:], "the valid sequences")
    out = _gpu(kc, vc, tbl, ln, qs, q, 0.125, max_q_len=5)   # sequence 1 has 6
    assert binding.pa_check_device_errors() & binding.DEVERR["CONTEXT"]
    assert torch.isnan(out[3:9].float()).all()
