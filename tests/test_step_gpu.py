"""GPU parity of the decode step executor (pa_step_*): each step's slots,
tables and lengths equal the oracle allocator model's bit for bit, the caches
after the step's copy-on-write and append equal the oracle's bit for bit, and
the output matches the fp64 oracle decode, |gpu - ref| <= 2e-3 + 1e-2 |ref|."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import workloads as wl

from _harness import THREADS, assert_close, bit_equal, nan_tails

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_103_gb300 import build
    build.build()
    binding.load()


def _state(N, bs, Hkv, d, dtype, seed, setup):
    """The product allocator and the oracle model driven through the same
    operations, and a seeded cache whose unused slots hold NaN."""
    order = np.random.default_rng(seed).permutation(N).astype(np.int32)
    cpp = binding.Allocator(N, bs, order)
    model = oracle.BlockManagerModel(N, bs, order)
    setup(cpp)
    setup(model)
    kc = wl.normal_tensor((N, bs, Hkv, d), dtype, seed * 5 + 1)
    vc = wl.normal_tensor((N, bs, Hkv, d), dtype, seed * 5 + 2)
    nan_tails(model, kc, vc)
    return cpp, model, kc, vc


def _step_and_check(step, model, ids, kc_host, vc_host, kc_dev, vc_dev, seed, scale, what):
    B, H, d = step.q.shape
    Hkv = step.k_new.shape[1]
    dt = step.q.dtype
    q = wl.normal_tensor((B, H, d), dt, seed)
    kn = wl.normal_tensor((B, Hkv, d), dt, seed + 1)
    vn = wl.normal_tensor((B, Hkv, d), dt, seed + 2)
    step.q.copy_(q)
    step.k_new.copy_(kn)
    step.v_new.copy_(vn)
    step.run(ids)
    assert binding.pa_check_device_errors() == 0
    slots, pairs = model.append_batch(ids)
    if pairs:
        oracle.copy_blocks([kc_host], [vc_host], pairs)
    oracle.reshape_and_cache(kn, vn, np.asarray(slots, np.int64), kc_host, vc_host)
    tbl, lens = model.export(ids, step.block_tables.shape[1])
    assert np.array_equal(step.slot_mapping.numpy(), np.asarray(slots, np.int64)), what
    assert np.array_equal(step.block_tables.numpy(), tbl), what
    assert np.array_equal(step.context_lens.numpy(), lens), what
    assert bit_equal(kc_dev, kc_host) and bit_equal(vc_dev, vc_host), what
    code = oracle.DTYPE_F16 if dt == torch.float16 else oracle.DTYPE_BF16
    ref = oracle.decode(wl.bits(q), wl.bits(kc_host), wl.bits(vc_host), tbl, lens, scale, code,
                        num_threads=THREADS)
    assert_close(step.out.clone(), ref, what)
    return len(pairs)


@pytest.mark.parametrize("H,Hkv,d,bs,dtype", [(8, 2, 128, 16, torch.float16),
                                              (40, 40, 128, 16, torch.float16),
                                              (28, 4, 128, 8, torch.bfloat16),
                                              (4, 1, 64, 32, torch.bfloat16)])
def test_three_steps_match_the_oracle(H, Hkv, d, bs, dtype):
    B = 12
    lens = np.random.default_rng(H + bs).integers(1, 400, size=B)
    lens[3] = bs            # the step opens a new block
    N = int(sum(math.ceil((n + 3) / bs) for n in lens) * 1.25) + 4

    def setup(a):
        for i, n in enumerate(lens):
            (a.alloc if hasattr(a, "alloc") else a.allocate)(i, int(n))

    cpp, model, kc, vc = _state(N, bs, Hkv, d, dtype, H + d, setup)
    kd, vd = kc.cuda(), vc.cuda()
    max_blocks = int(math.ceil((lens.max() + 3) / bs))
    scale = 1 / math.sqrt(d)
    step = binding.Step(cpp, B, H, Hkv, d, max_blocks, max_blocks * bs, kd, vd, scale)
    ids = list(range(B))
    for k in range(3):
        _step_and_check(step, model, ids, kc, vc, kd, vd, 100 * k + H, scale, "step %d" % k)
    step.close()


def test_copy_on_write_inside_the_step():
    """Six forks of a 37-token prompt share its partial last block: the first
    step copies it for five of them before their appends."""
    B, H, Hkv, d, bs = 6, 8, 4, 64, 16

    def setup(a):
        (a.alloc if hasattr(a, "alloc") else a.allocate)(0, 37)
        for c in range(1, B):
            a.fork(0, c)

    cpp, model, kc, vc = _state(40, bs, Hkv, d, torch.bfloat16, 7, setup)
    kd, vd = kc.cuda(), vc.cuda()
    step = binding.Step(cpp, B, H, Hkv, d, 4, 64, kd, vd, 0.125)
    ids = [2, 0, 5, 1, 4, 3]
    assert _step_and_check(step, model, ids, kc, vc, kd, vd, 11, 0.125, "cow") == B - 1
    assert _step_and_check(step, model, ids, kc, vc, kd, vd, 12, 0.125, "after cow") == 0
    step.close()


def test_bound_refusal_changes_nothing():
    B, H, Hkv, d, bs = 2, 4, 2, 64, 16

    def setup(a):
        (a.alloc if hasattr(a, "alloc") else a.allocate)(0, 20)
        (a.alloc if hasattr(a, "alloc") else a.allocate)(1, 32)

    cpp, model, kc, vc = _state(16, bs, Hkv, d, torch.float16, 9, setup)
    kd, vd = kc.cuda(), vc.cuda()
    step = binding.Step(cpp, B, H, Hkv, d, 2, 32, kd, vd, 0.125)
    before = (cpp.free_list(), cpp.stats())
    with pytest.raises(binding.PaError) as e:
        step.run([0, 1])                     # sequence 1 would reach 33 > 32 tokens
    assert binding.STATUS_NAMES[e.value.status] == "PA_ERR_BOUNDS"
    assert (cpp.free_list(), cpp.stats()) == before
    assert bit_equal(kd, kc) and bit_equal(vd, vc)
    step.close()


@pytest.mark.parametrize("fmt", ["fp8", "int8"])
def test_8bit_cache_with_copy_on_write(fmt):
    """The same step over an FP8 or INT8 cache: forks share a partial last
    block, so the first step copies codes and scales before quantising the
    new rows."""
    B, H, Hkv, d, bs, N = 6, 8, 2, 128, 16, 40

    def setup(a):
        (a.alloc if hasattr(a, "alloc") else a.allocate)(0, 37)
        for c in range(1, B):
            a.fork(0, c)

    order = np.random.default_rng(13).permutation(N).astype(np.int32)
    cpp = binding.Allocator(N, bs, order)
    model = oracle.BlockManagerModel(N, bs, order)
    setup(cpp)
    setup(model)
    w = wl.Workload("fp8_step", B, H, Hkv, d, bs, "bf16", np.full(B, 37, np.int32), N, order, 13)
    c = wl.fp8_cache(w) if fmt == "fp8" else wl.int8_cache(w)
    dev = {k: v.cuda() for k, v in c.items()}
    step = binding.Step(cpp, B, H, Hkv, d, 4, 64, dev["k_codes"], dev["v_codes"], 0.09,
                        k_scale=dev["k_scale"], v_scale=dev["v_scale"], dtype=torch.bfloat16,
                        kv_format=fmt)
    ids = [4, 1, 0, 5, 3, 2]
    for k in range(2):
        q = wl.normal_tensor((B, H, d), torch.bfloat16, 40 + k)
        kn = wl.normal_tensor((B, Hkv, d), torch.bfloat16, 50 + k)
        vn = wl.normal_tensor((B, Hkv, d), torch.bfloat16, 60 + k)
        step.q.copy_(q)
        step.k_new.copy_(kn)
        step.v_new.copy_(vn)
        step.run(ids)
        assert binding.pa_check_device_errors() == 0
        slots, pairs = model.append_batch(ids)
        assert len(pairs) == (B - 1 if k == 0 else 0)
        if pairs:
            oracle.copy_blocks([c["k_codes"], c["k_scale"]], [c["v_codes"], c["v_scale"]], pairs)
        getattr(oracle, "reshape_and_cache_" + fmt)(
            kn, vn, np.asarray(slots, np.int64), c["k_codes"].numpy(), c["v_codes"].numpy(),
            c["k_scale"].numpy(), c["v_scale"].numpy())
        for name in c:
            assert torch.equal(dev[name].cpu(), c[name]), (k, name)
        tbl, lens = model.export(ids, 4)
        assert np.array_equal(step.block_tables.numpy(), tbl)
        ref = getattr(oracle, "decode_" + fmt)(wl.bits(q), oracle.DTYPE_BF16, c["k_codes"].numpy(),
                                               c["v_codes"].numpy(), c["k_scale"].numpy(),
                                               c["v_scale"].numpy(), tbl, lens, 0.09)
        assert_close(step.out.clone(), ref, "%s step %d" % (fmt, k))
    step.close()


def test_two_slots_pipelined():
    """depth 2: step k + 1 is submitted (its host bookkeeping done, its graph
    queued) before step k is waited for; every step's output, slots and
    tables are checked against the oracle replaying the steps in order, and
    the caches at the end."""
    B, H, Hkv, d, bs = 10, 8, 2, 128, 16
    lens = np.random.default_rng(77).integers(1, 300, size=B)

    def setup(a):
        for i, n in enumerate(lens):
            (a.alloc if hasattr(a, "alloc") else a.allocate)(i, int(n))

    N = int(sum(math.ceil((n + 8) / bs) for n in lens) * 1.25) + 4
    cpp, model, kc, vc = _state(N, bs, Hkv, d, torch.float16, 31, setup)
    kd, vd = kc.cuda(), vc.cuda()
    max_blocks = int(math.ceil((lens.max() + 8) / bs))
    step = binding.Step(cpp, B, H, Hkv, d, max_blocks, max_blocks * bs, kd, vd, 0.1, depth=2)
    ids = [3, 1, 4, 0, 5, 9, 2, 6, 8, 7]
    inputs = {}

    def fill(k):
        xs = tuple(wl.normal_tensor(shape, torch.float16, 500 + 3 * k + j)
                   for j, shape in enumerate([(B, H, d), (B, Hkv, d), (B, Hkv, d)]))
        sl = step.slot(k % 2)
        for name, x in zip(("q", "k_new", "v_new"), xs):
            sl[name].copy_(x)
        inputs[k] = xs

    def check(k):
        step.wait(k % 2)
        q, kn, vn = inputs[k]
        slots, pairs = model.append_batch(ids)
        assert not pairs
        oracle.reshape_and_cache(kn, vn, np.asarray(slots, np.int64), kc, vc)
        tbl, lens_ = model.export(ids, max_blocks)
        sl = step.slot(k % 2)
        assert np.array_equal(sl["slot_mapping"].numpy(), np.asarray(slots, np.int64))
        assert np.array_equal(sl["block_tables"].numpy(), tbl)
        assert np.array_equal(sl["context_lens"].numpy(), lens_)
        ref = oracle.decode(wl.bits(q), wl.bits(kc), wl.bits(vc), tbl, lens_, 0.1,
                            oracle.DTYPE_F16, num_threads=THREADS)
        assert_close(sl["out"].clone(), ref, "pipelined step %d" % k)

    steps = 6
    for k in range(steps):
        if k >= 2:
            check(k - 2)          # frees slot k % 2 for step k
        fill(k)
        assert step.submit(ids) == k % 2
    for k in range(steps - 2, steps):
        check(k)
    assert binding.pa_check_device_errors() == 0
    assert bit_equal(kd, kc) and bit_equal(vd, vc)
    step.close()


@pytest.mark.parametrize("streams", [1, 2])
def test_pipelined_forks_frees_and_copy_on_write(streams):
    """depth 2 with the batch changing under the executor: before each submit
    one sequence of the batch is freed (the step before, which reads it, may
    still run) and a fork of another takes its place, so the fork's first
    append copies its parent's partial last block.  The pool has no spare
    blocks, so freed blocks come back as copy destinations and new blocks
    while the previous step is in flight.  The oracle model replays the same
    operations in order; every step's slots, tables, output and the final
    caches are checked.  With two streams consecutive steps are submitted on
    different streams (double-buffering by stream): the executor must still
    run each step's kernels after the previous step's decode."""
    B, H, Hkv, d, bs = 8, 8, 2, 128, 16
    rng = np.random.default_rng(1)
    lens = rng.integers(20, 120, size=B)
    lens = np.where(lens % bs == 0, lens + 3, lens)
    N = int(sum(math.ceil(int(n) / bs) for n in lens))
    order = np.random.default_rng(1001).permutation(N).astype(np.int32)
    cpp = binding.Allocator(N, bs, order)
    model = oracle.BlockManagerModel(N, bs, order)
    for i, n in enumerate(lens):
        cpp.alloc(i, int(n))
        model.allocate(i, int(n))
    kc = wl.normal_tensor((N, bs, Hkv, d), torch.float16, 71)
    vc = wl.normal_tensor((N, bs, Hkv, d), torch.float16, 72)
    nan_tails(model, kc, vc)
    kd, vd = kc.cuda(), vc.cuda()
    steps = 12
    max_blocks = int(math.ceil((lens.max() + steps + 1) / bs)) + 1
    step = binding.Step(cpp, B, H, Hkv, d, max_blocks, max_blocks * bs, kd, vd, 0.1, depth=2)
    ids = list(range(B))
    log, inputs, cows = [], {}, []
    replayed = [0]
    subs = [torch.cuda.Stream() for _ in range(streams)]

    def fill(k):
        xs = tuple(wl.normal_tensor(shape, torch.float16, 900 + 3 * k + j)
                   for j, shape in enumerate([(B, H, d), (B, Hkv, d), (B, Hkv, d)]))
        sl = step.slot(k % 2)
        for name, x in zip(("q", "k_new", "v_new"), xs):
            sl[name].copy_(x)
        inputs[k] = xs

    def check(k):
        step.wait(k % 2)
        while True:
            op = log[replayed[0]]
            replayed[0] += 1
            if op[0] == "free":
                model.free(op[1])
            elif op[0] == "fork":
                model.fork(op[1], op[2])
            else:
                break
        _, kk, ids_k = op
        assert kk == k
        q, kn, vn = inputs[k]
        slots, pairs = model.append_batch(ids_k)
        if pairs:
            oracle.copy_blocks([kc], [vc], pairs)
        oracle.reshape_and_cache(kn, vn, np.asarray(slots, np.int64), kc, vc)
        cows.append(len(pairs))
        tbl, lens_ = model.export(ids_k, max_blocks)
        sl = step.slot(k % 2)
        assert np.array_equal(sl["slot_mapping"].numpy(), np.asarray(slots, np.int64)), k
        assert np.array_equal(sl["block_tables"].numpy(), tbl), k
        assert np.array_equal(sl["context_lens"].numpy(), lens_), k
        ref = oracle.decode(wl.bits(q), wl.bits(kc), wl.bits(vc), tbl, lens_, 0.1,
                            oracle.DTYPE_F16, num_threads=THREADS)
        assert_close(sl["out"].clone(), ref, "step %d with forks and frees" % k)

    for k in range(steps):
        if k >= 2:
            check(k - 2)          # frees slot k % 2 for step k
        if k >= 1:
            j = (3 * k) % B
            x, parent, child = ids[j], ids[(j + 1 + k % (B - 1)) % B], 100 + k
            cpp.free(x)
            log.append(("free", x))
            cpp.fork(parent, child)
            log.append(("fork", parent, child))
            ids[j] = child
        fill(k)
        log.append(("step", k, list(ids)))
        assert step.submit(ids, subs[k % streams]) == k % 2
    for k in range(steps - 2, steps):
        check(k)
    torch.cuda.synchronize()
    assert sum(cows) >= steps - 2
    assert binding.pa_check_device_errors() == 0
    assert bit_equal(kd, kc) and bit_equal(vd, vc)
    step.close()
