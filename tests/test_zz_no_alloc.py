"""pa_decode_noalloc against pa_decode.

Callers that cannot allocate device memory (an allocator's own hooks, a host
framework that owns and pre-partitions device memory) use pa_decode_noalloc,
whose scratch is a fixed per-device array inside the library instead of a
caller-supplied workspace.  Its outputs must match the ordinary entry point
within the parity tolerance, on two calls in a row (the second reuses the
array the first left behind).  This file is collected last so that a failing
run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_103_gb300 import build
    build.build()
    binding.load()


def _case(w):
    host = wl.qkv(w, with_new=False)
    rng = np.random.default_rng(w.seed)
    order = rng.permutation(w.num_blocks)
    nbs = [(int(n) + w.block_size - 1) // w.block_size for n in w.context_lens]
    tbl = np.full((w.B, max(nbs)), -1, np.int32)
    off = 0
    for i, nb in enumerate(nbs):
        tbl[i, :nb] = order[off: off + nb]
        off += nb
    dev = {k: v.cuda() for k, v in host.items()}
    return dev, torch.from_numpy(tbl).cuda(), torch.from_numpy(w.context_lens).cuda()


@pytest.mark.parametrize("make", [lambda: wl.gqa7b(8, 4096), lambda: wl.llama13b(B=16),
                                  lambda: wl.tiny()])
def test_noalloc_matches_workspace_entry_point_twice(make):
    w = make()
    t, tbl, lens = _case(w)
    max_len = int(w.context_lens.max())
    ref = torch.empty_like(t["q"])
    ws = torch.empty(binding.pa_decode_workspace_size(w.B, w.H, w.d), dtype=torch.uint8,
                     device="cuda")
    binding.pa_decode_workspace_init(ws)
    binding.pa_decode(t["q"], t["k_cache"], t["v_cache"], tbl, lens, max_len, w.scale, ref, ws)
    for _ in range(2):
        out = torch.full_like(t["q"], float("nan"))
        binding.pa_decode_noalloc(t["q"], t["k_cache"], t["v_cache"], tbl, lens, max_len,
                                  w.scale, out)
        assert binding.pa_check_device_errors() == 0
        a, b = out.double().cpu(), ref.double().cpu()
        assert torch.isfinite(a).all()
        assert ((a - b).abs() <= ATOL + RTOL * b.abs()).all()


def test_noalloc_rejects_batches_beyond_its_scratch():
    q = torch.zeros(1, 1, 128, dtype=torch.bfloat16, device="cuda")
    big_B = 4096
    need = binding.pa_decode_workspace_size(big_B, 4096, 128)
    assert need > (16 << 20)
    lib = binding.load()
    st = lib.pa_decode_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), 1,
                               q.data_ptr(), 16, big_B, 4096, 256, 128, 16, 1, 0.1, 1,
                               q.data_ptr(), None)
    assert st == 6


def test_noalloc_on_a_side_stream_matches_workspace_entry_point():
    """The entry point on a non-default stream, twice in a row: its counter
    clear and its decode are both ordered on that stream."""
    w = wl.gqa7b(8, 4096)
    t, tbl, lens = _case(w)
    max_len = int(w.context_lens.max())
    ref = torch.empty_like(t["q"])
    ws = torch.empty(binding.pa_decode_workspace_size(w.B, w.H, w.d), dtype=torch.uint8,
                     device="cuda")
    binding.pa_decode_workspace_init(ws)
    binding.pa_decode(t["q"], t["k_cache"], t["v_cache"], tbl, lens, max_len, w.scale, ref, ws)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    for _ in range(2):
        out = torch.full_like(t["q"], float("nan"))
        side.wait_stream(torch.cuda.current_stream())
        binding.pa_decode_noalloc(t["q"], t["k_cache"], t["v_cache"], tbl, lens, max_len,
                                  w.scale, out, stream=side)
        assert binding.pa_check_device_errors(side) == 0
        a, b = out.double().cpu(), ref.double().cpu()
        assert torch.isfinite(a).all()
        assert ((a - b).abs() <= ATOL + RTOL * b.abs()).all()
