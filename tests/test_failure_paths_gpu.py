"""Failure paths on the GPU, without faulting it: a bounded wait on an mbarrier
that nothing arrives on gives up, reports PA_DEVERR_TIMEOUT through the error
word and leaves the context usable for the next decode."""
import numpy as np
import pytest
import torch

from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import workloads as wl

from _harness import GpuRun, assert_close, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_103_gb300 import build
    build.build()
    binding.load()


def test_bounded_wait_times_out_and_context_survives():
    assert binding.pa_check_device_errors() == 0
    binding.pa_selftest_wait_timeout(2000)                  # 2 ms on a flag nothing sets
    flags = binding.pa_check_device_errors()
    assert flags & binding.DEVERR["TIMEOUT"]
    assert binding.pa_check_device_errors() == 0            # the word was cleared
    # the context still runs kernels correctly
    w = wl.tiny(77)
    host = wl.qkv(w, with_new=False)
    order = np.random.default_rng(1).permutation(w.num_blocks)
    nbs = [(int(n) + 15) // 16 for n in w.context_lens]
    tbl = np.full((w.B, max(nbs)), -1, np.int32)
    off = 0
    for i, nb in enumerate(nbs):
        tbl[i, :nb] = order[off: off + nb]
        off += nb
    run = GpuRun(w, host)
    out = run.decode(tbl, w.context_lens)
    assert binding.pa_check_device_errors() == 0
    assert_close(out.cpu(), oracle_decode(w, host["q"], host["k_cache"], host["v_cache"], tbl,
                                          w.context_lens), "after-timeout")


def test_selftest_rejects_unbounded_limits():
    with pytest.raises(binding.PaError):
        binding.pa_selftest_wait_timeout(0)
    with pytest.raises(binding.PaError):
        binding.pa_selftest_wait_timeout(2_000_000)
