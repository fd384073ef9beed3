"""The mma.sync throughput-ceiling measurement aid: the launch runs, reports
the operation count its grid implies, leaves finite values and no error flags,
and refuses a sink smaller than its grid."""
import pytest
import torch

from paged_kv_cache_103_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_103_gb300 import build
    build.build()
    binding.load()


@pytest.mark.parametrize("bf16", [False, True])
def test_mma_ceiling_runs_and_counts(bf16):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid = 2 * sms
    sink = torch.full((grid * 256,), float("nan"), dtype=torch.float32, device="cuda")
    flops = binding.pa_measure_mma_ceiling(bf16, 64, sink)
    torch.cuda.synchronize()
    assert flops == 2 * 16 * 8 * 16 * 8 * 64 * grid * 8
    assert torch.isfinite(sink).all()
    assert binding.pa_check_device_errors() == 0


def test_mma_ceiling_refuses_a_small_sink():
    sink = torch.empty(256, dtype=torch.float32, device="cuda")
    with pytest.raises(binding.PaError):
        binding.pa_measure_mma_ceiling(True, 8, sink)
