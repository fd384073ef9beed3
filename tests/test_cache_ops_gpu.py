"""GPU parity of the KV append (pa_reshape_and_cache) and the copy-on-write
block copy (pa_copy_blocks) against the oracle's plain scatter and copy:
bit-exact, with padding slots skipped and bad indices flagged."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_103_gb300 import build
    build.build()
    binding.load()


def _eq(a, b):
    return torch.equal(a.cpu().view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("T,N,bs,Hkv,d,dtype", [(4, 64, 16, 2, 64, torch.float16),
                                                (256, 400, 16, 4, 128, torch.bfloat16),
                                                (1000, 3000, 8, 8, 128, torch.bfloat16),
                                                (77, 50, 32, 40, 128, torch.float16)])
def test_reshape_and_cache_bit_exact(T, N, bs, Hkv, d, dtype):
    rng = np.random.default_rng(T)
    slots = rng.choice(N * bs, size=T, replace=False).astype(np.int64)
    slots[::7] = -1                                   # padding tokens are skipped
    kc = wl.normal_tensor((N, bs, Hkv, d), dtype, 1)
    vc = wl.normal_tensor((N, bs, Hkv, d), dtype, 2)
    kn = wl.normal_tensor((T, Hkv, d), dtype, 3)
    vn = wl.normal_tensor((T, Hkv, d), dtype, 4)
    dk, dv = kc.cuda(), vc.cuda()
    binding.pa_reshape_and_cache(kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda(), dk, dv)
    assert binding.pa_check_device_errors() == 0
    oracle.reshape_and_cache(kn, vn, slots, kc, vc)
    assert _eq(dk, kc) and _eq(dv, vc)


def test_reshape_and_cache_flags_out_of_range_slot():
    N, bs, Hkv, d = 8, 16, 2, 64
    kc = torch.zeros(N, bs, Hkv, d, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    kn = torch.ones(2, Hkv, d, dtype=torch.float16, device="cuda")
    slots = torch.tensor([N * bs, 3], dtype=torch.int64, device="cuda")
    binding.pa_reshape_and_cache(kn, kn, slots, kc, vc)
    assert binding.pa_check_device_errors() & binding.DEVERR["SLOT"]
    assert torch.count_nonzero(kc).item() == Hkv * d          # only slot 3 written
    assert torch.equal(kc[0, 3], kn[1])


@pytest.mark.parametrize("layers", [1, 3, 40])
def test_copy_blocks_bit_exact(layers):
    N, bs, Hkv, d = 300, 16, 4, 128
    ks = [wl.normal_tensor((N, bs, Hkv, d), torch.bfloat16, 10 + l) for l in range(layers)]
    vs = [wl.normal_tensor((N, bs, Hkv, d), torch.bfloat16, 100 + l) for l in range(layers)]
    rng = np.random.default_rng(layers)
    perm = rng.permutation(N)
    pairs = [(int(perm[i]), int(perm[i + 128])) for i in range(100)]
    dk = [t.cuda() for t in ks]
    dv = [t.cuda() for t in vs]
    binding.pa_copy_blocks(dk, dv, torch.tensor(pairs, dtype=torch.int32).cuda())
    assert binding.pa_check_device_errors() == 0
    oracle.copy_blocks(ks, vs, pairs)
    for a, b in zip(dk + dv, ks + vs):
        assert _eq(a, b)


def test_copy_blocks_flags_bad_pair():
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    kc[1] = 1
    binding.pa_copy_blocks([kc], [vc], torch.tensor([[1, 9], [1, 2]], dtype=torch.int32).cuda())
    assert binding.pa_check_device_errors() & binding.DEVERR["PAIR"]
    assert torch.equal(kc[2], kc[1])
