"""The C-ABI library builds, loads without a GPU and exports every symbol the
header declares; host-side argument checks answer before any device work."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return binding.load()


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "pa.h"), encoding="utf-8") as f:
        text = f.read()
    return sorted(set(re.findall(r"PA_API\s+[^;(]*?\b(pa_\w+)\s*\(", text, flags=re.S)))


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for must in ("pa_decode", "pa_reshape_and_cache", "pa_copy_blocks", "pa_alloc", "pa_free",
                 "pa_append_slot", "pa_fork", "pa_export"):
        assert must in names
    assert set(names) == set(binding.SIGNATURES), set(names) ^ set(binding.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_only_the_abi_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         stdout=subprocess.PIPE, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {s for s in exported if s.startswith("pa_")}
    assert ours == set(_declared_symbols())


def test_status_strings_and_version(lib):
    assert lib.pa_version() == 1
    for s in range(8):
        assert lib.pa_status_str(s)


def test_decode_host_checks_answer_without_a_gpu(lib):
    P = ctypes.c_void_p(16 * 1024)  # never dereferenced: the checks fail first
    # head_dim 96 is outside the supported set
    st = lib.pa_decode(P, P, P, P, 4, P, 64, 2, 4, 2, 96, 16, 8, 0.1, 0, P, P, 1 << 20, None)
    assert st == 6
    # block size 64 unsupported
    st = lib.pa_decode(P, P, P, P, 4, P, 64, 2, 4, 2, 128, 64, 8, 0.1, 0, P, P, 1 << 20, None)
    assert st == 6
    # H not a multiple of Hkv
    st = lib.pa_decode(P, P, P, P, 4, P, 64, 2, 5, 2, 128, 16, 8, 0.1, 0, P, P, 1 << 20, None)
    assert st == 6
    # 17 query heads per KV head: above 16 and not a multiple of 16
    st = lib.pa_decode(P, P, P, P, 4, P, 64, 2, 34, 2, 128, 16, 8, 0.1, 0, P, P, 1 << 20, None)
    assert st == 6
    # workspace too small
    st = lib.pa_decode(P, P, P, P, 4, P, 64, 2, 4, 2, 128, 16, 8, 0.1, 0, P, P, 16, None)
    assert st == 1
    # empty batch is a no-op
    st = lib.pa_decode(None, None, None, None, 4, None, 0, 0, 4, 2, 128, 16, 8, 0.1, 0, None,
                       None, 0, None)
    assert st == 0


def test_workspace_size(lib):
    assert lib.pa_decode_workspace_size(64, 40, 128) > 0
    assert lib.pa_decode_workspace_size(64, 40, 96) == 0
    a = lib.pa_decode_workspace_size(1, 8, 128)
    b = lib.pa_decode_workspace_size(1000, 8, 128)
    assert b > a


def test_cache_op_host_checks(lib):
    P = ctypes.c_void_p(16 * 1024)
    assert lib.pa_reshape_and_cache(P, P, P, 0, P, P, 8, 16, 2, 64, 0, None) == 0   # T = 0
    assert lib.pa_reshape_and_cache(P, P, P, -1, P, P, 8, 16, 2, 64, 0, None) == 1
    assert lib.pa_reshape_and_cache(P, P, P, 1, P, P, 8, 16, 2, 64, 5, None) == 6   # dtype
    assert lib.pa_copy_blocks(None, None, 0, None, 0, 4096, 8, None) == 0
    assert lib.pa_copy_blocks(None, None, 1, None, 1, 4095, 8, None) == 1             # not x16


def test_step_layout_and_argument_checks(lib):
    """The executor's staging layout: every region 256-byte aligned, in the
    documented order, large enough for its tensor; bad descriptions refused."""
    d = binding.StepDesc(64, 40, 40, 128, 16, 5240, 128, 2048, 0, 0.088, 0, 1)
    L = binding.StepLayout()
    assert lib.pa_step_layout_get(ctypes.byref(d), ctypes.byref(L)) == 0
    order = ["q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens", "out"]
    sizes = {"q": 64 * 40 * 128 * 2, "k_new": 64 * 40 * 128 * 2, "v_new": 64 * 40 * 128 * 2,
             "slot_mapping": 64 * 8, "block_tables": 64 * 128 * 4, "context_lens": 64 * 4,
             "out": 64 * 40 * 128 * 2}
    offs = [getattr(L, n) for n in order]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    for a, b in zip(order, order[1:]):
        if a != "context_lens":
            assert getattr(L, b) - getattr(L, a) >= sizes[a]
    assert L.in_bytes == L.cow_pairs and L.in_bytes >= L.context_lens + sizes["context_lens"]
    assert L.out - L.cow_pairs >= 64 * 2 * 4 and L.total >= L.out + sizes["out"]
    for field, bad in [("max_context_len", 2049), ("d", 96), ("block_size", 64), ("B", 0),
                       ("Hkv", 3), ("dtype", 7), ("q8", 3), ("depth", 0), ("depth", 3)]:
        e = binding.StepDesc(64, 40, 40, 128, 16, 5240, 128, 2048, 0, 0.088, 0, 1)
        setattr(e, field, bad)
        assert lib.pa_step_layout_get(ctypes.byref(e), ctypes.byref(L)) == 1, field
    # creation refuses missing buffers before touching the device
    h = ctypes.c_void_p()
    assert lib.pa_step_create(ctypes.byref(d), None, None, None, None, None, None, None, None,
                              0, ctypes.byref(h)) == 1
    e = binding.StepDesc(64, 40, 40, 64, 16, 5240, 128, 2048, 0, 0.088, 1, 1)   # FP8 needs d 128
    assert lib.pa_step_layout_get(ctypes.byref(e), ctypes.byref(L)) == 1
    assert lib.pa_step_run(None, None, None) == 1
    assert lib.pa_step_submit(None, None, None, None) == 1
    assert lib.pa_step_wait(None, 0) == 1


def test_step_refuses_a_cache_of_the_wrong_format(lib):
    """The executor takes raw pool pointers, so the binding checks that the
    cache tensors match kv_format before anything reaches the library: an
    8-bit pool read as a 16-bit one would be written past its end."""
    import torch
    N, bs, Hkv, d = 8, 16, 2, 128
    u8 = torch.zeros((N, bs, Hkv, d), dtype=torch.uint8)
    f16 = torch.zeros((N, bs, Hkv, d), dtype=torch.float16)
    sc = torch.zeros((N, Hkv, bs), dtype=torch.float32)
    alloc = binding.Allocator(N, bs)
    cases = [dict(k_cache=u8, v_cache=u8, k_scale=sc, v_scale=sc, dtype=torch.bfloat16),
             dict(k_cache=u8, v_cache=u8),
             dict(k_cache=f16, v_cache=f16, k_scale=sc, v_scale=sc, dtype=torch.float16,
                  kv_format="int8"),
             dict(k_cache=u8, v_cache=u8, k_scale=sc[:, :1], v_scale=sc, dtype=torch.float16,
                  kv_format="fp8"),
             dict(k_cache=u8, v_cache=u8, k_scale=sc.double(), v_scale=sc.double(),
                  dtype=torch.float16, kv_format="int8")]
    for kw in cases:
        with pytest.raises(ValueError):
            binding.Step(alloc, 2, 4, Hkv, d, 4, 64, scale=0.1, **kw)


def test_step_create_refuses_an_allocator_of_another_pool(lib):
    """The executor indexes the cache with the allocator's blocks and slots, so
    an allocator whose pool or block size differs from the description is
    refused before anything touches a pointer (the pointers here are never
    dereferenced)."""
    fake = ctypes.c_void_p(1 << 20)                     # 256-byte aligned, never used
    ws = lib.pa_decode_workspace_size(4, 8, 128)
    for n, bs in [(64, 16), (32, 8)]:                   # the description says 32 x 16
        a = binding.Allocator(n, bs)
        d = binding.StepDesc(4, 8, 2, 128, 16, 32, 8, 128, 0, 0.088, 0, 1)
        h = ctypes.c_void_p()
        assert lib.pa_step_create(ctypes.byref(d), a._h, fake, fake, None, None, fake, fake, fake,
                                  ws, ctypes.byref(h)) == 1
        assert not h.value


def test_mma_ceiling_argument_checks(lib):
    """The measurement aid refuses bad arguments before touching the device."""
    f = ctypes.c_int64(0)
    sink = ctypes.c_void_p(1 << 20)                     # never dereferenced
    assert lib.pa_measure_mma_ceiling(1, 0, sink, 1 << 20, ctypes.byref(f), None) == 1
    assert lib.pa_measure_mma_ceiling(1, (1 << 20) + 1, sink, 1 << 20, ctypes.byref(f), None) == 1
    assert lib.pa_measure_mma_ceiling(1, 16, None, 1 << 20, ctypes.byref(f), None) == 1
    assert lib.pa_measure_mma_ceiling(1, 16, sink, 1 << 20, None, None) == 1


def _declared_parameter_counts():
    """name -> number of parameters, from every PA_API declaration of pa.h."""
    with open(os.path.join(ROOT, "include", "pa.h"), encoding="utf-8") as f:
        text = re.sub(r"/\*.*?\*/", " ", f.read(), flags=re.S)
    out = {}
    for m in re.finditer(r"PA_API\s+[^;(]*?\b(pa_\w+)\s*\(([^)]*)\)\s*;", text, flags=re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else len(params.split(","))
    return out


def test_binding_signatures_match_the_header():
    """Every ctypes signature of the binding takes as many arguments as the
    header declares (a drift here would pass garbage through the C ABI)."""
    counts = _declared_parameter_counts()
    assert set(counts) == set(binding.SIGNATURES)
    for name, (_, args) in binding.SIGNATURES.items():
        assert len(args) == counts[name], (name, len(args), counts[name])
