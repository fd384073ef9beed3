"""Pins for the FP8 (E4M3) KV-cache part of the oracle.

The code table is checked against torch's float8_e4m3fn for all 256 codes,
the encoder against torch's round-to-nearest-even conversion and against
explicit ties, the per-row quantiser against its error bound, and the FP8
decode against a library attention routine on the dequantised rows.
"""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_103_gb300 import workloads as wl

from test_oracle_pins import _contiguous_reference

fp8 = getattr(torch, "float8_e4m3fn", None)
needs_fp8 = pytest.mark.skipif(fp8 is None, reason="torch without float8_e4m3fn")


@needs_fp8
def test_code_table_matches_torch_for_all_codes(oracle_mod):
    codes = np.arange(256, dtype=np.uint32).astype(np.uint8)
    got = oracle_mod.e4m3_to_double(codes)
    ref = torch.from_numpy(codes.copy()).view(fp8).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


@needs_fp8
def test_encoder_matches_torch_rne_in_range(oracle_mod):
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 1e-2, 5000),
                        rng.normal(0, 3e-3, 5000)]).astype(np.float32)
    got = oracle_mod.e4m3_encode(x)
    ref = torch.from_numpy(x).to(fp8).view(torch.uint8).numpy()
    # +0 / -0 may differ only in sign of a zero result
    same = (got == ref) | ((got & 0x7F) == 0) & ((ref & 0x7F) == 0)
    assert same.all(), (x[~same][:5], got[~same][:5], ref[~same][:5])


def test_encoder_ties_go_to_even_and_saturate(oracle_mod):
    x = np.array([1.0625, 1.1875, 1.0, 448.0, 460.0, 1e6, -1e6, 2.0 ** -10, 3 * 2.0 ** -10],
                 np.float32)
    codes = oracle_mod.e4m3_encode(x)
    vals = oracle_mod.e4m3_to_double(codes)
    assert vals.tolist()[:3] == [1.0, 1.25, 1.0]          # ties to the even mantissa
    assert vals.tolist()[3:7] == [448.0, 448.0, 448.0, -448.0]   # saturation
    assert vals[7] == 0.0                                  # half the smallest subnormal -> 0 (even)
    assert vals[8] == 2.0 ** -8                            # 1.5 subnormal steps -> 2 (even)


def test_row_quantiser_error_bound_and_extremes(oracle_mod):
    rng = np.random.default_rng(7)
    x = rng.normal(0, 1, (200, 128)).astype(np.float32)
    x[3] = 0.0                                             # an all-zero row
    codes, s = oracle_mod.quantize_rows(x)
    assert s[3] == 0 and not codes[3].any()
    deq = oracle_mod.e4m3_to_double(codes) * s[:, None].astype(np.float64)
    # each row's largest magnitude maps to the largest code
    big = np.argmax(np.abs(x), axis=1)
    for r in range(200):
        if r != 3:
            assert codes[r, big[r]] & 0x7F == 0x7E
    # E4M3 has 3 mantissa bits: relative error <= 2^-4 for normals, and an
    # absolute error <= half a subnormal step (2^-10 * s) below 2^-6 * s
    err = np.abs(deq - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s[:, None] * 2.0 ** -10) * (1 + 1e-6)
    assert (err <= bound).all()


def test_fp8_decode_matches_sdpa_on_dequantised_rows(oracle_mod):
    rng = np.random.default_rng(11)
    B, H, Hkv, d, bs = 3, 8, 2, 128, 16
    lens = np.array([37, 100, 16], np.int32)
    nbs = [(int(n) + bs - 1) // bs for n in lens]
    N = sum(nbs) + 3
    perm = rng.permutation(N)
    tbl = np.full((B, max(nbs)), -1, np.int32)
    off = 0
    for i, nb in enumerate(nbs):
        tbl[i, :nb] = perm[off: off + nb]
        off += nb
    g = torch.Generator().manual_seed(12)
    K = torch.randn(N, bs, Hkv, d, generator=g).to(torch.bfloat16)
    V = torch.randn(N, bs, Hkv, d, generator=g).to(torch.bfloat16)
    q = torch.randn(B, H, d, generator=g).to(torch.bfloat16)
    kq, ks = oracle_mod.quantize_rows(K.float().numpy())
    vq, vs = oracle_mod.quantize_rows(V.float().numpy())
    k_scale = np.ascontiguousarray(ks.transpose(0, 2, 1))   # [N, Hkv, bs]
    v_scale = np.ascontiguousarray(vs.transpose(0, 2, 1))
    scale = 1.0 / math.sqrt(d)
    out = oracle_mod.decode_fp8(wl.bits(q), 1, kq, vq, k_scale, v_scale, tbl, lens, scale)
    Kd = oracle_mod.e4m3_to_double(kq) * ks[..., None]
    Vd = oracle_mod.e4m3_to_double(vq) * vs[..., None]
    for i in range(B):
        rows = [(tbl[i, j // bs], j % bs) for j in range(int(lens[i]))]
        Ki = np.stack([Kd[b, r] for b, r in rows])
        Vi = np.stack([Vd[b, r] for b, r in rows])
        ref = _contiguous_reference(q[i].double().numpy(), Ki, Vi, scale, H // Hkv)
        np.testing.assert_allclose(out[i], ref, rtol=1e-11, atol=1e-13)


def test_fp8_append_then_decode_through_the_allocator(oracle_mod):
    bs, N, Hkv, d, n = 16, 20, 2, 128, 45
    m = oracle_mod.BlockManagerModel(N, bs, np.random.default_rng(3).permutation(N))
    m.allocate(0, 0)
    slots = np.array([m.append_slot(0)[0] for _ in range(n)])
    g = torch.Generator().manual_seed(4)
    K = torch.randn(n, Hkv, d, generator=g).to(torch.float16)
    V = torch.randn(n, Hkv, d, generator=g).to(torch.float16)
    q = torch.randn(1, 4, d, generator=g).to(torch.float16)
    kc = np.zeros((N, bs, Hkv, d), np.uint8)
    vc = np.zeros_like(kc)
    ksc = np.zeros((N, Hkv, bs), np.float32)
    vsc = np.zeros_like(ksc)
    oracle_mod.reshape_and_cache_fp8(K, V, slots, kc, vc, ksc, vsc)
    tbl, lens = m.export([0])
    out = oracle_mod.decode_fp8(wl.bits(q), 0, kc, vc, ksc, vsc, tbl, lens, 1 / math.sqrt(d))
    kq, ks = oracle_mod.quantize_rows(K.float().numpy())
    vq, vs = oracle_mod.quantize_rows(V.float().numpy())
    Kd = oracle_mod.e4m3_to_double(kq) * ks[..., None]
    Vd = oracle_mod.e4m3_to_double(vq) * vs[..., None]
    ref = _contiguous_reference(q[0].double().numpy(), Kd, Vd, 1 / math.sqrt(d), 2)
    np.testing.assert_allclose(out[0], ref, rtol=1e-11, atol=1e-13)
