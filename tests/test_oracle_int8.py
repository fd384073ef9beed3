"""Pins for the INT8 KV-cache part of the oracle ("LLM推理优化技术地图：从KV Cache
到量化与投机解码", section 4.3; the format is a reading: symmetric, one fp32 scale
per (token, KV head), s = fl32(amax / 127)).

The encoder is checked on exact integers, ties (which must go to the even
neighbour) and saturation; the row quantiser against the nearest-multiple
property and its extremes; the INT8 decode against a library attention
routine on the dequantised rows, also through the allocator's slots.
"""
import math

import numpy as np
import torch

from paged_kv_cache_103_gb300 import workloads as wl

from test_oracle_pins import _contiguous_reference


def test_encoder_integers_ties_and_saturation(oracle_mod):
    ints = np.arange(-127, 128, dtype=np.float32)
    assert np.array_equal(oracle_mod.int8_encode(ints).view(np.int8), ints.astype(np.int8))
    halves = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, -126.5], np.float32)
    assert oracle_mod.int8_encode(halves).view(np.int8).tolist() == [0, 2, 2, 0, -2, -2, 126, -126]
    near = np.array([2.4999998, 2.5000002, -7.5000005], np.float32)
    assert oracle_mod.int8_encode(near).view(np.int8).tolist() == [2, 3, -8]
    big = np.array([127.4, 127.6, 300.0, -128.0, -1e30, 1e30], np.float32)
    assert oracle_mod.int8_encode(big).view(np.int8).tolist() == [127, 127, 127, -127, -127, 127]


def test_row_quantiser_nearest_multiple_and_extremes(oracle_mod):
    rng = np.random.default_rng(17)
    x = rng.normal(0, 1, (300, 128)).astype(np.float32)
    x[5] = 0.0                                              # an all-zero row
    x[6] = 0.0
    x[6, 9] = -3.0                                          # one non-zero element
    codes, s = oracle_mod.quantize_rows_int8(x)
    assert s[5] == 0 and not codes[5].any()
    c = codes.view(np.int8).astype(np.float64)
    assert c[6, 9] == -127 and not np.delete(c[6], 9).any()
    big = np.argmax(np.abs(x), axis=1)
    for r in range(300):
        if r != 5:
            assert abs(c[r, big[r]]) == 127
            assert s[r] == np.float32(np.max(np.abs(x[r])) / np.float32(127))
    # every code is a nearest multiple of s: |x - c s| <= s / 2 (up to the
    # fp32 rounding of x / s)
    err = np.abs(x.astype(np.float64) - c * s[:, None].astype(np.float64))
    assert (err <= s[:, None] * (0.5 + 1e-6) + 1e-30).all()


def _pool(rng, lens, bs, extra=3):
    nbs = [(int(n) + bs - 1) // bs for n in lens]
    N = sum(nbs) + extra
    perm = rng.permutation(N)
    tbl = np.full((len(lens), max(nbs)), -1, np.int32)
    off = 0
    for i, nb in enumerate(nbs):
        tbl[i, :nb] = perm[off: off + nb]
        off += nb
    return N, tbl


def test_int8_decode_matches_sdpa_on_dequantised_rows(oracle_mod):
    rng = np.random.default_rng(19)
    B, H, Hkv, d, bs = 3, 8, 2, 128, 16
    lens = np.array([37, 100, 16], np.int32)
    N, tbl = _pool(rng, lens, bs)
    g = torch.Generator().manual_seed(20)
    K = torch.randn(N, bs, Hkv, d, generator=g).to(torch.bfloat16)
    V = torch.randn(N, bs, Hkv, d, generator=g).to(torch.bfloat16)
    q = torch.randn(B, H, d, generator=g).to(torch.bfloat16)
    kq, ks = oracle_mod.quantize_rows_int8(K.float().numpy())
    vq, vs = oracle_mod.quantize_rows_int8(V.float().numpy())
    k_scale = np.ascontiguousarray(ks.transpose(0, 2, 1))   # [N, Hkv, bs]
    v_scale = np.ascontiguousarray(vs.transpose(0, 2, 1))
    scale = 1.0 / math.sqrt(d)
    out = oracle_mod.decode_int8(wl.bits(q), 1, kq, vq, k_scale, v_scale, tbl, lens, scale)
    Kd = kq.view(np.int8).astype(np.float64) * ks[..., None]
    Vd = vq.view(np.int8).astype(np.float64) * vs[..., None]
    for i in range(B):
        rows = [(tbl[i, j // bs], j % bs) for j in range(int(lens[i]))]
        Ki = np.stack([Kd[b, r] for b, r in rows])
        Vi = np.stack([Vd[b, r] for b, r in rows])
        ref = _contiguous_reference(q[i].double().numpy(), Ki, Vi, scale, H // Hkv)
        np.testing.assert_allclose(out[i], ref, rtol=1e-11, atol=1e-13)
    # and it is not the E4M3 reading of the same bytes
    other = oracle_mod.decode_fp8(wl.bits(q), 1, kq, vq, k_scale, v_scale, tbl, lens, scale)
    assert not np.allclose(other, out)


def test_int8_append_then_decode_through_the_allocator(oracle_mod):
    bs, N, Hkv, d, n = 8, 20, 2, 64, 45
    m = oracle_mod.BlockManagerModel(N, bs, np.random.default_rng(5).permutation(N))
    m.allocate(0, 0)
    slots = np.array([m.append_slot(0)[0] for _ in range(n)])
    g = torch.Generator().manual_seed(6)
    K = torch.randn(n, Hkv, d, generator=g).to(torch.float16)
    V = torch.randn(n, Hkv, d, generator=g).to(torch.float16)
    q = torch.randn(1, 4, d, generator=g).to(torch.float16)
    kc = np.zeros((N, bs, Hkv, d), np.uint8)
    vc = np.zeros_like(kc)
    ksc = np.zeros((N, Hkv, bs), np.float32)
    vsc = np.zeros_like(ksc)
    oracle_mod.reshape_and_cache_int8(K, V, slots, kc, vc, ksc, vsc)
    tbl, lens = m.export([0])
    out = oracle_mod.decode_int8(wl.bits(q), 0, kc, vc, ksc, vsc, tbl, lens, 1 / math.sqrt(d))
    kq, ks = oracle_mod.quantize_rows_int8(K.float().numpy())
    vq, vs = oracle_mod.quantize_rows_int8(V.float().numpy())
    Kd = kq.view(np.int8).astype(np.float64) * ks[..., None]
    Vd = vq.view(np.int8).astype(np.float64) * vs[..., None]
    ref = _contiguous_reference(q[0].double().numpy(), Kd, Vd, 1 / math.sqrt(d), 2)
    np.testing.assert_allclose(out[0], ref, rtol=1e-11, atol=1e-13)
