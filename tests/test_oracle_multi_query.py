"""Pins for the oracle's multi-token query (chunked prefill / speculative
verification over the paged cache; "vLLM 深度拆解：当大模型推理学会「分页注意力」",
section 5).  Reading: a sequence's queries are its last qlen cached tokens and
query r attends to cached tokens 0 .. n - qlen + r.

Each pin is independent of the oracle's own code: torch SDPA in fp64 with an
explicitly built mask on the gathered contiguous K/V; the invariance of a
prompt's rows under cutting it into chunks; and closed forms.
"""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_103_gb300 import workloads as wl


def _pool(rng, lens, bs, N_extra=3):
    nbs = [max(1, math.ceil(n / bs)) for n in lens]
    N = sum(nbs) + N_extra
    perm = rng.permutation(N)
    tbl = np.full((len(lens), max(nbs)), -1, np.int32)
    off = 0
    for i, nb in enumerate(nbs):
        tbl[i, :nb] = perm[off: off + nb]
        off += nb
    return N, tbl


def _gather(cache, tbl_row, n, bs):
    return torch.stack([cache[tbl_row[j // bs], j % bs] for j in range(n)])


def _sdpa_rows(q_rows, K, V, n, G, scale):
    """q_rows [qlen, H, d], K/V [n, Hkv, d] (fp64): causal with offset n - qlen."""
    qlen = q_rows.shape[0]
    Kx = K.repeat_interleave(G, dim=1).permute(1, 0, 2)       # [H, n, d]
    Vx = V.repeat_interleave(G, dim=1).permute(1, 0, 2)
    r = torch.arange(qlen)[:, None]
    j = torch.arange(n)[None, :]
    allowed = j <= (n - qlen + r)                               # [qlen, n]
    mask = torch.zeros(qlen, n, dtype=torch.float64).masked_fill(~allowed, float("-inf"))
    out = torch.nn.functional.scaled_dot_product_attention(
        q_rows.permute(1, 0, 2), Kx, Vx, attn_mask=mask, scale=scale)
    return out.permute(1, 0, 2)                                  # [qlen, H, d]


@pytest.mark.parametrize("H,Hkv,d,bs,dtype", [(4, 2, 64, 16, torch.float16),
                                              (28, 4, 128, 8, torch.bfloat16),
                                              (8, 8, 128, 32, torch.float16)])
def test_multi_query_matches_sdpa_with_causal_offset(oracle_mod, H, Hkv, d, bs, dtype):
    rng = np.random.default_rng(H + bs)
    lens = [37, 6, 70, 1, 129]
    qlens = [6, 6, 33, 1, 5]
    N, tbl = _pool(rng, lens, bs)
    K = wl.normal_tensor((N, bs, Hkv, d), dtype, 1)
    V = wl.normal_tensor((N, bs, Hkv, d), dtype, 2)
    q_start = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = wl.normal_tensor((int(q_start[-1]), H, d), dtype, 3)
    code = oracle_mod.DTYPE_F16 if dtype == torch.float16 else oracle_mod.DTYPE_BF16
    scale = 1 / math.sqrt(d)
    out = oracle_mod.multi_query(wl.bits(q), q_start, wl.bits(K), wl.bits(V), tbl, lens, scale,
                                 code, num_threads=4)
    for i, n in enumerate(lens):
        Ki = _gather(K, tbl[i], n, bs).double()
        Vi = _gather(V, tbl[i], n, bs).double()
        rows = q[q_start[i]:q_start[i + 1]].double()
        ref = _sdpa_rows(rows, Ki, Vi, n, H // Hkv, scale).numpy()
        np.testing.assert_allclose(out[q_start[i]:q_start[i + 1]], ref, rtol=1e-10, atol=1e-12)


def test_chunked_prompt_equals_whole_prompt(oracle_mod):
    """A prompt attended in chunks (each chunk's queries over the cache holding
    everything up to the chunk's end) gives the rows of one whole-prompt call."""
    bs, H, Hkv, d, P = 16, 8, 2, 64, 150
    rng = np.random.default_rng(5)
    N, tbl = _pool(rng, [P], bs)
    K = wl.normal_tensor((N, bs, Hkv, d), torch.float16, 4)
    V = wl.normal_tensor((N, bs, Hkv, d), torch.float16, 5)
    q = wl.normal_tensor((P, H, d), torch.float16, 6)
    whole = oracle_mod.multi_query(wl.bits(q), [0, P], wl.bits(K), wl.bits(V), tbl, [P], 0.125,
                                   oracle_mod.DTYPE_F16)
    rows = []
    for a, b in [(0, 1), (1, 17), (17, 64), (64, 149), (149, 150)]:
        rows.append(oracle_mod.multi_query(wl.bits(q[a:b]), [0, b - a], wl.bits(K), wl.bits(V),
                                           tbl, [b], 0.125, oracle_mod.DTYPE_F16))
    assert np.array_equal(np.concatenate(rows), whole)


def test_closed_forms(oracle_mod):
    bs, H, Hkv, d = 16, 2, 1, 64
    rng = np.random.default_rng(9)
    N, tbl = _pool(rng, [20], bs)
    K = wl.normal_tensor((N, bs, Hkv, d), torch.float16, 7)
    V = wl.normal_tensor((N, bs, Hkv, d), torch.float16, 8)
    q = wl.normal_tensor((20, H, d), torch.float16, 9)
    out = oracle_mod.multi_query(wl.bits(q), [0, 20], wl.bits(K), wl.bits(V), tbl, [20], 0.125,
                                 oracle_mod.DTYPE_F16)
    v0 = V[tbl[0, 0], 0, 0].double().numpy()
    # the first token of a fresh prompt sees only itself
    assert np.array_equal(out[0, 0], v0) and np.array_equal(out[0, 1], v0)
    # with every key equal, each row is the mean of the V rows it sees
    Kc = K.clone()
    Kc[:] = K[tbl[0, 0], 0]
    out = oracle_mod.multi_query(wl.bits(q), [0, 20], wl.bits(Kc), wl.bits(V), tbl, [20], 0.125,
                                 oracle_mod.DTYPE_F16)
    Vi = _gather(V, tbl[0], 20, bs).double()[:, 0]
    for r in (0, 7, 19):
        np.testing.assert_allclose(out[r, 1], Vi[: r + 1].mean(0).numpy(), rtol=1e-12, atol=1e-12)


def test_rejects_more_queries_than_context(oracle_mod):
    K = np.zeros((2, 16, 1, 64), np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.multi_query(np.zeros((5, 1, 64), np.uint16), [0, 5], K, K,
                               np.zeros((1, 1), np.int32), [4], 0.125, 0)
