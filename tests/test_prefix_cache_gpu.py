"""GPU parity of decoding through prefix-cached blocks.

Every token's K/V row is a fixed function of (token id, position) -- a
token-embedding row plus a position row -- so a block-aligned prefix shared by
two prompts has identical K/V.  Sequences of a multi-turn trace are created
with pa_alloc_prompt; each writes K/V (pa_reshape_and_cache) only for the
tokens the cache did not hold, grows by pa_append_batch_tokens, and turns end
with pa_free.  The decode over the final tables (pa_decode) must match the
fp64 oracle run on a cache the oracle's own allocator model and scatter built
from the same trace, and, for sampled sequences, attention over the
contiguous rows f(token_j, j) -- which holds only if every cached block
really carries the prefix's K/V.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import workloads as wl

from _harness import THREADS, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_103_gb300 import build
    build.build()
    binding.load()


def _rows(emb, pos, tokens, positions):
    return (emb[tokens] + pos[positions]).to(torch.bfloat16)


def _run_trace(trace, N, bs, Hkv, d, emb_k, pos_k, emb_v, pos_v, use_model):
    """Plays the trace on the product allocator + GPU (use_model False) or on
    the oracle's model + host scatter (use_model True).  Returns the final
    tables, lengths, token lists and the cache (device or host)."""
    if use_model:
        alloc = oracle.BlockManagerModel(N, bs, trace["order"])
        kc = torch.zeros(N, bs, Hkv, d, dtype=torch.bfloat16)
    else:
        alloc = binding.Allocator(N, bs, trace["order"])
        kc = torch.zeros(N, bs, Hkv, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    toks = {}
    hit_tokens = prompt_tokens = 0

    def write(sid, start, count):
        if count == 0:
            return
        t = torch.tensor(toks[sid][start:start + count])
        p = torch.arange(start, start + count)
        kn, vn = _rows(emb_k, pos_k, t, p), _rows(emb_v, pos_v, t, p)
        if use_model:
            slots = [alloc.slot_of(sid, start + i) for i in range(count)]
            oracle.reshape_and_cache(kn, vn, slots, kc, vc)
        else:
            slots = torch.from_numpy(alloc.seq_slots(sid, start, count)).cuda()
            binding.pa_reshape_and_cache(kn.cuda(), vn.cuda(), slots, kc, vc)

    for turn in trace["turns"]:
        for sid, prompt in turn["prompts"]:
            toks[sid] = list(prompt)
            cached = (alloc.allocate_prompt(sid, prompt) if use_model
                      else alloc.alloc_prompt(sid, prompt))
            hit_tokens += cached
            prompt_tokens += len(prompt)
            write(sid, cached, len(prompt) - cached)
        for step in turn["replies"]:              # one token per live sequence per step
            ids = [s for s, _ in step]
            tk = [t for _, t in step]
            starts = [len(toks[s]) for s in ids]
            if use_model:
                alloc.append_batch(ids, tk)
            else:
                alloc.append_batch(ids, tokens=tk)
            for s, t, j in zip(ids, tk, starts):
                toks[s].append(t)
                write(s, j, 1)
        for sid in turn["free"]:
            alloc.free(sid)
            del toks[sid]
    live = sorted(toks)
    w = max(math.ceil(len(toks[s]) / bs) for s in live)
    tbl, lens = alloc.export(live, w)
    return live, tbl, lens, toks, kc, vc, hit_tokens / max(prompt_tokens, 1)


@pytest.mark.parametrize("seed", [3, 4])
def test_decode_through_prefix_cached_blocks(seed):
    bs, H, Hkv, d = 16, 28, 4, 128
    tr = wl.multiturn_trace(seed, convs=24, turns=3, system=160)
    g = torch.Generator().manual_seed(seed)
    maxpos = 4096
    emb_k = torch.randn(tr["vocab"], Hkv, d, generator=g)
    pos_k = torch.randn(maxpos, Hkv, d, generator=g) * 0.5
    emb_v = torch.randn(tr["vocab"], Hkv, d, generator=g)
    pos_v = torch.randn(maxpos, Hkv, d, generator=g) * 0.5
    live, tbl, lens, toks, kc, vc, hit = _run_trace(tr, tr["N"], bs, Hkv, d, emb_k, pos_k,
                                                    emb_v, pos_v, use_model=False)
    live2, tbl2, lens2, _, kc2, vc2, hit2 = _run_trace(tr, tr["N"], bs, Hkv, d, emb_k, pos_k,
                                                       emb_v, pos_v, use_model=True)
    assert live == live2 and np.array_equal(tbl, tbl2) and np.array_equal(lens, lens2)
    assert hit == hit2 and hit > 0.7                     # shared system prompt + history
    B = len(live)
    q = wl.normal_tensor((B, H, d), torch.bfloat16, seed)
    out = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(binding.pa_decode_workspace_size(B, H, d), dtype=torch.uint8, device="cuda")
    binding.pa_decode_workspace_init(ws)
    binding.pa_decode(q.cuda(), kc, vc, torch.from_numpy(tbl).cuda(),
                      torch.from_numpy(lens).cuda(), int(lens.max()), 1 / math.sqrt(d), out, ws)
    assert binding.pa_check_device_errors() == 0
    ref = oracle.decode(wl.bits(q), wl.bits(kc2), wl.bits(vc2), tbl2, lens2, 1 / math.sqrt(d),
                        oracle.DTYPE_BF16, num_threads=THREADS)
    assert_close(out.cpu(), ref, "prefix-cached decode")
    # contiguous rows f(token_j, j): the cached blocks hold the prefix's K/V
    G = H // Hkv
    for r in (0, B // 2, B - 1):
        t = torch.tensor(toks[live[r]])
        p = torch.arange(len(t))
        K = _rows(emb_k, pos_k, t, p).double()
        V = _rows(emb_v, pos_v, t, p).double()
        qr = q[r].double()
        for h in range(H):
            s = (K[:, h // G] @ qr[h]) / math.sqrt(d)
            w = torch.softmax(s, 0)
            np.testing.assert_allclose(ref[r, h], (w[:, None] * V[:, h // G]).sum(0).numpy(),
                                       rtol=1e-10, atol=1e-12)
