"""Seeded synthetic workloads for the tests and the benchmark.

This module only draws random inputs of the right shapes, sizes and length
mixes; it holds none of the attention arithmetic and imports neither the CUDA
library nor the oracle, so both sides can take their inputs from it.

The shapes follow the pages' own examples:

* ``tiny``: 4 sequences, lengths uniform in [1, 64], 4 query / 2 KV heads,
  head dim 64, fp16, block size 16, a 64-block pool in random order.
* ``llama13b``: LLaMA-13B-shaped MHA (40 heads of 128, fp16, block size 16),
  batch 64, lengths uniform in [128, 2048] ("LLM推理优化：vLLM PagedAttention
  深度解析与工程实践", section 二 and section 3.1).
* ``gqa7b``: 7B GQA (32 query / 8 KV heads of 128, bf16, block size 16), every
  sequence at full length, (batch, length) in {(1,1024), (8,4096), (8,8192),
  (16,32768)} -- the rows of the KV-size table in "LLM推理优化技术地图：从KV
  Cache到量化与投机解码", section 2.2.
* ``qwen_longtail``: Qwen2.5-7B-shaped (28 query / 4 KV heads of 128, bf16),
  batch 128: 95% of lengths lognormal with median 1500 clipped to [1, 8192]
  and 5% (6 sequences, at seeded positions) uniform in [16384, 24576]; block
  size 8, 16 or 32 (the length mix of the Qwen2.5-7B deployment page at
  mhpq.cn/news/468822, section 1.3: 95% of requests under 8K tokens, a few
  near 20K).  The lognormal sigma (1.0) is not on the page; with it the 95th
  percentile is about 7.8K.
* ``prefix_share``: 256 sequences sharing a 1024-token prefix (64 blocks of
  16) plus unique suffixes uniform in [64, 512]; ``prefix_share_cow`` uses a
  1000-token prefix with no suffix, so the shared last block is partial.
* ``multiturn_trace`` / ``multiturn_prefix``: conversations that all start
  with the same system prompt, several turns each; turn t's prompt is the
  conversation so far plus a new user message, the reply is generated token
  by token, and the previous turn's sequence is freed once the next exists --
  the multi-turn, shared-system-prompt case the prefix-caching pages describe
  ("LLM推理优化：vLLM PagedAttention深度解析与工程实践", section 4.2).  Token ids are
  uniform over a small vocabulary; the sizes are this module's choice.

Pools hold 1.25 x the blocks the lengths need and are handed out in a seeded
random order, so blocks land scattered over the pool.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    d: int
    block_size: int
    dtype: str                      # "f16" or "bf16"
    context_lens: np.ndarray        # int32 [B]: tokens in the cache per sequence
    num_blocks: int                 # pool size N
    free_order: np.ndarray          # int32 [N]: the allocator's initial free list
    seed: int
    layers: int = 1                 # model depth the shape is taken from (tokens/s)
    prefix_len: int = 0             # shared prefix (prefix_share only)
    suffix_lens: np.ndarray | None = None
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "f16" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 2


def _pool(lens, bs, factor=1.25, minimum=0):
    need = int(sum((int(n) + bs - 1) // bs for n in lens))
    return max(int(math.ceil(factor * need)), minimum, 1)


def _perm(n, seed):
    return np.random.default_rng(seed).permutation(n).astype(np.int32)


def tiny(seed: int = 1001) -> Workload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 65, size=4).astype(np.int32)
    return Workload("tiny", 4, 4, 2, 64, 16, "f16", lens, 64, _perm(64, seed + 1), seed)


def llama13b(seed: int = 1002, B: int = 64) -> Workload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(128, 2049, size=B).astype(np.int32)
    N = _pool(lens + 1, 16)
    return Workload("llama13b", B, 40, 40, 128, 16, "f16", lens, N, _perm(N, seed + 1), seed,
                    layers=40)


def gqa7b(B: int, n: int, seed: int = 1003) -> Workload:
    lens = np.full(B, n, dtype=np.int32)
    N = _pool(lens + 1, 16)
    return Workload("gqa7b_b%d_n%d" % (B, n), B, 32, 8, 128, 16, "bf16", lens, N,
                    _perm(N, seed + 1), seed, layers=32)


def qwen_longtail(block_size: int = 16, seed: int = 1004, B: int = 128) -> Workload:
    rng = np.random.default_rng(seed)
    n_long = int(round(0.05 * B))
    lens = np.clip(np.rint(rng.lognormal(mean=math.log(1500.0), sigma=1.0, size=B)), 1,
                   8192).astype(np.int64)
    long_pos = rng.choice(B, size=n_long, replace=False)
    lens[long_pos] = rng.integers(16384, 24577, size=n_long)
    lens = lens.astype(np.int32)
    N = _pool(lens + 1, block_size)
    return Workload("qwen_longtail_bs%d" % block_size, B, 28, 4, 128, block_size, "bf16", lens,
                    N, _perm(N, seed + 1), seed, layers=28, extra={"long_pos": long_pos})


def prefix_share(seed: int = 1005, B: int = 256, prefix_len: int = 1024,
                 with_suffix: bool = True) -> Workload:
    rng = np.random.default_rng(seed)
    suffix = (rng.integers(64, 513, size=B) if with_suffix else np.zeros(B, dtype=np.int64))
    suffix = suffix.astype(np.int32)
    lens = (prefix_len + suffix).astype(np.int32)
    bs = 16
    prefix_blocks = (prefix_len + bs - 1) // bs
    own = sum((int(n) + bs - 1) // bs - prefix_len // bs for n in lens + 1)
    N = int(math.ceil(1.25 * (prefix_blocks + own)))
    name = "prefix_share" if with_suffix else "prefix_share_cow"
    return Workload(name, B, 28, 4, 128, bs, "bf16", lens, N, _perm(N, seed + 1), seed,
                    layers=28, prefix_len=prefix_len, suffix_lens=suffix)


def multiturn_trace(seed: int, convs: int, turns: int, system: int, user=(8, 60),
                    reply=(4, 40), vocab: int = 500, block_size: int = 16,
                    pool_factor: float = 2.5) -> dict:
    """A multi-turn serving trace (token ids only).

    ``turns`` is a list of turns; each holds ``prompts`` [(seq_id, tokens)],
    ``replies`` (decode steps, each a list of (seq_id, token) for the
    conversations still generating) and ``free`` (the previous turn's
    sequence ids).  ``history`` holds each conversation's final tokens,
    ``last`` its final sequence id; ``N`` and ``order`` size and order a pool.
    """
    rng = np.random.default_rng(seed)
    sys_p = rng.integers(0, vocab, system).tolist()
    hist = {c: list(sys_p) for c in range(convs)}
    sid, cur, out = 0, {}, []
    for _ in range(turns):
        prompts, old = [], dict(cur)
        for c in range(convs):
            hist[c] += rng.integers(0, vocab, int(rng.integers(user[0], user[1]))).tolist()
            prompts.append((sid, list(hist[c])))
            cur[c] = sid
            sid += 1
        lens = {c: int(rng.integers(reply[0], reply[1])) for c in range(convs)}
        replies = []
        for k in range(max(lens.values())):
            step = []
            for c in range(convs):
                if k < lens[c]:
                    tok = int(rng.integers(0, vocab))
                    hist[c].append(tok)
                    step.append((cur[c], tok))
            replies.append(step)
        out.append({"prompts": prompts, "replies": replies, "free": sorted(old.values())})
    need = sum(math.ceil(len(h) / block_size) for h in hist.values())
    N = int(need * pool_factor)
    return {"turns": out, "history": hist, "last": dict(cur), "N": N, "vocab": vocab,
            "order": np.random.default_rng(seed + 1).permutation(N).astype(np.int32)}


def multiturn_prefix(seed: int = 1006, convs: int = 128, turns: int = 4) -> Workload:
    """Decode batch at the end of a multi-turn trace: ``convs`` conversations,
    a 1024-token system prompt, user messages U[32, 256], replies U[64, 512],
    Qwen2.5-7B shape (28 / 4 heads of 128, bf16, block 16)."""
    bs = 16
    tr = multiturn_trace(seed, convs, turns, 1024, user=(32, 257), reply=(64, 513),
                         vocab=32000, block_size=bs)
    lens = np.array([len(tr["history"][c]) for c in range(convs)], dtype=np.int32)
    return Workload("multiturn_prefix", convs, 28, 4, 128, bs, "bf16", lens, tr["N"],
                    tr["order"], seed, layers=28, extra={"trace": tr})


def normal_tensor(shape, dtype, seed: int, chunk: int = 1 << 26) -> torch.Tensor:
    """N(0, 1) drawn in fp32 from a seeded CPU generator, cast to ``dtype``
    with round-to-nearest-even; drawn in chunks to bound host memory."""
    gen = torch.Generator().manual_seed(int(seed))
    total = int(np.prod(shape))
    out = torch.empty(total, dtype=dtype)
    for s in range(0, total, chunk):
        e = min(total, s + chunk)
        out[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32).to(dtype)
    return out.view(*shape)


def qkv(w: Workload, with_new: bool = True, with_cache: bool = True):
    """Seeded tensors on the host: ``q [B,H,d]``, with ``with_cache`` the
    ``k_cache``/``v_cache [N,bs,Hkv,d]`` and, with ``with_new``, one new
    token's ``k_new``/``v_new [B,Hkv,d]`` per sequence."""
    dt = w.torch_dtype
    out = {"q": normal_tensor((w.B, w.H, w.d), dt, w.seed * 16 + 1)}
    if with_cache:
        out["k_cache"] = normal_tensor((w.num_blocks, w.block_size, w.Hkv, w.d), dt,
                                       w.seed * 16 + 2)
        out["v_cache"] = normal_tensor((w.num_blocks, w.block_size, w.Hkv, w.d), dt,
                                       w.seed * 16 + 3)
    if with_new:
        out["k_new"] = normal_tensor((w.B, w.Hkv, w.d), dt, w.seed * 16 + 4)
        out["v_new"] = normal_tensor((w.B, w.Hkv, w.d), dt, w.seed * 16 + 5)
    return out


def fp8_cache(w: Workload, seed_offset: int = 0):
    """Seeded FP8 cache contents on the host, drawn directly (no quantisation):
    ``k_codes``/``v_codes [N,bs,Hkv,d]`` uint8 with the magnitude code uniform
    over the 127 finite E4M3 magnitudes (0x00..0x7E) and a random sign bit, and
    ``k_scale``/``v_scale [N,Hkv,bs]`` float32 uniform in [0.004, 0.012] (the
    size of amax / 448 for N(0, 1) rows of 128)."""
    rng = np.random.default_rng(w.seed * 16 + 6 + seed_offset)
    shape = (w.num_blocks, w.block_size, w.Hkv, w.d)
    out = {}
    for name in ("k", "v"):
        mag = rng.integers(0, 0x7F, size=shape, dtype=np.uint8)
        sign = rng.integers(0, 2, size=shape, dtype=np.uint8) << 7
        out[name + "_codes"] = torch.from_numpy(mag | sign)
        out[name + "_scale"] = torch.from_numpy(
            rng.uniform(0.004, 0.012, size=(w.num_blocks, w.Hkv, w.block_size)).astype(np.float32))
    return out


def int8_cache(w: Workload, seed_offset: int = 0):
    """Seeded INT8 cache contents on the host, drawn directly: codes
    ``[N,bs,Hkv,d]`` (int8 values uniform over -127..127, stored as uint8
    bytes) and ``k_scale``/``v_scale [N,Hkv,bs]`` float32 uniform in
    [0.014, 0.042] (the size of amax / 127 for N(0, 1) rows of 128)."""
    rng = np.random.default_rng(w.seed * 16 + 7 + seed_offset)
    shape = (w.num_blocks, w.block_size, w.Hkv, w.d)
    out = {}
    for name in ("k", "v"):
        codes = rng.integers(-127, 128, size=shape, dtype=np.int64).astype(np.int8)
        out[name + "_codes"] = torch.from_numpy(codes.view(np.uint8))
        out[name + "_scale"] = torch.from_numpy(
            rng.uniform(0.014, 0.042, size=(w.num_blocks, w.Hkv, w.block_size)).astype(np.float32))
    return out


def bits(t: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of an fp16 / bf16 host tensor (no copy)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
