"""Plain CPU oracle for paged KV-cache decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` import this package.  It shares no code
with the CUDA path (``paged_kv_cache_103_gb300``) and never imports it.

Sources, cited by page title and section:

* [P1] "LLM推理优化：vLLM PagedAttention深度解析与工程实践" (lpnh.cn/news/754185):
  section 二 (attention formula and the per-token KV-size formula),
  section 3.1 (block table), section 3.2 (BlockManager: free list, allocate,
  free), section 4.1 (paged K layout).
* [P2] "vLLM推理加速深度解析：从PagedAttention原理到生产部署实战"
  (kwkr.cn/news/169259): section 2.2 (workflow: each new token's K/V goes into
  the physical block the current logical block points to; a full block gets a
  new free block).
* [P3] "vLLM 深度拆解：当大模型推理学会「分页注意力」" (chenxutan.com/d/4834.html):
  section 2.1 (block table diagram), section 3.3 (BlockSpaceManager:
  append_slot, free, copy-on-write sharing).
* [P4] "LLM推理优化技术地图：从KV Cache到量化与投机解码" (qwbw.cn/news/280730):
  section 2.2 (KV size formula 2 x layers x kv_heads x head_dim x seq x batch x
  bytes), section 2.3 (GQA grouping).
* [P5] untitled Qwen2.5-7B deployment page (mhpq.cn/news/468822), section 1.2
  (57344 bytes of KV per token for 28 layers x 4 KV heads x 128 x 2 bytes).

Contents:

* :func:`decode` -- the fp64 attention over a block table (C, ``pa_oracle.c``).
* :func:`multi_query` -- several causal query tokens per sequence over the
  same table (chunked prefill / speculative verification, [P3] section 5).
* :func:`reshape_and_cache` -- the KV append: a plain per-token scatter.
* :func:`copy_blocks` -- the copy-on-write block copy: plain slice copies.
* :class:`BlockManagerModel` -- the allocator, restated from [P1] section 3.2
  and [P3] section 3.3.
* :func:`kv_bytes_per_token` / :func:`kv_cache_bytes` -- the closed forms.
* :func:`reshape_and_cache_fp8`, :func:`decode_fp8`, :func:`e4m3_encode` -- the
  FP8 KV cache (a reading, see the comment above :data:`E4M3_MAX`).
* :func:`reshape_and_cache_int8`, :func:`decode_int8`, :func:`int8_encode` -- the
  INT8 KV cache (a reading, see the comment above :data:`INT8_MAX`).
* ``BlockManagerModel.allocate_prompt`` / ``append_token`` -- automatic prefix
  caching of full blocks ([P5] section 3.2, [P1] section 4.2; a reading, see
  the class docstring).
* ``BlockManagerModel.swap_out`` / ``swap_in`` and :func:`swap_blocks` --
  moving a sequence's blocks to a host pool and back ([P1] section 3.2, [P2]
  section 4; a reading, see ``swap_out``).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from collections import deque

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libpa_oracle.so")

DTYPE_F16 = 0
DTYPE_BF16 = 1


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` with gcc into ``oracle/_build``.

    ``-ffp-contract=off`` keeps every multiply and add separately rounded, so
    x86 and Arm hosts produce the same fp64 values.
    """
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c99",
                               "-o", tmp, _SRC, "-lpthread", "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.pa_oracle_decode.restype = ctypes.c_int
        lib.pa_oracle_decode.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64, f64,
                                         i32, P, i32]
        lib.pa_oracle_weights.restype = ctypes.c_int
        lib.pa_oracle_weights.argtypes = [P, P, P, i32, P, i32, i32, i32, i32, i32, i64, f64, i32,
                                          i32, i32, P]
        lib.pa_oracle_to_double.restype = ctypes.c_int
        lib.pa_oracle_to_double.argtypes = [P, i64, i32, P]
        lib.pa_oracle_e4m3_to_double.restype = ctypes.c_int
        lib.pa_oracle_e4m3_to_double.argtypes = [P, i64, P]
        lib.pa_oracle_multi_query.restype = ctypes.c_int
        lib.pa_oracle_multi_query.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                              i64, f64, i32, P, i32]
        for name in ("pa_oracle_decode_fp8", "pa_oracle_decode_int8"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [P, i32, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i64, f64, P]
        _lib = lib
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("expected fp16/bf16 bit patterns as uint16, got %s" % a.dtype)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def multi_query(q, q_start, k_cache, v_cache, block_tables, context_lens, scale: float,
                dtype: int, num_threads: int = 1) -> np.ndarray:
    """fp64 attention of several query tokens per sequence over the paged cache
    (chunked prefill / speculative verification, [P3] section 5).  Sequence
    i's queries are rows ``q_start[i] .. q_start[i+1]-1`` of ``q [T, H, d]``
    (uint16) and are its LAST ``q_start[i+1] - q_start[i]`` cached tokens;
    query r attends causally to tokens ``0 .. context_lens[i] - qlen + r``
    (a reading: the pages give no formula).  Returns ``out[T, H, d]`` float64.
    """
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    qs = np.ascontiguousarray(q_start, dtype=np.int32)
    tbl = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    T, H, d = q.shape
    N, bs, Hkv, _ = k_cache.shape
    B = lens.shape[0]
    if qs.shape[0] != B + 1 or qs[-1] != T:
        raise ValueError("q_start must have B + 1 entries ending at T")
    out = np.zeros((T, H, d), dtype=np.float64)
    rc = _load().pa_oracle_multi_query(_ptr(q), _ptr(qs), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(tbl), tbl.shape[1], _ptr(lens), B, H, Hkv, d, bs, N,
                                       float(scale), int(dtype), _ptr(out), int(num_threads))
    if rc:
        raise ValueError("pa_oracle_multi_query failed (%d)" % rc)
    return out


def to_double(bits, dtype: int) -> np.ndarray:
    """Exact fp64 values of fp16 (dtype 0) or bf16 (dtype 1) bit patterns."""
    x = _u16(bits)
    y = np.empty(x.shape, dtype=np.float64)
    rc = _load().pa_oracle_to_double(_ptr(x), x.size, dtype, _ptr(y))
    if rc:
        raise ValueError("pa_oracle_to_double failed (%d)" % rc)
    return y


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, dtype: int,
           num_threads: int = 1) -> np.ndarray:
    """fp64 paged decode attention; returns ``out[B, H, d]`` as float64.

    ``q``: uint16 ``[B, H, d]``; caches: uint16 ``[N, bs, Hkv, d]``;
    ``block_tables``: int32 ``[B, max_blocks]``; ``context_lens``: int32 ``[B]``.
    Follows [P1] section 二 for the arithmetic, section 3.1 / 4.1 for the table
    walk and [P4] section 2.3 for the head grouping (see ``pa_oracle.c``).
    """
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    tbl = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, H, d = q.shape
    N, bs, Hkv, d2 = k_cache.shape
    if d2 != d or v_cache.shape != k_cache.shape or lens.shape != (B,) or tbl.shape[0] != B:
        raise ValueError("shape mismatch")
    out = np.empty((B, H, d), dtype=np.float64)
    rc = _load().pa_oracle_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(tbl), tbl.shape[1],
                                  _ptr(lens), B, H, Hkv, d, bs, N, float(scale), dtype, _ptr(out),
                                  int(num_threads))
    if rc:
        raise ValueError("pa_oracle_decode failed (%d)" % rc)
    return out


def weights(q, k_cache, block_tables, context_lens, scale: float, dtype: int, i: int,
            h: int) -> np.ndarray:
    """The softmax weights of one (sequence, query head), fp64."""
    q, k_cache = _u16(q), _u16(k_cache)
    tbl = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, H, d = q.shape
    N, bs, Hkv, _ = k_cache.shape
    w = np.empty(max(int(lens[i]), 1), dtype=np.float64)
    rc = _load().pa_oracle_weights(_ptr(q), _ptr(k_cache), _ptr(tbl), tbl.shape[1], _ptr(lens), B,
                                   H, Hkv, d, bs, N, float(scale), dtype, i, h, _ptr(w))
    if rc:
        raise ValueError("pa_oracle_weights failed (%d)" % rc)
    return w[: int(lens[i])]


# ----------------------------------------------------------------- FP8 KV cache
# Reading (the pages only say that quantising the KV cache to 8 bits halves its
# bytes, "LLM推理优化技术地图：从KV Cache到量化与投机解码" section 4.3): codes are OCP
# FP8 E4M3 (bias 7, no infinities, NaN at S.1111.111, largest finite 448); each
# (token, KV head) row of head_dim values gets its own fp32 scale
# s = fl32(amax / 448), amax = max |x| over the row (exact in fp32), and code
# = RNE-saturating E4M3 of fl32(x / s) (fp32 division); an all-zero row gets
# s = 0 and zero codes.  Scales are laid out [num_blocks][Hkv][block_size].
E4M3_MAX = 448.0


def e4m3_to_double(codes) -> np.ndarray:
    """Exact values of E4M3 codes (uint8)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    y = np.empty(c.shape, dtype=np.float64)
    _load().pa_oracle_e4m3_to_double(_ptr(c), c.size, _ptr(y))
    return y


_E4M3_POS = None


def _e4m3_positive_table():
    global _E4M3_POS
    if _E4M3_POS is None:
        codes = np.arange(0x7F, dtype=np.uint8)          # 0x00 .. 0x7E: all finite >= 0
        _E4M3_POS = e4m3_to_double(codes)
    return _E4M3_POS


def e4m3_encode(x) -> np.ndarray:
    """Round fp32 values to the nearest E4M3 code, ties to the even code,
    saturating at +-448 (NaN maps to 0x7F with its sign)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    vals = _e4m3_positive_table()                         # ascending, 127 entries
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, len(vals) - 1)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((hi & 1) == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == vals[hi], hi, code).astype(np.uint8)
    code = code | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    code = np.where(np.isnan(x), (0x7F | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8), code)
    return code.astype(np.uint8)


def quantize_rows(x_fp32):
    """Quantise rows (last axis) of fp32 values: returns (codes uint8, scales fp32)."""
    x = np.asarray(x_fp32, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1).astype(np.float32)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(s == 0, np.float32(1), s).astype(np.float32)
    codes = e4m3_encode((x / safe[..., None]).astype(np.float32))
    codes = np.where((s == 0)[..., None], 0, codes).astype(np.uint8)
    return codes, s


def reshape_and_cache_fp8(k_new, v_new, slot_mapping, k_codes, v_codes, k_scale, v_scale):
    """The FP8 KV append: token t's K/V rows [Hkv, d] (fp16/bf16 host tensors)
    are quantised per KV head and written to slot s (codes at
    [s // bs, s % bs, h, :], scale at [s // bs, h, s % bs]); negative slots skip."""
    bs = k_codes.shape[1]
    kq, ks = quantize_rows(k_new.float().numpy())
    vq, vs = quantize_rows(v_new.float().numpy())
    for t in range(k_new.shape[0]):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        k_codes[s // bs, s % bs] = kq[t]
        v_codes[s // bs, s % bs] = vq[t]
        k_scale[s // bs, :, s % bs] = ks[t]
        v_scale[s // bs, :, s % bs] = vs[t]


def decode_fp8(q, q_dtype: int, k_codes, v_codes, k_scale, v_scale, block_tables,
               context_lens, scale: float, _fn="pa_oracle_decode_fp8") -> np.ndarray:
    """fp64 paged decode over an FP8 cache: the attention of :func:`decode` on
    the dequantised rows code_value * scale."""
    q = _u16(q)
    kc = np.ascontiguousarray(k_codes, dtype=np.uint8)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    tbl = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, H, d = q.shape
    N, bs, Hkv, _ = kc.shape
    out = np.empty((B, H, d), dtype=np.float64)
    rc = getattr(_load(), _fn)(_ptr(q), q_dtype, _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs),
                               _ptr(tbl), tbl.shape[1], _ptr(lens), B, H, Hkv, d, bs, N,
                               float(scale), _ptr(out))
    if rc:
        raise ValueError("%s failed (%d)" % (_fn, rc))
    return out


# INT8 KV cache ("LLM推理优化技术地图：从KV Cache到量化与投机解码", section 4.3: 8-bit
# KV quantisation; the pages fix no format).  Reading: symmetric, one fp32
# scale per (token, KV head) row, s = fl32(amax / 127); code = the integer
# nearest fl32(x / s) (fp32 division, ties to even), clamped to [-127, 127];
# an all-zero row gets s = 0 and zero codes.  Element = code * s.  Same
# layouts as the FP8 cache; codes are stored as their two's-complement bytes.
INT8_MAX = 127.0


def int8_encode(x) -> np.ndarray:
    """fp32 values to INT8 codes (uint8 bytes of int8): nearest integer, ties
    to even, clamped to [-127, 127]."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    c = np.clip(np.rint(x), -INT8_MAX, INT8_MAX)
    return c.astype(np.int64).astype(np.int8).view(np.uint8)


def quantize_rows_int8(x_fp32):
    """Quantise rows (last axis) of fp32 values to INT8: (codes uint8, scales fp32)."""
    x = np.asarray(x_fp32, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1).astype(np.float32)
    s = (amax / np.float32(INT8_MAX)).astype(np.float32)
    safe = np.where(s == 0, np.float32(1), s).astype(np.float32)
    codes = int8_encode((x / safe[..., None]).astype(np.float32))
    codes = np.where((s == 0)[..., None], 0, codes).astype(np.uint8)
    return codes, s


def reshape_and_cache_int8(k_new, v_new, slot_mapping, k_codes, v_codes, k_scale, v_scale):
    """The INT8 KV append: as :func:`reshape_and_cache_fp8` with INT8 codes."""
    bs = k_codes.shape[1]
    kq, ks = quantize_rows_int8(k_new.float().numpy())
    vq, vs = quantize_rows_int8(v_new.float().numpy())
    for t in range(k_new.shape[0]):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        k_codes[s // bs, s % bs] = kq[t]
        v_codes[s // bs, s % bs] = vq[t]
        k_scale[s // bs, :, s % bs] = ks[t]
        v_scale[s // bs, :, s % bs] = vs[t]


def decode_int8(q, q_dtype: int, k_codes, v_codes, k_scale, v_scale, block_tables,
                context_lens, scale: float) -> np.ndarray:
    """fp64 paged decode over an INT8 cache (rows code * scale)."""
    return decode_fp8(q, q_dtype, k_codes, v_codes, k_scale, v_scale, block_tables,
                      context_lens, scale, _fn="pa_oracle_decode_int8")


def swap_blocks(src_pools, dst_pools, pairs) -> None:
    """The swap copies: for every pool pair (a layer's K or V, on the device
    and in host memory) and every pair ``(s, d)``, block ``d`` of the
    destination becomes a copy of block ``s`` of the source."""
    for src, dst in zip(src_pools, dst_pools):
        for s, d in pairs:
            dst[int(d)] = src[int(s)]


def reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache) -> None:
    """The KV append, in place: token t goes to ``cache[s // bs, s % bs]``.

    [P2] section 2.2: each generated token's K/V is stored into the physical
    block the current logical block points to.  The slot of a token is
    ``physical_block * block_size + offset`` (a reading: the pages give no
    formula).  A negative slot marks padding and is skipped.
    """
    bs = k_cache.shape[1]
    for t in range(k_new.shape[0]):
        s = int(slot_mapping[t])
        if s < 0:
            continue
        k_cache[s // bs, s % bs] = k_new[t]
        v_cache[s // bs, s % bs] = v_new[t]


def copy_blocks(k_caches, v_caches, pairs) -> None:
    """Copy-on-write block copies, in place, for every layer's cache.

    [P3] section 3.3: a shared block is copied only when a sharer must write
    into it.  ``pairs`` is a sequence of (src, dst) physical block ids.
    """
    for kc, vc in zip(k_caches, v_caches):
        for src, dst in pairs:
            kc[int(dst)] = kc[int(src)]
            vc[int(dst)] = vc[int(src)]


def kv_bytes_per_token(num_layers: int, kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    """[P4] section 2.2 / [P5] section 1.2: 2 (K and V) x layers x KV heads x
    head dim x element bytes.  For MHA, kv_heads x head_dim is d_model ([P1]
    section 二)."""
    return 2 * num_layers * kv_heads * head_dim * dtype_bytes


def kv_cache_bytes(num_layers: int, kv_heads: int, head_dim: int, seq_len: int, batch: int,
                   dtype_bytes: int) -> int:
    """[P4] section 2.2: the per-token size times sequence length times batch."""
    return kv_bytes_per_token(num_layers, kv_heads, head_dim, dtype_bytes) * seq_len * batch


class OracleOOM(Exception):
    """Raised when the free list cannot cover a request ([P1] section 3.2)."""


class OracleInvalid(Exception):
    """Raised for an operation on an unknown / duplicate sequence."""


class BlockManagerModel:
    """The block allocator, restated from the pages.

    [P1] section 3.2: the free list starts as the block ids in order, a block is
    taken from the FRONT of the free list and a freed block is put at the BACK,
    in the order of the sequence's table; ``allocate(seq, num_tokens)`` gives a
    sequence enough blocks to hold ``num_tokens`` tokens, checking the free
    list before taking anything (all or nothing).  [P3] section 3.3:
    ``append_slot`` writes into the current last block if it has room, else
    takes a new block; sharing is by reference, and a shared block is copied
    only when a sharer writes into it (copy-on-write).

    Readings where the pages are silent: ``init_free_order`` replaces the
    initial ``0..N-1`` order (random placement is a permutation); a shared
    block carries a reference count and returns to the free list when it
    drops to zero; ``fork`` copies the parent's table and raises the counts;
    a sequence that writes into a shared, partially filled last block takes a
    new block from the front of the free list, the pair (old, new) is reported
    for a copy and the old block's count drops by one -- the last sharer left
    writes in place.

    Automatic prefix caching ([P5] section 3.2: a prompt is cut into blocks of
    block_size tokens, each block's KV is cached under a hash of its token ids,
    and a new request reuses the cached blocks of a prefix that matches token
    for token and is aligned to block boundaries -- a change in the first block
    invalidates every later one; [P1] section 4.2: the reuse spans requests,
    e.g. turns of a conversation).  Reading: a FULL block's key is (the id of
    the cache entry holding the previous block's content, or 0 for the first
    block, the block's token ids), so a key names its whole prefix; entry ids
    are never reused.  ``allocate_prompt`` walks the prompt's full blocks and
    reuses each block found (reference +1; a block found on the free list is
    taken off it) until the first miss, then allocates the rest from the front
    of the free list and registers every new full block.  ``append_token``
    appends like ``append_slot`` and registers the sequence's block when it
    becomes full (if its key is already cached, the sequence's chain continues
    from that entry and its own block stays unregistered).  A freed block keeps
    its entry while it waits on the free list; a block taken from the front of
    the free list loses its entry (eviction, oldest freed first).  Sequences
    created or grown without token ids (``allocate``, ``append_slot``,
    ``append_batch``) are not tracked and register nothing.
    """

    def __init__(self, num_blocks: int, block_size: int, init_free_order=None):
        if num_blocks < 0 or block_size <= 0:
            raise OracleInvalid("bad pool")
        order = list(range(num_blocks)) if init_free_order is None else [int(b) for b in init_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise OracleInvalid("init_free_order must be a permutation of 0..N-1")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free_blocks = deque(order)
        self.allocated: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self.ref = [0] * num_blocks
        # prefix cache
        self.cache: dict[tuple, tuple[int, int]] = {}   # key -> (entry id, block)
        self.block_key: dict[int, tuple] = {}           # block -> key of its entry
        self.next_entry = 1
        self.tracked: dict[int, bool] = {}
        self.pending: dict[int, list[int]] = {}         # token ids of the partial last block
        self.chain: dict[int, int] = {}                 # entry id of the last full block's content
        self.pstats = {"lookups": 0, "hits": 0, "registered": 0, "evicted": 0}
        # swap space
        self.host_free: deque[int] = deque()
        self.host_blocks = 0
        self.swapped: dict[int, list[int]] = {}          # seq -> host blocks in table order

    def _take_front(self) -> int:
        b = self.free_blocks.popleft()
        key = self.block_key.pop(b, None)
        if key is not None:
            del self.cache[key]
            self.pstats["evicted"] += 1
        self.ref[b] = 1
        return b

    def _untrack(self, seq_id: int) -> None:
        self.tracked[seq_id] = False
        self.pending[seq_id] = []

    # -- [P1] section 3.2 -------------------------------------------------
    def allocate(self, seq_id: int, num_tokens: int) -> None:
        if num_tokens < 0 or seq_id in self.swapped:
            raise OracleInvalid("negative token count or swapped sequence")
        table = self.allocated.get(seq_id, [])
        cur_len = self.lens.get(seq_id, 0)
        already_used = len(table) * self.block_size
        if (num_tokens > cur_len and cur_len % self.block_size != 0 and table
                and self.ref[table[-1]] > 1):
            raise OracleInvalid("growing into a shared partial block needs append_slot")
        if already_used < num_tokens:
            need = math.ceil((num_tokens - already_used) / self.block_size)
            if len(self.free_blocks) < need:
                raise OracleOOM("need %d blocks, %d free" % (need, len(self.free_blocks)))
            for _ in range(need):
                table.append(self._take_front())
        self.allocated[seq_id] = table
        if num_tokens > cur_len or seq_id not in self.tracked:
            self._untrack(seq_id)
            self.chain.setdefault(seq_id, 0)
        self.lens[seq_id] = max(cur_len, num_tokens)

    def free(self, seq_id: int) -> None:
        if seq_id not in self.allocated:
            raise OracleInvalid("unknown sequence")
        for h in self.swapped.pop(seq_id, []):
            self.host_free.append(h)
        for b in self.allocated[seq_id]:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free_blocks.append(b)
        del self.allocated[seq_id]
        del self.lens[seq_id]
        del self.tracked[seq_id], self.pending[seq_id], self.chain[seq_id]

    # -- [P3] section 3.3 -------------------------------------------------
    def _blocks_needed_for_append(self, seq_id: int, ref_view) -> int:
        pos = self.lens[seq_id]
        table = self.allocated[seq_id]
        if pos == len(table) * self.block_size:
            return 1
        return 1 if ref_view(table[pos // self.block_size]) > 1 else 0

    def append_slot(self, seq_id: int):
        """Reserve the slot of the sequence's next token.

        Returns ``(slot, cow)`` where ``cow`` is ``None`` or ``(src, dst)``.
        """
        if seq_id not in self.allocated or seq_id in self.swapped:
            raise OracleInvalid("unknown or swapped sequence")
        if self._blocks_needed_for_append(seq_id, lambda b: self.ref[b]) > len(self.free_blocks):
            raise OracleOOM("no free block")
        self._untrack(seq_id)
        return self._append_unchecked(seq_id)

    def _append_unchecked(self, seq_id: int):
        bs = self.block_size
        table = self.allocated[seq_id]
        pos = self.lens[seq_id]
        cow = None
        if pos == len(table) * bs:
            table.append(self._take_front())
        else:
            last = table[pos // bs]
            if self.ref[last] > 1:
                new = self._take_front()
                self.ref[last] -= 1
                table[pos // bs] = new
                cow = (last, new)
        self.lens[seq_id] = pos + 1
        slot = table[pos // bs] * bs + pos % bs
        return slot, cow

    def append_batch(self, seq_ids, tokens=None):
        """One new token for each sequence of a decode batch, all or nothing.

        Sequences are served in the given order (so with k sharers of one
        partial block in the batch, the first k-1 copy it and the last writes
        in place).  Returns ``(slots, cow_pairs)``.  With ``tokens`` (one token
        id per sequence) each append is an :meth:`append_token`.
        """
        seq_ids = [int(s) for s in seq_ids]
        if tokens is not None and len(tokens) != len(seq_ids):
            raise OracleInvalid("one token per sequence")
        if len(set(seq_ids)) != len(seq_ids):
            raise OracleInvalid("duplicate sequence in batch")
        for s in seq_ids:
            if s not in self.allocated or s in self.swapped:
                raise OracleInvalid("unknown or swapped sequence")
        # count the blocks the whole batch takes, with the counts it changes
        delta: dict[int, int] = {}
        need = 0
        for s in seq_ids:
            n = self._blocks_needed_for_append(s, lambda b: self.ref[b] + delta.get(b, 0))
            pos = self.lens[s]
            table = self.allocated[s]
            if n and pos != len(table) * self.block_size:
                last = table[pos // self.block_size]
                delta[last] = delta.get(last, 0) - 1
            need += n
        if need > len(self.free_blocks):
            raise OracleOOM("batch needs %d blocks, %d free" % (need, len(self.free_blocks)))
        slots, pairs = [], []
        for r, s in enumerate(seq_ids):
            if tokens is None:
                self._untrack(s)
                slot, cow = self._append_unchecked(s)
            else:
                slot, cow = self._append_token_unchecked(s, int(tokens[r]))
            slots.append(slot)
            if cow is not None:
                pairs.append(cow)
        return slots, pairs

    # -- automatic prefix caching ([P5] section 3.2, [P1] section 4.2) ---------
    def allocate_prompt(self, seq_id: int, tokens) -> int:
        """Creates ``seq_id`` holding the prompt ``tokens``; returns how many of
        its tokens were found in the cache (a multiple of block_size)."""
        tokens = [int(t) for t in tokens]
        if seq_id in self.allocated:
            raise OracleInvalid("sequence exists")
        bs = self.block_size
        n = len(tokens)
        full = n // bs
        chain, hits = 0, []
        for i in range(full):          # the walk stops at the first miss
            self.pstats["lookups"] += 1
            key = (chain, tuple(tokens[i * bs:(i + 1) * bs]))
            found = self.cache.get(key)
            if found is None:
                break
            chain = found[0]
            hits.append(found[1])
        revive = sum(1 for b in hits if self.ref[b] == 0)
        need = math.ceil(n / bs) - len(hits)
        if need > len(self.free_blocks) - revive:
            self.pstats["lookups"] -= min(full, len(hits) + 1)
            raise OracleOOM("need %d blocks, %d free" % (need, len(self.free_blocks) - revive))
        self.pstats["hits"] += len(hits)
        table = []
        for b in hits:
            if self.ref[b] == 0:
                self.free_blocks.remove(b)
            self.ref[b] += 1
            table.append(b)
        for i in range(len(hits), math.ceil(n / bs)):
            b = self._take_front()
            table.append(b)
            if i < full:
                chain = self._register(chain, tokens[i * bs:(i + 1) * bs], b)
        self.allocated[seq_id] = table
        self.lens[seq_id] = n
        self.tracked[seq_id] = True
        self.pending[seq_id] = tokens[full * bs:]
        self.chain[seq_id] = chain
        return len(hits) * bs

    def _register(self, chain: int, block_tokens, block: int) -> int:
        key = (chain, tuple(block_tokens))
        found = self.cache.get(key)
        if found is not None:
            return found[0]
        eid = self.next_entry
        self.next_entry += 1
        self.cache[key] = (eid, block)
        self.block_key[block] = key
        self.pstats["registered"] += 1
        return eid

    def append_token(self, seq_id: int, token: int):
        """:meth:`append_slot` that also records the token id; returns
        ``(slot, cow)``."""
        if seq_id not in self.allocated or seq_id in self.swapped:
            raise OracleInvalid("unknown or swapped sequence")
        if self._blocks_needed_for_append(seq_id, lambda b: self.ref[b]) > len(self.free_blocks):
            raise OracleOOM("no free block")
        return self._append_token_unchecked(seq_id, int(token))

    def _append_token_unchecked(self, seq_id: int, token: int):
        slot, cow = self._append_unchecked(seq_id)
        if self.tracked[seq_id]:
            pend = self.pending[seq_id]
            pend.append(token)
            if len(pend) == self.block_size:
                pos = self.lens[seq_id] - 1
                block = self.allocated[seq_id][pos // self.block_size]
                self.chain[seq_id] = self._register(self.chain[seq_id], pend, block)
                self.pending[seq_id] = []
        return slot, cow

    # -- swapping ([P1] section 3.2, [P2] section 4) -------------------------
    def set_swap_pool(self, num_host_blocks: int) -> None:
        if self.host_blocks or num_host_blocks < 0:
            raise OracleInvalid("swap pool already set")
        self.host_blocks = num_host_blocks
        self.host_free = deque(range(num_host_blocks))

    def swap_out(self, seq_id: int):
        """Moves a sequence out of device memory ([P1] section 3.2: allocation
        that finds too few free blocks needs swap or preemption; [P2] section
        4: with swap space the KV cache goes to CPU memory).  Reading: the unit
        is one sequence; every block of its table, in order, gets a host block
        from the front of the host free list (all or nothing); each device
        block's count drops by one and blocks reaching zero go to the back of
        the device free list.  Returns the copies ``[(device, host)]`` to make
        before the device blocks are reused."""
        if seq_id not in self.allocated or seq_id in self.swapped:
            raise OracleInvalid("unknown or swapped sequence")
        table = self.allocated[seq_id]
        if len(table) > len(self.host_free):
            raise OracleOOM("swap space full")
        hosts = [self.host_free.popleft() for _ in table]
        for b in table:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free_blocks.append(b)
        self.swapped[seq_id] = hosts
        self.allocated[seq_id] = []
        return list(zip(table, hosts))

    def swap_in(self, seq_id: int):
        """Brings a swapped sequence back: one block from the front of the
        device free list per host block (all or nothing), host blocks return
        to the back of the host free list in table order.  Returns the copies
        ``[(host, device)]``; the sequence's blocks are private afterwards."""
        if seq_id not in self.swapped:
            raise OracleInvalid("sequence is not swapped out")
        hosts = self.swapped[seq_id]
        if len(hosts) > len(self.free_blocks):
            raise OracleOOM("no device blocks to swap in")
        table = [self._take_front() for _ in hosts]
        for h in hosts:
            self.host_free.append(h)
        del self.swapped[seq_id]
        self.allocated[seq_id] = table
        return list(zip(hosts, table))

    def prefix_stats(self) -> dict:
        d = dict(self.pstats)
        d["entries"] = len(self.cache)
        d["cached_free"] = sum(1 for b in self.free_blocks if b in self.block_key)
        return d

    def fork(self, parent: int, child: int) -> None:
        """[P4] section 3.3 / [P3] section 3.3: the child shares the parent's
        blocks; only the table is copied."""
        if parent not in self.allocated or child in self.allocated or parent in self.swapped:
            raise OracleInvalid("bad fork")
        table = list(self.allocated[parent])
        for b in table:
            self.ref[b] += 1
        self.allocated[child] = table
        self.lens[child] = self.lens[parent]
        self.tracked[child] = self.tracked[parent]
        self.pending[child] = list(self.pending[parent])
        self.chain[child] = self.chain[parent]

    # -- exports ------------------------------------------------------------
    def slot_of(self, seq_id: int, pos: int) -> int:
        table = self.allocated[seq_id]
        return table[pos // self.block_size] * self.block_size + pos % self.block_size

    def export(self, seq_ids, max_blocks: int | None = None):
        """``(block_tables [B, max_blocks] int32 padded with -1, context_lens [B] int32)``."""
        seq_ids = [int(s) for s in seq_ids]
        if max_blocks is None:
            max_blocks = max([len(self.allocated[s]) for s in seq_ids] + [1])
        tbl = np.full((len(seq_ids), max_blocks), -1, dtype=np.int32)
        lens = np.zeros(len(seq_ids), dtype=np.int32)
        for r, s in enumerate(seq_ids):
            if s in self.swapped:
                raise OracleInvalid("swapped sequence")
            t = self.allocated[s]
            if len(t) > max_blocks:
                raise OracleInvalid("table wider than max_blocks")
            tbl[r, : len(t)] = t
            lens[r] = self.lens[s]
        return tbl, lens

    def stats(self) -> dict:
        used = sum(1 for r in self.ref if r > 0)
        shared = sum(1 for r in self.ref if r > 1)
        return {"num_blocks": self.num_blocks, "free_blocks": len(self.free_blocks),
                "used_blocks": used, "shared_blocks": shared, "num_seqs": len(self.allocated),
                "num_tokens": sum(self.lens.values())}
