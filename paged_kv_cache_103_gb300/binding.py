"""ctypes binding of ``libpa.so`` (``include/pa.h``), with the C names.

Argument marshalling only: tensors become raw pointers and sizes, statuses
become :class:`PaError`.  Every step runs inside the library.  The library
must have been built (``paged_kv_cache_103_gb300.build.build()``); loading
fails loudly if it is missing -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

PA_OK = 0
PA_F16, PA_BF16 = 0, 1
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_INVALID", 2: "PA_ERR_OOM", 3: "PA_ERR_NOT_FOUND",
                4: "PA_ERR_BOUNDS", 5: "PA_ERR_CUDA", 6: "PA_ERR_UNSUPPORTED",
                7: "PA_ERR_TIMEOUT"}
DEVERR = {"BLOCK_ID": 0x1, "TABLE_WIDTH": 0x2, "SLOT": 0x4, "TIMEOUT": 0x8, "PAIR": 0x10,
          "CONTEXT": 0x20}

# Every symbol pa.h declares, with (restype, argtypes).
_P, _I32, _I64, _SZ, _F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_ST = ctypes.c_int


class AllocStats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("free_blocks", ctypes.c_int32), ("used_blocks", ctypes.c_int32),
                ("shared_blocks", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("num_tokens", ctypes.c_int64)]


class SwapStats(ctypes.Structure):
    _fields_ = [("host_blocks", ctypes.c_int32), ("host_free", ctypes.c_int32),
                ("swapped_seqs", ctypes.c_int32)]


class StepDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("max_context_len", ctypes.c_int32), ("dtype", ctypes.c_int),
                ("scale", ctypes.c_float), ("q8", ctypes.c_int32), ("depth", ctypes.c_int32)]


class StepLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("q", "k_new", "v_new", "slot_mapping",
                                                "block_tables", "context_lens", "in_bytes",
                                                "cow_pairs", "out", "total")]


class PrefixStats(ctypes.Structure):
    _fields_ = [("lookups", ctypes.c_int64), ("hits", ctypes.c_int64),
                ("registered", ctypes.c_int64), ("evicted", ctypes.c_int64),
                ("entries", ctypes.c_int64), ("cached_free", ctypes.c_int64)]


SIGNATURES = {
    "pa_status_str": (ctypes.c_char_p, [_ST]),
    "pa_version": (_I32, []),
    "pa_alloc_create": (_ST, [_I32, _I32, _P, ctypes.POINTER(_P)]),
    "pa_alloc_destroy": (None, [_P]),
    "pa_alloc": (_ST, [_P, _I64, _I32]),
    "pa_append_slot": (_ST, [_P, _I64, _P, _P, _P]),
    "pa_append_batch": (_ST, [_P, _P, _I32, _P, _P, _P]),
    "pa_fork": (_ST, [_P, _I64, _I64]),
    "pa_free": (_ST, [_P, _I64]),
    "pa_export": (_ST, [_P, _P, _I32, _I32, _P, _P]),
    "pa_seq_slots": (_ST, [_P, _I64, _I32, _I32, _P]),
    "pa_seq_info": (_ST, [_P, _I64, _P, _P]),
    "pa_block_ref": (_ST, [_P, _I32, _P]),
    "pa_free_list": (_ST, [_P, _P, _I32, _P]),
    "pa_alloc_stats_get": (_ST, [_P, ctypes.POINTER(AllocStats)]),
    "pa_alloc_prompt": (_ST, [_P, _I64, _P, _I32, _P]),
    "pa_append_token": (_ST, [_P, _I64, _I32, _P, _P, _P]),
    "pa_append_batch_tokens": (_ST, [_P, _P, _P, _I32, _P, _P, _P]),
    "pa_prefix_stats_get": (_ST, [_P, ctypes.POINTER(PrefixStats)]),
    "pa_alloc_set_swap_pool": (_ST, [_P, _I32]),
    "pa_swap_out": (_ST, [_P, _I64, _P, _I32, _P]),
    "pa_swap_in": (_ST, [_P, _I64, _P, _I32, _P]),
    "pa_swap_stats_get": (_ST, [_P, ctypes.POINTER(SwapStats)]),
    "pa_host_free_list": (_ST, [_P, _P, _I32, _P]),
    "pa_swap_blocks": (_ST, [_P, _P, _I32, _P, _I32, _I64, _I32, _I32, _P]),
    "pa_reshape_and_cache": (_ST, [_P, _P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _ST, _P]),
    "pa_reshape_and_cache_fp8": (_ST, [_P, _P, _P, _I32, _P, _P, _P, _P, _I32, _I32, _I32, _I32,
                                       _ST, _P]),
    "pa_copy_blocks": (_ST, [_P, _P, _I32, _P, _I32, _I64, _I32, _P]),
    "pa_decode_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "pa_decode_workspace_init": (_ST, [_P, _SZ, _P]),
    "pa_decode": (_ST, [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                        _F32, _ST, _P, _P, _SZ, _P]),
    "pa_multi_query_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32]),
    "pa_multi_query": (_ST, [_P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                             _I32, ctypes.c_float, _ST, _P, _P, _SZ, _P]),
    "pa_multi_query_tc_workspace_size": (_SZ, [_I32, _I32, _I32, _I32]),
    "pa_multi_query_tc": (_ST, [_P, _P, _I32, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32,
                                _I32, _I32, ctypes.c_float, _ST, _P, _P, _SZ, _P]),
    "pa_decode_fp8": (_ST, [_P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                            _I32, ctypes.c_float, _ST, _P, _P, _SZ, _P]),
    "pa_reshape_and_cache_int8": (_ST, [_P, _P, _P, _I32, _P, _P, _P, _P, _I32, _I32, _I32, _I32,
                                        _ST, _P]),
    "pa_decode_int8": (_ST, [_P, _P, _P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                             _I32, ctypes.c_float, _ST, _P, _P, _SZ, _P]),
    "pa_decode_noalloc": (_ST, [_P, _P, _P, _P, _I32, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                                _I32, _F32, _ST, _P, _P]),
    "pa_step_layout_get": (_ST, [ctypes.POINTER(StepDesc), ctypes.POINTER(StepLayout)]),
    "pa_step_create": (_ST, [ctypes.POINTER(StepDesc), _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                             ctypes.POINTER(_P)]),
    "pa_step_submit": (_ST, [_P, _P, _P, _P]),
    "pa_step_wait": (_ST, [_P, _I32]),
    "pa_step_run": (_ST, [_P, _P, _P]),
    "pa_step_destroy": (None, [_P]),
    "pa_check_device_errors": (_ST, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "pa_decode_grid_size": (_I32, []),
    "pa_selftest_wait_timeout": (_ST, [ctypes.c_uint32, _P]),
    "pa_measure_mma_ceiling": (_ST, [_I32, _I32, _P, _SZ, ctypes.POINTER(_I64), _P]),
}


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (%s)" % (what, STATUS_NAMES.get(status, status),
                                          _lib_status_str(status)))


_lib = None


def _lib_status_str(status: int) -> str:
    if _lib is None:
        return "?"
    s = _lib.pa_status_str(status)
    return s.decode() if s else "?"


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Loads libpa.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError("libpa.so is not built (%s); run __graft_entry__.build() or "
                               "python -m paged_kv_cache_103_gb300.build" % path)
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PaError(status, what)


def _stream_ptr(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError("fp16 or bf16 expected, got %s" % t.dtype)


def _dev(t, dtype=None):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("contiguous CUDA tensor expected")
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s expected, got %s" % (dtype, t.dtype))
    return t.data_ptr()


# --------------------------------------------------------------------------- device ops
def pa_reshape_and_cache(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None) -> None:
    """``k_new/v_new [T, Hkv, d]``, ``slot_mapping [T] int64``, caches ``[N, bs, Hkv, d]``."""
    import torch
    T, Hkv, d = k_new.shape
    N, bs = k_cache.shape[0], k_cache.shape[1]
    _check(load().pa_reshape_and_cache(_dev(k_new), _dev(v_new), _dev(slot_mapping, torch.int64),
                                       T, _dev(k_cache), _dev(v_cache), N, bs, Hkv, d,
                                       _dtype_code(k_cache), _stream_ptr(stream)),
           "pa_reshape_and_cache")


def pa_reshape_and_cache_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                             stream=None, _name="pa_reshape_and_cache_fp8") -> None:
    """Quantising append: ``k_new/v_new [T, Hkv, 128]`` fp16/bf16, caches
    ``[N, bs, Hkv, 128]`` uint8 (E4M3 codes), scales ``[N, Hkv, bs]`` float32."""
    import torch
    T, Hkv, d = k_new.shape
    N, bs = k_cache.shape[0], k_cache.shape[1]
    _check(getattr(load(), _name)(
        _dev(k_new), _dev(v_new), _dev(slot_mapping, torch.int64), T, _dev(k_cache, torch.uint8),
        _dev(v_cache, torch.uint8), _dev(k_scale, torch.float32), _dev(v_scale, torch.float32),
        N, bs, Hkv, d, _dtype_code(k_new), _stream_ptr(stream)), _name)


def pa_reshape_and_cache_int8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                              stream=None) -> None:
    """``pa_reshape_and_cache_fp8`` with INT8 codes (the int8 bytes in uint8 tensors)."""
    pa_reshape_and_cache_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                             stream, _name="pa_reshape_and_cache_int8")


def pa_copy_blocks(k_caches, v_caches, pairs, stream=None) -> None:
    """Copies block ``pairs[p][0]`` onto ``pairs[p][1]`` in every layer's caches."""
    import torch
    L = len(k_caches)
    P = int(pairs.shape[0])
    kc = (ctypes.c_void_p * max(L, 1))(*[_dev(t) for t in k_caches])
    vc = (ctypes.c_void_p * max(L, 1))(*[_dev(t) for t in v_caches])
    ref = k_caches[0]
    block_bytes = ref[0].numel() * ref.element_size()
    _check(load().pa_copy_blocks(kc, vc, L, _dev(pairs, torch.int32), P, block_bytes,
                                 int(ref.shape[0]), _stream_ptr(stream)), "pa_copy_blocks")


def pa_swap_blocks(src_pools, dst_pools, pairs, stream=None) -> None:
    """Copies block ``pairs[p][0]`` of ``src_pools[l]`` onto block ``pairs[p][1]`` of
    ``dst_pools[l]`` for every pool pair; pools are CUDA tensors or pinned host
    tensors ``[blocks, ...]`` of the same block size; ``pairs`` is an int32
    ``[P, 2]`` tensor on the device or in pinned host memory."""
    import torch
    L = len(src_pools)
    if len(dst_pools) != L:
        raise ValueError("one destination per source pool")

    def ptr(t):
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError("contiguous CUDA or pinned host tensor expected")
        return t.data_ptr()
    sp = (ctypes.c_void_p * max(L, 1))(*[ptr(t) for t in src_pools])
    dp = (ctypes.c_void_p * max(L, 1))(*[ptr(t) for t in dst_pools])
    ref_s, ref_d = src_pools[0], dst_pools[0]
    block_bytes = ref_s[0].numel() * ref_s.element_size()
    if ref_d[0].numel() * ref_d.element_size() != block_bytes:
        raise ValueError("source and destination blocks differ in size")
    if pairs.dtype != torch.int32:
        raise TypeError("int32 pairs expected")
    _check(load().pa_swap_blocks(sp, dp, L, ptr(pairs), int(pairs.shape[0]), block_bytes,
                                 int(ref_s.shape[0]), int(ref_d.shape[0]), _stream_ptr(stream)),
           "pa_swap_blocks")


def pa_decode_workspace_size(B: int, H: int, d: int) -> int:
    return int(load().pa_decode_workspace_size(B, H, d))


def pa_decode_workspace_init(workspace, stream=None) -> None:
    _check(load().pa_decode_workspace_init(_dev(workspace), workspace.numel() *
                                           workspace.element_size(), _stream_ptr(stream)),
           "pa_decode_workspace_init")


def pa_decode(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
              scale: float, out, workspace, stream=None) -> None:
    """``q/out [B, H, d]``, caches ``[N, bs, Hkv, d]``, ``block_tables [B, max_blocks]``
    int32, ``context_lens [B]`` int32, ``workspace`` a zero-initialised byte tensor."""
    import torch
    B, H, d = q.shape
    N, bs, Hkv, _ = k_cache.shape
    _check(load().pa_decode(_dev(q), _dev(k_cache), _dev(v_cache),
                            _dev(block_tables, torch.int32), int(block_tables.shape[1]),
                            _dev(context_lens, torch.int32), int(max_context_len), B, H, Hkv, d,
                            bs, N, float(scale), _dtype_code(q), _dev(out), _dev(workspace),
                            workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "pa_decode")


def pa_multi_query_workspace_size(B: int, H: int, Hkv: int, d: int, max_q_len: int) -> int:
    return int(load().pa_multi_query_workspace_size(B, H, Hkv, d, max_q_len))


def pa_multi_query(q, q_start, k_cache, v_cache, block_tables, context_lens, max_q_len: int,
                   scale: float, out, workspace, stream=None) -> None:
    """``q/out [T, H, d]`` (the last ``q_start[i+1]-q_start[i]`` tokens of sequence i,
    concatenated), ``q_start [B+1]`` int32, caches ``[N, bs, Hkv, d]``,
    ``block_tables [B, max_blocks]`` and ``context_lens [B]`` int32, ``workspace`` a
    zero-initialised byte tensor of ``pa_multi_query_workspace_size`` bytes."""
    import torch
    T, H, d = q.shape
    N, bs, Hkv, _ = k_cache.shape
    B = int(context_lens.shape[0])
    _check(load().pa_multi_query(_dev(q), _dev(q_start, torch.int32), _dev(k_cache),
                                 _dev(v_cache), _dev(block_tables, torch.int32),
                                 int(block_tables.shape[1]), _dev(context_lens, torch.int32),
                                 int(max_q_len), B, H, Hkv, d, bs, N, float(scale),
                                 _dtype_code(q), _dev(out), _dev(workspace),
                                 workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream)),
           "pa_multi_query")


def pa_multi_query_tc_workspace_size(B: int, H: int, Hkv: int, d: int) -> int:
    return int(load().pa_multi_query_tc_workspace_size(B, H, Hkv, d))


def pa_multi_query_tc(q, q_start, k_cache, v_cache, block_tables, context_lens, max_q_len: int,
                      scale: float, out, workspace=None, stream=None) -> None:
    """``pa_multi_query`` on the tcgen05 tensor cores: ``q/out [T, H, 128]``,
    ``q_start [B+1]`` int32, caches ``[N, bs, Hkv, 128]``, ``block_tables
    [B, max_blocks]`` and ``context_lens [B]`` int32; ``workspace`` a
    zero-initialised byte tensor of ``pa_multi_query_tc_workspace_size``
    bytes (needed when ``max_q_len * H / Hkv <= 128``)."""
    import torch
    T, H, d = q.shape
    N, bs, Hkv, _ = k_cache.shape
    B = int(context_lens.shape[0])
    ws_ptr, ws_bytes = (None, 0) if workspace is None else (
        _dev(workspace), workspace.numel() * workspace.element_size())
    _check(load().pa_multi_query_tc(_dev(q), _dev(q_start, torch.int32), T, _dev(k_cache),
                                    _dev(v_cache), _dev(block_tables, torch.int32),
                                    int(block_tables.shape[1]), _dev(context_lens, torch.int32),
                                    int(max_q_len), B, H, Hkv, d, bs, N, float(scale),
                                    _dtype_code(q), _dev(out), ws_ptr, ws_bytes,
                                    _stream_ptr(stream)),
           "pa_multi_query_tc")


def pa_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                  max_context_len: int, scale: float, out, workspace, stream=None,
                  _name="pa_decode_fp8") -> None:
    """``pa_decode`` over an FP8 cache: ``k_cache/v_cache [N, bs, Hkv, 128]`` uint8
    codes and ``k_scale/v_scale [N, Hkv, bs]`` float32 scales."""
    import torch
    B, H, d = q.shape
    N, bs, Hkv, _ = k_cache.shape
    _check(getattr(load(), _name)(_dev(q), _dev(k_cache, torch.uint8), _dev(v_cache, torch.uint8),
                                _dev(k_scale, torch.float32), _dev(v_scale, torch.float32),
                                _dev(block_tables, torch.int32), int(block_tables.shape[1]),
                                _dev(context_lens, torch.int32), int(max_context_len), B, H, Hkv,
                                d, bs, N, float(scale), _dtype_code(q), _dev(out),
                                _dev(workspace), workspace.numel() * workspace.element_size(),
                                _stream_ptr(stream)),
           _name)


def pa_decode_int8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                   max_context_len: int, scale: float, out, workspace, stream=None) -> None:
    """``pa_decode_fp8`` over an INT8 cache (from ``pa_reshape_and_cache_int8``)."""
    pa_decode_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                  max_context_len, scale, out, workspace, stream, _name="pa_decode_int8")


def pa_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                      scale: float, out, stream=None) -> None:
    """``pa_decode`` for callers that cannot allocate: the scratch is the
    library's own per-device array, so no workspace is passed.  Calls that
    overlap on the GPU share that array and must be serialised."""
    import torch
    B, H, d = q.shape
    N, bs, Hkv, _ = k_cache.shape
    _check(load().pa_decode_noalloc(_dev(q), _dev(k_cache), _dev(v_cache),
                                    _dev(block_tables, torch.int32), int(block_tables.shape[1]),
                                    _dev(context_lens, torch.int32), int(max_context_len), B, H,
                                    Hkv, d, bs, N, float(scale), _dtype_code(q), _dev(out),
                                    _stream_ptr(stream)),
           "pa_decode_noalloc")


def pa_check_device_errors(stream=None) -> int:
    """Synchronises the stream; returns the error word's bits (and clears them)."""
    flags = ctypes.c_uint32(0)
    st = load().pa_check_device_errors(_stream_ptr(stream), ctypes.byref(flags))
    if st not in (PA_OK, 4, 7):
        raise PaError(st, "pa_check_device_errors")
    return int(flags.value)


def pa_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launches the bounded-wait self-test (see pa.h); read the result with
    pa_check_device_errors()."""
    _check(load().pa_selftest_wait_timeout(int(limit_us), _stream_ptr(stream)),
           "pa_selftest_wait_timeout")


def pa_measure_mma_ceiling(bf16: bool, iters: int, sink, stream=None) -> int:
    """Launches the mma.sync throughput-ceiling kernel (see pa.h) writing into
    the device tensor ``sink``; returns the launch's floating-point operations."""
    flops = ctypes.c_int64(0)
    _check(load().pa_measure_mma_ceiling(int(bool(bf16)), int(iters), sink.data_ptr(),
                                         sink.numel() * sink.element_size(),
                                         ctypes.byref(flops), _stream_ptr(stream)),
           "pa_measure_mma_ceiling")
    return int(flops.value)


def pa_decode_grid_size() -> int:
    return int(load().pa_decode_grid_size())


# ------------------------------------------------------------------------- allocator
def _np_ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Allocator:
    """The host block allocator (``pa_alloc_*``); owns one ``pa_allocator``."""

    def __init__(self, num_blocks: int, block_size: int, init_free_order=None):
        self._lib = load()
        self._h = ctypes.c_void_p()
        order = None
        if init_free_order is not None:
            self._order = np.ascontiguousarray(init_free_order, dtype=np.int32)
            order = _np_ptr(self._order)
        _check(self._lib.pa_alloc_create(num_blocks, block_size, order, ctypes.byref(self._h)),
               "pa_alloc_create")
        self.num_blocks, self.block_size = num_blocks, block_size

    def close(self):
        if self._h:
            self._lib.pa_alloc_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc(self, seq_id: int, num_tokens: int) -> None:
        _check(self._lib.pa_alloc(self._h, seq_id, num_tokens), "pa_alloc")

    def append_slot(self, seq_id: int):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.pa_append_slot(self._h, seq_id, ctypes.byref(slot), ctypes.byref(src),
                                        ctypes.byref(dst)), "pa_append_slot")
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def append_batch(self, seq_ids, slot_mapping=None, cow_pairs=None, tokens=None):
        """Returns ``(slot_mapping int64 [B], cow_pairs int32 [P, 2])``; output arrays may
        be passed in (e.g. pinned host memory as numpy views).  With ``tokens`` (one id
        per sequence) this is ``pa_append_batch_tokens``."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        B = ids.shape[0]
        slots = np.empty(B, np.int64) if slot_mapping is None else slot_mapping
        pairs = np.empty((max(B, 1), 2), np.int32) if cow_pairs is None else cow_pairs
        n = ctypes.c_int32()
        if tokens is None:
            _check(self._lib.pa_append_batch(self._h, _np_ptr(ids), B, _np_ptr(slots),
                                             _np_ptr(pairs), ctypes.byref(n)), "pa_append_batch")
        else:
            tok = np.ascontiguousarray(tokens, dtype=np.int32)
            if tok.shape[0] != B:
                raise ValueError("one token per sequence")
            _check(self._lib.pa_append_batch_tokens(self._h, _np_ptr(ids), _np_ptr(tok), B,
                                                    _np_ptr(slots), _np_ptr(pairs),
                                                    ctypes.byref(n)), "pa_append_batch_tokens")
        return slots, pairs[: n.value]

    def alloc_prompt(self, seq_id: int, tokens) -> int:
        """``pa_alloc_prompt``: returns the number of leading tokens already cached."""
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        cached = ctypes.c_int32()
        _check(self._lib.pa_alloc_prompt(self._h, seq_id, _np_ptr(tok) if tok.size else None,
                                         int(tok.shape[0]), ctypes.byref(cached)),
               "pa_alloc_prompt")
        return cached.value

    def append_token(self, seq_id: int, token: int):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.pa_append_token(self._h, seq_id, int(token), ctypes.byref(slot),
                                         ctypes.byref(src), ctypes.byref(dst)), "pa_append_token")
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def set_swap_pool(self, num_host_blocks: int) -> None:
        _check(self._lib.pa_alloc_set_swap_pool(self._h, num_host_blocks),
               "pa_alloc_set_swap_pool")
        self.host_blocks = num_host_blocks

    def _swap(self, fn, name, seq_id):
        cap = max(self.num_blocks, getattr(self, "host_blocks", 0), 1)
        out = np.empty((cap, 2), np.int32)
        n = ctypes.c_int32()
        _check(fn(self._h, seq_id, _np_ptr(out), cap, ctypes.byref(n)), name)
        return out[: n.value]

    def swap_out(self, seq_id: int) -> np.ndarray:
        """``pa_swap_out``: the copies ``[n, 2]`` {device block, host block}."""
        return self._swap(self._lib.pa_swap_out, "pa_swap_out", seq_id)

    def swap_in(self, seq_id: int) -> np.ndarray:
        """``pa_swap_in``: the copies ``[n, 2]`` {host block, device block}."""
        return self._swap(self._lib.pa_swap_in, "pa_swap_in", seq_id)

    def swap_stats(self) -> dict:
        s = SwapStats()
        _check(self._lib.pa_swap_stats_get(self._h, ctypes.byref(s)), "pa_swap_stats_get")
        return {f: getattr(s, f) for f, _ in SwapStats._fields_}

    def host_free_list(self):
        cap = max(getattr(self, "host_blocks", 0), 1)
        out = np.empty(cap, np.int32)
        n = ctypes.c_int32()
        _check(self._lib.pa_host_free_list(self._h, _np_ptr(out), cap, ctypes.byref(n)),
               "pa_host_free_list")
        return out[: n.value].tolist()

    def prefix_stats(self) -> dict:
        s = PrefixStats()
        _check(self._lib.pa_prefix_stats_get(self._h, ctypes.byref(s)), "pa_prefix_stats_get")
        return {f: getattr(s, f) for f, _ in PrefixStats._fields_}

    def fork(self, parent: int, child: int) -> None:
        _check(self._lib.pa_fork(self._h, parent, child), "pa_fork")

    def free(self, seq_id: int) -> None:
        _check(self._lib.pa_free(self._h, seq_id), "pa_free")

    def export(self, seq_ids, max_blocks: int, block_tables=None, context_lens=None):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        B = ids.shape[0]
        tbl = np.empty((B, max_blocks), np.int32) if block_tables is None else block_tables
        lens = np.empty(B, np.int32) if context_lens is None else context_lens
        _check(self._lib.pa_export(self._h, _np_ptr(ids), B, max_blocks, _np_ptr(tbl),
                                   _np_ptr(lens)), "pa_export")
        return tbl, lens

    def seq_slots(self, seq_id: int, start: int, count: int) -> np.ndarray:
        out = np.empty(max(count, 1), np.int64)
        _check(self._lib.pa_seq_slots(self._h, seq_id, start, count, _np_ptr(out)),
               "pa_seq_slots")
        return out[:count]

    def seq_info(self, seq_id: int):
        ln, nb = ctypes.c_int32(), ctypes.c_int32()
        _check(self._lib.pa_seq_info(self._h, seq_id, ctypes.byref(ln), ctypes.byref(nb)),
               "pa_seq_info")
        return ln.value, nb.value

    def block_ref(self, block: int) -> int:
        r = ctypes.c_int32()
        _check(self._lib.pa_block_ref(self._h, block, ctypes.byref(r)), "pa_block_ref")
        return r.value

    def free_list(self):
        out = np.empty(max(self.num_blocks, 1), np.int32)
        n = ctypes.c_int32()
        _check(self._lib.pa_free_list(self._h, _np_ptr(out), self.num_blocks, ctypes.byref(n)),
               "pa_free_list")
        return out[: n.value].tolist()

    def stats(self) -> dict:
        s = AllocStats()
        _check(self._lib.pa_alloc_stats_get(self._h, ctypes.byref(s)), "pa_alloc_stats_get")
        return {f: getattr(s, f) for f, _ in AllocStats._fields_}


class Step:
    """The decode step executor (``pa_step_*``) for one layer's caches.

    Allocates its two staging buffers (pinned host, device; ``depth`` slots
    each) and the decode workspace as torch tensors and exposes each slot's
    host regions as tensors (``slot(i)``; ``q``, ``k_new``, ``v_new``, ``out``
    are slot 0's).  Fill a slot's inputs, then :meth:`run` (submit and wait),
    or :meth:`submit` / :meth:`wait` to overlap the next step's host work with
    this one's device work.  With ``kv_format`` "fp8" or "int8" the caches
    are 8-bit codes (uint8) with ``k_scale``/``v_scale``, and ``dtype`` gives
    the 16-bit type of the inputs."""

    def __init__(self, alloc: Allocator, B: int, H: int, Hkv: int, d: int, max_blocks: int,
                 max_context_len: int, k_cache, v_cache, scale: float, k_scale=None,
                 v_scale=None, dtype=None, depth: int = 1, kv_format: str = "native"):
        import torch
        self._lib = load()
        N, bs = int(k_cache.shape[0]), int(k_cache.shape[1])
        if tuple(k_cache.shape) != (N, bs, Hkv, d) or v_cache.shape != k_cache.shape:
            raise ValueError("caches must be [num_blocks, block_size, Hkv, d]")
        q8 = {"native": 0, "fp8": 1, "int8": 2}[kv_format]
        if q8 and (k_scale is None or v_scale is None or
                   dtype not in (torch.float16, torch.bfloat16)):
            raise ValueError("an 8-bit cache needs k_scale, v_scale and dtype (of q, k/v_new)")
        # the library sees raw pointers: a pool of the wrong element size
        # would be written past its end, so the format must match the tensors
        want = (torch.uint8,) if q8 else (torch.float16, torch.bfloat16)
        if k_cache.dtype not in want or v_cache.dtype != k_cache.dtype:
            raise ValueError("kv_format %r needs caches of %s, got %s" % (kv_format, want,
                                                                         k_cache.dtype))
        if not q8 and (k_scale is not None or v_scale is not None):
            raise ValueError("scales given for a 16-bit cache: pass kv_format")
        if q8 and (tuple(k_scale.shape) != (N, Hkv, bs) or tuple(v_scale.shape) != (N, Hkv, bs)
                   or k_scale.dtype != torch.float32 or v_scale.dtype != torch.float32):
            raise ValueError("scales must be float32 [num_blocks, Hkv, block_size]")
        dt = dtype if q8 else k_cache.dtype
        self.desc = StepDesc(B, H, Hkv, d, bs, N, max_blocks, max_context_len,
                             PA_F16 if dt == torch.float16 else PA_BF16, scale, q8, depth)
        lay = StepLayout()
        _check(self._lib.pa_step_layout_get(ctypes.byref(self.desc), ctypes.byref(lay)),
               "pa_step_layout_get")
        self.layout = {f: getattr(lay, f) for f, _ in StepLayout._fields_}
        dev = k_cache.device
        total = depth * lay.total
        # 256-byte alignment: over-allocate and take an aligned view
        self._host_raw = torch.empty(total + 256, dtype=torch.uint8, pin_memory=True)
        self._dev_raw = torch.empty(total + 256, dtype=torch.uint8, device=dev)
        self.host = self._aligned(self._host_raw, total)
        self.dev = self._aligned(self._dev_raw, total)
        self.ws = torch.zeros(pa_decode_workspace_size(B, H, d), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize(dev)
        self._caches = (k_cache, v_cache, k_scale, v_scale)
        self.alloc = alloc
        self._h = ctypes.c_void_p()
        _check(self._lib.pa_step_create(ctypes.byref(self.desc), alloc._h, _dev(k_cache),
                                        _dev(v_cache),
                                        _dev(k_scale, torch.float32) if q8 else None,
                                        _dev(v_scale, torch.float32) if q8 else None,
                                        self.host.data_ptr(), self.dev.data_ptr(),
                                        self.ws.data_ptr(), self.ws.numel(),
                                        ctypes.byref(self._h)), "pa_step_create")
        shapes = {"q": ((B, H, d), dt), "k_new": ((B, Hkv, d), dt), "v_new": ((B, Hkv, d), dt),
                  "out": ((B, H, d), dt), "slot_mapping": ((B,), torch.int64),
                  "block_tables": ((B, max_blocks), torch.int32),
                  "context_lens": ((B,), torch.int32)}
        self._slots = []
        for i in range(depth):
            views = {}
            for name, (shape, dtype_) in shapes.items():
                n = int(np.prod(shape)) * torch.empty(0, dtype=dtype_).element_size()
                off = i * lay.total + self.layout[name]
                views[name] = self.host[off: off + n].view(dtype_).view(*shape)
            self._slots.append(views)
        for name in shapes:
            setattr(self, name, self._slots[0][name])

    @staticmethod
    def _aligned(raw, n):
        off = (-raw.data_ptr()) % 256
        return raw[off: off + n]

    def slot(self, i: int) -> dict:
        """The host regions of staging slot i (q, k_new, v_new, out, slot_mapping,
        block_tables, context_lens)."""
        return self._slots[i]

    def _ids(self, seq_ids):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        if ids.shape[0] != self.desc.B:
            raise ValueError("the executor runs %d sequences per step" % self.desc.B)
        return ids

    def submit(self, seq_ids, stream=None) -> int:
        """Submits one step (no wait); returns its slot."""
        slot = ctypes.c_int32()
        _check(self._lib.pa_step_submit(self._h, _np_ptr(self._ids(seq_ids)), _stream_ptr(stream),
                                        ctypes.byref(slot)), "pa_step_submit")
        return slot.value

    def wait(self, slot: int) -> None:
        _check(self._lib.pa_step_wait(self._h, slot), "pa_step_wait")

    def run(self, seq_ids, stream=None) -> None:
        _check(self._lib.pa_step_run(self._h, _np_ptr(self._ids(seq_ids)), _stream_ptr(stream)),
               "pa_step_run")

    def close(self):
        if self._h:
            self._lib.pa_step_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
