"""Shared helpers of the parity tests: one workload, run by the oracle on the
host and by libpa.so on the GPU, with the same seeded inputs."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from paged_kv_cache_103_gb300 import binding
from paged_kv_cache_103_gb300 import workloads as wl

ATOL, RTOL = 2e-3, 1e-2   # |gpu - ref| <= ATOL + RTOL * |ref| per element
THREADS = max(1, os.cpu_count() or 1)


def build_tables(w: wl.Workload):
    """Block tables from the oracle's allocator model.

    Without a shared prefix every sequence holds n - 1 tokens and the step
    appends its n-th (the slot returned is where the step's new K/V goes), so
    the decode reads n tokens.  With a shared prefix the history is the prefix
    (shared by forks) plus each sequence's suffix; the step decodes first and
    appends afterwards.
    """
    m = oracle.BlockManagerModel(w.num_blocks, w.block_size, w.free_order)
    B = w.B
    if w.prefix_len:
        m.allocate(0, w.prefix_len)
        for s in range(1, B):
            m.fork(0, s)
        for s in range(B):
            for _ in range(int(w.context_lens[s]) - w.prefix_len):
                m.append_slot(s)
        return m, None
    for i in range(B):
        m.allocate(i, int(w.context_lens[i]) - 1)
    slots, pairs = m.append_batch(range(B))
    assert not pairs
    return m, np.asarray(slots, dtype=np.int64)


def nan_tails(m, k_cache, v_cache):
    """Fills the unused slots of every sequence's last block with NaN."""
    bs = m.block_size
    nan = torch.tensor(float("nan"), dtype=k_cache.dtype)
    for s, table in m.allocated.items():
        n = m.lens[s]
        for pos in range(n, len(table) * bs):
            k_cache[table[pos // bs], pos % bs] = nan
            v_cache[table[pos // bs], pos % bs] = nan


def dtype_code(w):
    return oracle.DTYPE_F16 if w.dtype == "f16" else oracle.DTYPE_BF16


def oracle_decode(w, q, k_cache, v_cache, tbl, lens):
    return oracle.decode(wl.bits(q), wl.bits(k_cache), wl.bits(v_cache), tbl, lens, w.scale,
                         dtype_code(w), num_threads=THREADS)


def assert_close(gpu: torch.Tensor, ref: np.ndarray, what=""):
    g = gpu.double().numpy()
    assert g.shape == ref.shape
    assert np.isfinite(g).all(), "%s: non-finite output" % what
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    rel = err / np.maximum(np.abs(ref), 1e-30)
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError("%s: %d elements out of tolerance; worst at %s gpu=%r ref=%r; "
                             "max abs %.3g max rel %.3g" % (what, int(bad.sum()), idx, g[idx],
                                                          ref[idx], err.max(), rel.max()))
    return float(err.max(initial=0.0)), float(rel[np.abs(ref) > 1e-3].max(initial=0.0))


class GpuRun:
    """Device copies of a workload's tensors plus a decode workspace."""

    def __init__(self, w, host, dev="cuda"):
        self.w = w
        self.q = host["q"].to(dev)
        self.k_cache = host["k_cache"].to(dev)
        self.v_cache = host["v_cache"].to(dev)
        self.out = torch.empty_like(self.q)
        self.ws = torch.empty(binding.pa_decode_workspace_size(w.B, w.H, w.d), dtype=torch.uint8,
                              device=dev)
        binding.pa_decode_workspace_init(self.ws)

    def append(self, k_new, v_new, slots):
        binding.pa_reshape_and_cache(k_new.cuda(), v_new.cuda(),
                                     torch.from_numpy(np.asarray(slots, np.int64)).cuda(),
                                     self.k_cache, self.v_cache)

    def decode(self, tbl, lens):
        self.tbl = torch.from_numpy(np.ascontiguousarray(tbl, np.int32)).cuda()
        self.lens = torch.from_numpy(np.ascontiguousarray(lens, np.int32)).cuda()
        binding.pa_decode(self.q, self.k_cache, self.v_cache, self.tbl, self.lens,
                          int(np.max(lens)) if len(lens) else 0, self.w.scale, self.out, self.ws)
        return self.out


def bit_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.contiguous().view(torch.int16).cpu(), b.contiguous().view(torch.int16))
