#!/usr/bin/env python3
"""Benchmark of one paged decode layer-step on a GB300.

Workload: the LLaMA-13B-shaped MHA decode batch -- 64 sequences, 40 query
heads = 40 KV heads of 128, fp16, block size 16, context lengths uniform in
[128, 2048], blocks scattered over a pool of 1.25x the need.  A step is the
whole hot path over the batch: the KV append of each sequence's new token
(pa_reshape_and_cache) and the decode attention over its context (pa_decode);
the e2e leg adds the host allocator step (pa_append_batch + pa_export), the
host->device copies of that step's inputs from pinned memory and the
device->host copy of the output.

The metric is KV-cache bytes attended per second (GB/s): the K and V bytes of
every context token, divided by the step time.  One JSON line is printed.

With ``--kv-format fp8`` (or ``int8``) the cache holds E4M3 (or INT8) codes
with one fp32 scale per (token, KV head) (pa_reshape_and_cache_fp8 /
pa_decode_fp8, or their _int8 forms); the bytes are then the codes and scales
actually read, and ``tokens_per_s`` compares the formats.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV GB/s (% of GB300 HBM peak); decode tokens/s"
L2_BYTES = 129 * 10 ** 6
FALLBACK_HBM_GBS = 6800.0


def kv_bytes(lens, Hkv, d, e=2, fp8=False):
    """K and V bytes of every context token: 16-bit values, or E4M3 codes plus
    one fp32 scale per (token, KV head)."""
    tokens = int(sum(int(n) for n in lens))
    if fp8:
        return 2 * tokens * Hkv * (d + 4)
    return 2 * tokens * Hkv * d * e


def algorithmic_bytes(lens, B, H, Hkv, d, bs, e=2, fp8=False):
    """Bytes the decode must move: K and V of every context token, Q and the
    output, the used table entries and the lengths."""
    table = sum((int(n) + bs - 1) // bs for n in lens) * 4
    return kv_bytes(lens, Hkv, d, e, fp8) + 2 * B * H * d * 2 + table + 4 * B


def max_over_ranks(value, dist, device):
    """The largest `value` over all ranks (the slowest replica sets the time);
    `dist` is torch.distributed or None for a single process."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, ms):
    """Units per second over all replicas: every rank processes its own copy
    of the batch (weak scaling), timed by the slowest rank."""
    return world * units_per_rank / (ms * 1e-3)


def load_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(name):
    """Per-launch DRAM bytes from the committed ncu summary of this kernel and
    workload, or None if the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", name)
    src = os.path.join(ROOT, "paged_kv_cache_103_gb300", "csrc", "pa_decode.cu")
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and not line.startswith(" "):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        with open(src, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()[:16]
        if fields.get("pa_decode.cu sha256 prefix") != sha:
            return None
        return int(float(fields["dram bytes per launch"]))
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1, t_pre=None):
        """Clocks over [t_pre, t1]: the untimed pre-roll (if any) and the timed
        region right after it, one stretch of the same load."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        start = t0 if t_pre is None else t_pre
        inside = [s for t, s in self.samples if start <= t <= t1]
        timed = sum(1 for t, _ in self.samples if t0 <= t <= t1)
        note = "timed region" if t_pre is None else "pre-roll + timed region (one stretch of load)"
        if not inside:   # region shorter than the sampling period: nearest samples
            inside = [s for t, s in self.samples if start - 0.25 <= t <= t1 + 0.25]
            note = "within 250 ms of the timed region"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in inside:
            try:
                sm.append(float(s[0]))
                mx.append(float(s[1]))
                for n, v in zip(names, s[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
            except Exception:
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_timed_region": timed, "window": note,
                "window_s": round(t1 - start, 3)}


WORKLOADS = {
    "llama13b": lambda B: wl_mod().llama13b(B=B or 64),
    "gqa7b_1x1024": lambda B: wl_mod().gqa7b(1, 1024),
    "gqa7b_8x4096": lambda B: wl_mod().gqa7b(8, 4096),
    "gqa7b_8x8192": lambda B: wl_mod().gqa7b(8, 8192),
    "gqa7b_16x32768": lambda B: wl_mod().gqa7b(16, 32768),
    "qwen_longtail_bs8": lambda B: wl_mod().qwen_longtail(8),
    "qwen_longtail_bs16": lambda B: wl_mod().qwen_longtail(16),
    "qwen_longtail_bs32": lambda B: wl_mod().qwen_longtail(32),
    "prefix_share": lambda B: wl_mod().prefix_share(),
    "multiturn_prefix": lambda B: wl_mod().multiturn_prefix(convs=B or 128),
}
CONTEXT_MIX = {
    "llama13b": "uniform[128,2048]",
    "gqa7b_1x1024": "all 1024", "gqa7b_8x4096": "all 4096", "gqa7b_8x8192": "all 8192",
    "gqa7b_16x32768": "all 32768",
    "qwen_longtail_bs8": "95% lognormal(median 1500, sigma 1) <= 8192, 5% uniform[16384,24576]",
    "qwen_longtail_bs16": "95% lognormal(median 1500, sigma 1) <= 8192, 5% uniform[16384,24576]",
    "qwen_longtail_bs32": "95% lognormal(median 1500, sigma 1) <= 8192, 5% uniform[16384,24576]",
    "prefix_share": "1024-token prefix shared by 256 sequences + uniform[64,512] suffixes",
    "multiturn_prefix": "end of 4-turn conversations: 1024-token shared system prompt, user "
                        "U[32,256] and reply U[64,512] tokens per turn, prefix-cached allocation",
}


def preroll_replays(stream, replay, seconds):
    """Untimed replays for about `seconds` of GPU time, queued back to back
    (one replay is timed first to size the count)."""
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        replay()
        e1.record(stream)
    e1.synchronize()
    one = max(e0.elapsed_time(e1) * 1e-3, 1e-6)
    n = max(1, int(math.ceil(seconds / one)))
    with torch.cuda.stream(stream):
        for _ in range(n):
            replay()
    return {"replays": n + 1, "seconds": round((n + 1) * one, 3), "timed": False}


def unique_roofline(roof, alg_unique, dec_ms, peak):
    """For workloads whose tables share blocks: `achieved` and `frac` divide
    the unique bytes (a shared block's rows once: the most DRAM has to move),
    the logical ones (a shared block once per sequence that reads it) move to
    `achieved_logical` / `frac_logical`."""
    achieved = alg_unique / (dec_ms * 1e-3) / 1e9
    roof["achieved_logical"] = roof["achieved"]
    roof["frac_logical"] = roof["frac"]
    roof["logical_bytes_per_launch"] = roof["algorithmic_bytes_per_launch"]
    roof["algorithmic_bytes_per_launch"] = int(alg_unique)
    roof["achieved"] = round(achieved, 1)
    roof["frac"] = round(achieved / peak, 4)
    roof["bytes"] = ("unique: K/V of the distinct cache rows the tables reach (a shared block's "
                     "rows once) + q + out + table entries + lengths")
    return roof


def wl_mod():
    from paged_kv_cache_103_gb300 import workloads
    return workloads


def play_trace(alloc, tr):
    """Runs a multi-turn trace through the product allocator with prefix
    caching (pa_alloc_prompt, pa_append_batch_tokens, pa_free) and times the
    host calls (ctypes overhead included)."""
    import numpy as np
    t_prompt = t_append = 0.0
    prompts = prompt_tokens = cached_tokens = appended = 0
    for turn in tr["turns"]:
        for sid, prompt in turn["prompts"]:
            p = np.asarray(prompt, dtype=np.int32)
            t0 = time.perf_counter()
            cached_tokens += alloc.alloc_prompt(sid, p)
            t_prompt += time.perf_counter() - t0
            prompts += 1
            prompt_tokens += len(prompt)
        for step in turn["replies"]:
            ids = np.asarray([s for s, _ in step], dtype=np.int64)
            tok = np.asarray([t for _, t in step], dtype=np.int32)
            t0 = time.perf_counter()
            alloc.append_batch(ids, tokens=tok)
            t_append += time.perf_counter() - t0
            appended += len(step)
        for sid in turn["free"]:
            alloc.free(sid)
    st = alloc.prefix_stats()
    return {"prompts": prompts, "prompt_tokens": prompt_tokens, "cached_tokens": cached_tokens,
            "token_hit_rate": round(cached_tokens / max(prompt_tokens, 1), 4),
            "block_hit_rate": round(st["hits"] / max(st["lookups"], 1), 4),
            "us_per_prompt": round(t_prompt * 1e6 / max(prompts, 1), 2),
            "us_per_appended_token": round(t_append * 1e6 / max(appended, 1), 3),
            "cache_entries": st["entries"], "evicted": st["evicted"],
            "note": "host allocator via ctypes; the cached tokens skip prefill"}


def grow_pool_for_e2e(w, e2e_extra):
    """Room for the e2e leg's two loops of e2e_extra appended tokens per
    sequence: extra blocks at the back of the free list, so the batch's own
    blocks (and the timed decode over them) are as the workload has them.
    The prefix-cached trace keeps its pool: its size is part of that workload."""
    import numpy as np

    if "trace" in w.extra:
        return
    grow = w.B * (int(math.ceil((2 * e2e_extra + 1) / w.block_size)) + 1)
    w.free_order = np.concatenate([np.asarray(w.free_order, dtype=np.int32),
                                   np.arange(w.num_blocks, w.num_blocks + grow, dtype=np.int32)])
    w.num_blocks += grow


def populate(alloc, w):
    """Every sequence's history in the allocator (all but the step's own
    token): prefix-shared workloads fork one prompt and append each suffix."""
    if w.prefix_len:
        alloc.alloc(0, w.prefix_len)
        for s in range(1, w.B):
            alloc.fork(0, s)
        for s in range(w.B):
            for _ in range(int(w.context_lens[s]) - 1 - w.prefix_len):
                alloc.append_slot(s)
    else:
        for i in range(w.B):
            alloc.alloc(i, int(w.context_lens[i]) - 1)


def build_tables(w, e2e_extra):
    """The product allocator holding every sequence's history (all but the
    step's own token), then the step's token appended; returns the allocator,
    the step's slots, the exported tables and lengths, the table width and the
    decode batch's sequence ids."""
    import numpy as np

    from paged_kv_cache_103_gb300 import binding

    alloc = binding.Allocator(w.num_blocks, w.block_size, w.free_order)
    if "trace" in w.extra:
        tr = w.extra["trace"]
        w.extra["prefix_cache"] = play_trace(alloc, tr)
        seqs = [tr["last"][c] for c in range(w.B)]
        step_tok = np.random.default_rng(w.seed).integers(0, tr["vocab"], w.B).astype(np.int32)
        slots, pairs = alloc.append_batch(seqs, tokens=step_tok)
        assert len(pairs) == 0
        max_blocks = int(math.ceil((int(w.context_lens.max()) + 1 + 2 * e2e_extra)
                                   / w.block_size)) + 1
        tbl, lens = alloc.export(seqs, max_blocks)
        return alloc, slots, tbl, lens, max_blocks, seqs
    populate(alloc, w)
    seqs = list(range(w.B))
    slots, pairs = alloc.append_batch(seqs)
    assert len(pairs) == 0
    # room for the e2e leg's two loops of e2e_extra steps
    max_blocks = int(math.ceil((int(w.context_lens.max()) + 2 * e2e_extra)
                               / w.block_size)) + 1
    tbl, lens = alloc.export(seqs, max_blocks)
    return alloc, slots, tbl, lens, max_blocks, seqs


def unique_kv_bytes(tbl, lens, bs, Hkv, d, e=2, fp8=False):
    """K and V bytes of the distinct cache rows a decode reads: a physical
    block shared by several tables counts once, with the most rows any of
    them uses."""
    rows = {}
    for i, n in enumerate(lens):
        n = int(n)
        for j in range((n + bs - 1) // bs):
            b = int(tbl[i, j])
            r = min(bs, n - j * bs)
            if rows.get(b, 0) < r:
                rows[b] = r
    tokens = sum(rows.values())
    return 2 * tokens * Hkv * ((d + 4) if fp8 else d * e)


def headline_config(args, w, lens, kvb, flush_l2):
    """The `config` object of the JSON line; both arms print the same one."""
    fp8 = args.kv_format != "native"
    fmt = args.kv_format
    l2_note = ("inputs larger than L2 (%.2f GB of KV per step)" % (kvb / 1e9) if not flush_l2
               else "L2 flushed between steps (512 MiB write + read outside the timed kernels; %.3f GB "
                    "of KV per step)" % (kvb / 1e9))
    return {"workload": args.workload + ("_%skv" % fmt if fp8 else "") + "_decode_layer_step",
            "batch": w.B, "kv_format": "%s + fp32 scale per (token, KV head)"
            % ("e4m3" if fmt == "fp8" else "int8") if fp8 else w.dtype,
            "q_heads": w.H, "kv_heads": w.Hkv, "head_dim": w.d,
            "block_size": w.block_size, "context_lens": CONTEXT_MIX[args.workload],
            "total_context_tokens": int(lens.sum()), "pool_blocks": w.num_blocks,
            "l2": l2_note}


def setup_workload(args):
    """The named workload, its host tensors and the product allocator holding
    every sequence's history; the step's own token is appended last, so the
    decode reads context_lens[i] tokens including it.  Returns the decode
    batch's sequence ids too."""
    w = WORKLOADS[args.workload](args.batch)
    grow_pool_for_e2e(w, args.e2e_extra)
    fp8 = args.kv_format != "native"      # an 8-bit cache: E4M3 or INT8 codes
    host = wl_mod().qkv(w, with_cache=not fp8)
    if fp8:
        host.update(wl_mod().fp8_cache(w) if args.kv_format == "fp8" else wl_mod().int8_cache(w))
    alloc, slots, tbl, lens, max_blocks, seqs = build_tables(w, args.e2e_extra)
    return w, host, alloc, slots, tbl, lens, max_blocks, seqs


def run_gpu(args):
    import numpy as np
    import torch

    from paged_kv_cache_103_gb300 import binding
    from paged_kv_cache_103_gb300 import build as pa_build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pa_build.build()
    binding.load()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    w, host, alloc, slots, tbl, lens, max_blocks, seqs = setup_workload(args)
    fp8 = args.kv_format != "native"      # an 8-bit cache: E4M3 or INT8 codes
    fmt = args.kv_format
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        q = host["q"].to(dev)
        if fp8:
            kc = host["k_codes"].to(dev)
            vc = host["v_codes"].to(dev)
            ks = host["k_scale"].to(dev)
            vs = host["v_scale"].to(dev)
        else:
            kc = host["k_cache"].to(dev)
            vc = host["v_cache"].to(dev)
        kn = host["k_new"].to(dev)
        vn = host["v_new"].to(dev)
        slots_d = torch.from_numpy(slots).to(dev)
        tbl_d = torch.from_numpy(tbl).to(dev)
        lens_d = torch.from_numpy(lens).to(dev)
        out = torch.empty_like(q)
        ws = torch.empty(binding.pa_decode_workspace_size(w.B, w.H, w.d), dtype=torch.uint8,
                         device=dev)
        binding.pa_decode_workspace_init(ws, stream)
    stream.synchronize()
    max_len = int(lens.max())

    # the step's two calls through the C ABI, for either cache format
    if fp8:
        q8_append = getattr(binding, "pa_reshape_and_cache_" + fmt)
        q8_decode = getattr(binding, "pa_decode_" + fmt)

        def append(kn_, vn_, slots_):
            q8_append(kn_, vn_, slots_, kc, vc, ks, vs, stream)

        def decode(q_, tbl_, lens_, max_len_, out_):
            q8_decode(q_, kc, vc, ks, vs, tbl_, lens_, max_len_, w.scale, out_, ws, stream)
    else:
        def append(kn_, vn_, slots_):
            binding.pa_reshape_and_cache(kn_, vn_, slots_, kc, vc, stream)

        def decode(q_, tbl_, lens_, max_len_, out_):
            binding.pa_decode(q_, kc, vc, tbl_, lens_, max_len_, w.scale, out_, ws, stream)

    def step():
        append(kn, vn, slots_d)
        decode(q, tbl_d, lens_d, max_len, out)

    for _ in range(args.warmup):
        step()
    if binding.pa_check_device_errors(stream):
        raise RuntimeError("device error flags set during warm-up")

    # ---- device-timed leg: inputs resident in HBM.  The step is replayed from
    # one CUDA graph (no host launch cost in the way) with an event on either
    # side; when the step's KV bytes would fit in L2, a 512 MiB write and
    # read-back before every timed replay evicts them, outside the events.
    kvb = kv_bytes(lens, w.Hkv, w.d, fp8=fp8)
    flush_l2 = kvb < 2 * L2_BYTES
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if flush_l2 else None
    # the step (append, then decode) as one graph; the decode alone as another
    # for the roofline
    g_step, g_decode = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        append(kn, vn, slots_d)
        decode(q, tbl_d, lens_d, max_len, out)
    with torch.cuda.graph(g_decode, stream=stream):
        decode(q, tbl_d, lens_d, max_len, out)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_step.replay()
            g_decode.replay()
    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)]
    evd = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)]
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)

    def evict():
        flush_buf.zero_()                   # write, then read back so
        torch.count_nonzero(flush_buf)      # that no dirty lines remain

    # Untimed pre-roll: step replays for at least `preroll_s` seconds right
    # before the timed region, so that clocks and power have settled and the
    # clock sampler has samples under this load.
    t_pre0 = time.time()
    preroll = preroll_replays(stream, lambda: (evict() if flush_l2 else None, g_step.replay()),
                              args.preroll_s)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()

    # each timed step is followed by one decode-alone replay, timed on its own
    # for the roofline; the step rate counts the step events only
    with torch.cuda.stream(stream):
        for k in range(K):
            if flush_l2:
                evict()
            ev[2 * k].record(stream)
            g_step.replay()
            ev[2 * k + 1].record(stream)
            if flush_l2:
                evict()
            evd[2 * k].record(stream)
            g_decode.replay()
            evd[2 * k + 1].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist:
        dist.barrier()
    step_ms = [ev[2 * k].elapsed_time(ev[2 * k + 1]) for k in range(K)]
    decode_ms = [evd[2 * k].elapsed_time(evd[2 * k + 1]) for k in range(K)]
    total_ms = sum(step_ms)              # the steps' kernels only
    total_ms = max_over_ranks(total_ms, dist, dev)
    flags = binding.pa_check_device_errors(stream)
    if flags:
        raise RuntimeError("device error flags 0x%x in the timed region" % flags)

    ms_per_step = total_ms / K
    value = whole_job_rate(kvb, world, ms_per_step) / 1e9
    alg = algorithmic_bytes(lens, w.B, w.H, w.Hkv, w.d, w.block_size, fp8=fp8)
    dec_avg_ms = sum(decode_ms) / len(decode_ms)
    achieved = alg / (dec_avg_ms * 1e-3) / 1e9
    peak, peak_kind = load_peak()

    # ---- e2e leg through the C ABI: host allocator step, pinned H2D, kernels, D2H
    e2e = run_e2e(args, w, host, alloc, kc, vc, ks if fp8 else None, vs if fp8 else None,
                  stream, max_blocks, fp8, seqs)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("%s KV, f16 MMA, fp32 accumulate" % ("e4m3" if fmt == "fp8" else "int8")
                  if fp8 else w.dtype),
        "data": ("synthetic (seeded N(0,1) Q and new K/V, seeded %s codes and scales, seeded "
                 "context lengths, random block placement)" % ("E4M3" if fmt == "fp8" else "INT8")
                 if fp8 else
                 "synthetic (seeded N(0,1) Q/K/V, seeded context lengths, random block placement)"),
        "config": headline_config(args, w, lens, kvb, flush_l2),
        "pct_of_hbm_peak": round(100 * value / peak, 1),
        "tokens_per_s": round(w.B / (ms_per_step * 1e-3 * w.layers), 1),
        "us_per_layer_step": round(ms_per_step * 1e3, 2),
        "clocks": sampler.summary(t_wall0, t_wall1, t_pre0) if sampler else None,
        "preroll": preroll,
        "e2e": e2e,
        "gpu_launches": 3 * K,
        "timing": "each step (append + decode) replayed from one CUDA graph, CUDA events on the "
                  "launching stream around it; after each step one decode replayed alone from "
                  "its own graph and timed for the roofline",
        "roofline": {"kernel": "pa_decode_" + fmt if fp8 else "pa_decode", "bound": "hbm",
                     "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind
                     if peak_kind == "measured" else "fallback",
                     "traffic": recorded_traffic("pa_decode_%s_llama13b.txt" % fmt if fp8
                                                 else "pa_decode_llama13b.txt")
                     if args.workload == "llama13b" and w.B == 64 else None,
                     "algorithmic_bytes_per_launch": alg,
                     "avg_launch_us": round(dec_avg_ms * 1e3, 2)},
    }
    if "prefix_cache" in w.extra:
        result["prefix_cache"] = w.extra["prefix_cache"]
    if w.prefix_len or "trace" in w.extra:
        ukv = unique_kv_bytes(tbl, lens, w.block_size, w.Hkv, w.d, fp8=fp8)
        unique_roofline(result["roofline"], alg - kvb + ukv, dec_avg_ms, peak)
        result["unique_kv_gbs"] = round(ukv / (ms_per_step * 1e-3) / 1e9, 2)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, host, tbl, lens, args.cpu_seconds, fmt)
    # free the headline's buffers before the sweep
    del host, kc, vc, q, out, ws, kn, vn, g_step, g_decode, flush_buf
    if fp8:
        del ks, vs
    torch.cuda.empty_cache()
    if args.sweep != "none" and not fp8 and args.workload == "llama13b":
        result["sweep"], result["launch_floor"] = run_sweep(args, dev, stream, sampler, peak,
                                                             peak_kind, local)
    # The extras below add figures to the line; a failure in one is recorded in
    # its own object and never costs the headline.
    if args.multi_query == "on" and rank == 0 and not fp8 and args.workload == "llama13b":
        torch.cuda.synchronize()
        try:
            result["multi_query"] = multi_query_summary(measure_multi_query(args, with_cpu=False))
        except Exception as e:   # noqa: BLE001 -- reported, not hidden
            result["multi_query"] = {"error": "%s: %s" % (type(e).__name__, str(e)[:500])}
    if args.kv8 == "on" and rank == 0 and world == 1 and not fp8 and args.workload == "llama13b":
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        result["kv8"] = {}
        for f in ("fp8", "int8"):
            try:
                result["kv8"][f] = kv8_summary(f, args)
            except Exception as e:   # noqa: BLE001 -- reported, not hidden
                result["kv8"][f] = {"error": "%s: %s" % (type(e).__name__, str(e)[:500])}
    if sampler:
        sampler.stop()
    if rank == 0:
        print(json.dumps(result))
    if dist:
        dist.destroy_process_group()


SWEEP = ["gqa7b_1x1024", "gqa7b_8x4096", "gqa7b_8x8192", "gqa7b_16x32768",
         "qwen_longtail_bs8", "qwen_longtail_bs16", "qwen_longtail_bs32",
         "prefix_share", "multiturn_prefix"]


def launch_floor(dev, stream, reps=50, n=32):
    """The launch-latency floor on this machine: a one-element fill kernel (it
    stands for an empty kernel) replayed from a one-node CUDA graph between
    two events, median of `reps`; and per launch inside a graph of `n` such
    kernels."""
    import torch

    x = torch.zeros(1, device=dev)
    g1, gn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=stream):
        x.fill_(1.0)
    with torch.cuda.graph(gn, stream=stream):
        for _ in range(n):
            x.fill_(1.0)
    ts1, tsn = [], []
    with torch.cuda.stream(stream):
        for _ in range(3):
            g1.replay()
            gn.replay()
        for _ in range(reps):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(stream)
            g1.replay()
            e[1].record(stream)
            e[2].record(stream)
            gn.replay()
            e[3].record(stream)
            e[3].synchronize()
            ts1.append(e[0].elapsed_time(e[1]) * 1e3)
            tsn.append(e[2].elapsed_time(e[3]) * 1e3 / n)
    return {"single_graph_replay_us": round(statistics.median(ts1), 2),
            "per_launch_in_graph_us": round(statistics.median(tsn), 2),
            "kernel": "one-element fill (stands for an empty kernel)",
            "how": "median of %d: one-node graph replay between two events; a %d-node graph "
                   "replay / %d" % (reps, n, n)}


def sweep_entry(name, args, dev, stream, sampler, peak, floor):
    """One decode workload of the sweep, timed as a model runs it: one CUDA
    graph holds one layer-step's decode per layer (at least the model's
    layer count), each over its own layer's cache.  Caches are cycled so that
    at least 4x L2 of other layers' KV is read between two reads of one cache
    (the tables, lengths and q are shared by the layers, as a model's are).
    Timed: K graph replays between events after an untimed pre-roll;
    avg_launch_us = replay time / launches.  Context: one launch alone after
    an L2 flush (events around a one-launch graph), and the launch floor."""
    import numpy as np
    import torch

    from paged_kv_cache_103_gb300 import binding

    w = WORKLOADS[name](None)
    alloc, _, tbl, lens, max_blocks, _ = build_tables(w, 0)
    alloc.close()
    B, H, Hkv, d, bs, N = w.B, w.H, w.Hkv, w.d, w.block_size, w.num_blocks
    dt = w.torch_dtype
    pool_bytes = 2 * N * bs * Hkv * d * 2
    n_caches = max(1, int(math.ceil(4 * L2_BYTES / pool_bytes)))
    n_launch = n_caches * int(math.ceil(w.layers / n_caches))
    gen = torch.Generator(device=dev).manual_seed(w.seed)
    kc = torch.randn((n_caches, N, bs, Hkv, d), generator=gen, device=dev, dtype=dt)
    vc = torch.randn((n_caches, N, bs, Hkv, d), generator=gen, device=dev, dtype=dt)
    q = torch.randn((B, H, d), generator=gen, device=dev, dtype=dt)
    out = torch.empty_like(q)
    ws = torch.empty(binding.pa_decode_workspace_size(B, H, d), dtype=torch.uint8, device=dev)
    tbl_d = torch.from_numpy(tbl).to(dev)
    lens_d = torch.from_numpy(lens).to(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        binding.pa_decode_workspace_init(ws, stream)
    max_len = int(lens.max())

    def decode(c):
        binding.pa_decode(q, kc[c], vc[c], tbl_d, lens_d, max_len, w.scale, out, ws, stream)

    g_layers, g_one = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_layers, stream=stream):
        for layer in range(n_launch):
            decode(layer % n_caches)
    with torch.cuda.graph(g_one, stream=stream):
        decode(0)
    K = min(args.steps, 50)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_layers.replay()
    t_pre = time.time()
    pre = preroll_replays(stream, g_layers.replay, args.sweep_preroll_s)
    torch.cuda.synchronize()
    t0 = time.time()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)]
    with torch.cuda.stream(stream):
        for k in range(K):
            ev[2 * k].record(stream)
            g_layers.replay()
            ev[2 * k + 1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    rep_ms = [ev[2 * k].elapsed_time(ev[2 * k + 1]) for k in range(K)]
    clocks = sampler.summary(t0, t1, t_pre) if sampler else None
    # one launch alone, L2 flushed before it (outside the events)
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)]
    with torch.cuda.stream(stream):
        for k in range(K):
            flush.zero_()
            torch.count_nonzero(flush)
            ev1[2 * k].record(stream)
            g_one.replay()
            ev1[2 * k + 1].record(stream)
    torch.cuda.synchronize()
    one_ms = [ev1[2 * k].elapsed_time(ev1[2 * k + 1]) for k in range(K)]
    flags = binding.pa_check_device_errors(stream)
    if flags:
        raise RuntimeError("device error flags 0x%x in sweep entry %s" % (flags, name))
    if not torch.isfinite(out.float()).all():
        raise RuntimeError("non-finite decode output in sweep entry %s" % name)
    avg_ms = sum(rep_ms) / K / n_launch
    kvb = kv_bytes(lens, Hkv, d)
    alg = algorithmic_bytes(lens, B, H, Hkv, d, bs)
    achieved = alg / (avg_ms * 1e-3) / 1e9
    roof = {"kernel": "pa_decode", "bound": "hbm", "achieved": round(achieved, 1),
            "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "algorithmic_bytes_per_launch": alg, "avg_launch_us": round(avg_ms * 1e3, 2),
            "traffic": None}
    entry = {"workload": name + "_decode_layer_step", "batch": B, "q_heads": H, "kv_heads": Hkv,
             "head_dim": d, "block_size": bs, "dtype": w.dtype,
             "context_lens": CONTEXT_MIX[name], "total_context_tokens": int(lens.sum()),
             "kv_gbs": round(kvb / (avg_ms * 1e-3) / 1e9, 1),
             "us_per_layer_step": round(avg_ms * 1e3, 2),
             "tokens_per_s": round(B / (avg_ms * 1e-3 * w.layers), 1),
             "roofline": roof,
             "single_launch_us": round(statistics.median(one_ms) * 1e3, 2),
             "launch_floor_us": floor["single_graph_replay_us"],
             "graph": {"launches": n_launch, "distinct_layer_caches": n_caches,
                       "model_layers": w.layers, "replays_timed": K,
                       "l2": "%.0f MB of other layers' KV read between two reads of one cache"
                             % ((n_caches - 1) * kvb / 1e6) if n_caches > 1 else
                             "one cache of %.2f GB KV (> 4x L2)" % (kvb / 1e9)},
             "preroll": pre, "clocks": clocks, "gpu_launches": K * (n_launch + 1)}
    if w.prefix_len or "trace" in w.extra:
        ukv = unique_kv_bytes(tbl, lens, bs, Hkv, d)
        unique_roofline(roof, alg - kvb + ukv, avg_ms, peak)
        entry["unique_kv_gbs"] = round(ukv / (avg_ms * 1e-3) / 1e9, 1)
    if "prefix_cache" in w.extra:
        entry["prefix_cache"] = w.extra["prefix_cache"]
    del kc, vc, q, out, ws, flush, g_layers, g_one
    torch.cuda.empty_cache()
    return entry


def run_sweep(args, dev, stream, sampler, peak, peak_kind, local):
    """The other decode workloads after the headline, in the same process:
    7B GQA at its four (batch, length) points, the Qwen long tail at block
    size 8 / 16 / 32 and the two prefix-sharing workloads."""
    floor = launch_floor(dev, stream)
    names = SWEEP if args.sweep == "all" else args.sweep.split(",")
    entries = [sweep_entry(n, args, dev, stream, sampler, peak, floor) for n in names]
    return entries, floor


def run_e2e(args, w, host, alloc, kc, vc, ks, vs, stream, max_blocks, fp8, seqs):
    """Real decode steps through the C ABI with host buffers.  Each step is
    pa_step_submit: the host allocator appends one token per sequence
    (pa_append_batch) and exports the tables (pa_export) into a pinned staging
    slot, then one host->device copy of q / new K / new V / slots / tables /
    lengths (the executor's copy-in stream), the executor's CUDA graph of the
    append and the decode, and one device->host copy of the output (its
    copy-out stream); the host waits for each step's output (pa_step_wait).
    Two slots let step k + 1's host work and input copy overlap step k's
    decode; a second loop runs the same steps
    with a wait after every submit (pa_step_run), reported as "synchronous".
    The inputs are written into both pinned slots once (the same synthetic
    rows every step); each step still copies them to the device.
    Copy-on-write cannot arise here: no sequence shares a partial block."""
    import numpy as np
    import torch

    from paged_kv_cache_103_gb300 import binding

    steps = min(args.steps, args.e2e_extra)
    B, H, Hkv, d, bs = w.B, w.H, w.Hkv, w.d, w.block_size
    dt = torch.float16 if w.dtype == "f16" else torch.bfloat16
    step = binding.Step(alloc, B, H, Hkv, d, max_blocks, max_blocks * bs, kc, vc, w.scale,
                        k_scale=ks if fp8 else None, v_scale=vs if fp8 else None, dtype=dt,
                        depth=2, kv_format=args.kv_format if fp8 else "native")
    for i in range(2):
        sl = step.slot(i)
        sl["q"].copy_(host["q"])
        sl["k_new"].copy_(host["k_new"])
        sl["v_new"].copy_(host["v_new"])
    ids = np.asarray(seqs, dtype=np.int64)
    h2d = step.layout["in_bytes"]
    d2h = step.out.numel() * step.out.element_size()

    def kv_of_loop(final):
        # each step appends one token to every sequence: step k of the loop
        # attends to the final lengths minus (steps - 1 - k)
        return sum(kv_bytes(final - (steps - 1 - k), Hkv, d, fp8=fp8) for k in range(steps))

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    prev = None
    for _ in range(steps):
        slot = step.submit(ids, stream)
        if prev is not None:
            step.wait(prev)              # the previous step's output is on the host
        prev = slot
    step.wait(prev)
    t1 = time.perf_counter()
    kv_pipe = kv_of_loop(step.slot(prev)["context_lens"].numpy().astype(np.int64))
    for _ in range(steps):
        step.run(ids, stream)
    t2 = time.perf_counter()
    last = (2 * steps - 1) % 2
    kv_sync = kv_of_loop(step.slot(last)["context_lens"].numpy().astype(np.int64))
    if binding.pa_check_device_errors(stream):
        raise RuntimeError("device error flags set in the e2e leg")
    if not torch.isfinite(step.slot(last)["out"].float()).all():
        raise RuntimeError("non-finite output in the e2e leg")
    step.close()
    return {"value": round(kv_pipe / (t1 - t0) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "ms_per_step": round((t1 - t0) * 1e3 / steps, 4),
            "gpu_launches": 2 * steps,
            "synchronous": {"value": round(kv_sync / (t2 - t1) / 1e9, 2), "unit": "GB/s",
                            "ms_per_step": round((t2 - t1) * 1e3 / steps, 4),
                            "includes": "the same steps with a wait after every submit"},
            "includes": "per step (C ABI) pa_step_submit: host pa_append_batch + pa_export into "
                        "a pinned staging slot, one pinned H2D of q/k_new/v_new/slots/tables/lens "
                        "(copy-in stream), the library's CUDA graph of reshape_and_cache%s and "
                        "decode%s, one D2H of out (copy-out stream); pa_step_wait for every "
                        "step's output (two slots: step k+1's host work and input copy overlap "
                        "step k's decode, step k's output copy overlaps step k+1's)"
                        % (("_" + args.kv_format,) * 2 if fp8 else ("", ""))}


def oracle_sample_run(w, host, tbl, lens, seqs, threads, fmt="native"):
    """Runs the oracle on the sequences `seqs` (cache taken as it stands)."""
    import numpy as np

    import oracle
    from paged_kv_cache_103_gb300 import workloads as wl

    sel = np.asarray(seqs)
    q = wl.bits(host["q"])[sel]
    code = oracle.DTYPE_F16 if w.dtype == "f16" else oracle.DTYPE_BF16
    if fmt != "native":   # the 8-bit oracles run on one thread
        return getattr(oracle, "decode_" + fmt)(q, code, host["k_codes"].numpy(),
                                                host["v_codes"].numpy(), host["k_scale"].numpy(),
                                                host["v_scale"].numpy(), tbl[sel], lens[sel],
                                                w.scale)
    return oracle.decode(q, wl.bits(host["k_cache"]), wl.bits(host["v_cache"]), tbl[sel],
                         lens[sel], w.scale, code, num_threads=threads)


def cpu_baseline(w, host, tbl, lens, seconds, fmt="native"):
    """The oracle on the host cores over a bounded sample of the same batch:
    whole-batch passes repeated until about `seconds` of wall time."""
    fp8 = fmt != "native"
    threads = 1 if fp8 else os.cpu_count() or 1
    seqs = list(range(w.B))
    passes, dt = 0, 0.0
    t0 = time.perf_counter()
    while passes == 0 or dt < seconds:
        oracle_sample_run(w, host, tbl, lens, seqs, threads, fmt)
        passes += 1
        dt = time.perf_counter() - t0
    kvb = passes * kv_bytes(lens, w.Hkv, w.d, fp8=fp8)
    out = {"value": round(kvb / dt / 1e9, 4), "unit": "GB/s", "cores": min(threads, w.B),
           "kind": "oracle", "seconds": round(dt, 2),
           "sample": "%d passes over the whole %d-sequence batch (%d context tokens each), "
                     "fp64 C oracle on %d threads" % (passes, w.B, int(lens.sum()),
                                                     min(threads, w.B))}
    if threads > 1:
        # the same oracle on one thread, over the first sequences for about a
        # fifth of the time
        n1, done, t1 = 0, 0, time.perf_counter()
        while n1 < w.B and (n1 == 0 or time.perf_counter() - t1 < seconds / 5):
            oracle_sample_run(w, host, tbl, lens, [n1], 1, fmt)
            done += int(lens[n1])
            n1 += 1
        dt1 = time.perf_counter() - t1
        b1 = kv_bytes(lens[:n1], w.Hkv, w.d, fp8=fp8)
        out["single_thread"] = {"value": round(b1 / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                                "sample": "the first %d sequences (%d context tokens)" % (n1, done)}
    return out


def run_reference(args):
    """The reference arm: the fp64 oracle as it stands, on the host cores."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    oracle.build()
    from paged_kv_cache_103_gb300 import workloads as wl
    import numpy as np

    w = WORKLOADS[args.workload](args.batch)
    grow_pool_for_e2e(w, args.e2e_extra)     # the GPU arm's pool (spare blocks at the back)
    fmt = args.kv_format
    fp8 = fmt != "native"                 # an 8-bit cache: E4M3 or INT8 codes
    host = wl.qkv(w, with_cache=not fp8)
    if fp8:
        host.update(wl.fp8_cache(w) if fmt == "fp8" else wl.int8_cache(w))
    m = oracle.BlockManagerModel(w.num_blocks, w.block_size, w.free_order)
    if w.prefix_len:
        m.allocate(0, w.prefix_len)
        for s in range(1, w.B):
            m.fork(0, s)
        for s in range(w.B):
            for _ in range(int(w.context_lens[s]) - 1 - w.prefix_len):
                m.append_slot(s)
    else:
        for i in range(w.B):
            m.allocate(i, int(w.context_lens[i]) - 1)
    slots, _ = m.append_batch(range(w.B))
    if fp8:
        getattr(oracle, "reshape_and_cache_" + fmt)(
            host["k_new"], host["v_new"], slots, host["k_codes"].numpy(), host["v_codes"].numpy(),
            host["k_scale"].numpy(), host["v_scale"].numpy())
    else:
        oracle.reshape_and_cache(host["k_new"], host["v_new"], slots, host["k_cache"],
                                 host["v_cache"])
    tbl, lens = m.export(range(w.B))
    threads = 1 if fp8 else os.cpu_count() or 1   # the 8-bit oracles run on one thread
    # each step: a bounded sample of sequences, sized so that the whole run takes
    # about two minutes (and a step at most `ref_step_seconds`)
    per_step = min(args.ref_step_seconds, 120.0 / max(1, args.steps + args.warmup))
    t0 = time.perf_counter()
    oracle_sample_run(w, host, tbl, lens, [0], 1, fmt)
    one = max(time.perf_counter() - t0, 1e-4)   # one sequence on one thread
    k = int(max(1, min(w.B, min(threads, w.B) * per_step / one)))
    seqs = list(range(k))
    for _ in range(args.warmup):
        oracle_sample_run(w, host, tbl, lens, seqs[:1], threads, fmt)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_run(w, host, tbl, lens, seqs, threads, fmt)
    dt = (time.perf_counter() - t0) / args.steps
    value = kv_bytes(lens[:k], w.Hkv, w.d, fp8=fp8) / dt / 1e9
    kvb_all = kv_bytes(lens, w.Hkv, w.d, fp8=fp8)
    used = min(threads, k)
    sample = ("first %d of %d sequences of the batch per step (%d context tokens), all heads, "
              "fp64 C oracle%s on %d threads" % (k, w.B, int(lens[:k].sum()),
                                                 " over the %s cache" % fmt if fp8 else "", used))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) Q/K/V, seeded context lengths, random block placement)",
        "config": headline_config(args, w, lens, kvb_all, kvb_all < 2 * L2_BYTES),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": used,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0, "roofline": None, "clocks": None,   # the oracle runs on the host
    }))


def run_swap(args):
    """Swap bandwidth: one pa_swap_blocks launch moves the blocks of 16 of the
    llama13b batch's sequences (all 8 layers' K and V: 16 pools) from the
    device pools to a pinned host pool, and another moves them back; each is
    timed with CUDA events over repeated launches (the copies are idempotent).
    Baselines on the same box: one cudaMemcpyAsync of a contiguous buffer of
    the same bytes (the copy engines' rate over the host link) and one
    cudaMemcpyAsync per block and pool."""
    import numpy as np
    import torch

    from paged_kv_cache_103_gb300 import binding
    from paged_kv_cache_103_gb300 import build as pa_build

    pa_build.build()
    binding.load()
    w = wl_mod().llama13b()
    layers, nseq = 8, 16
    alloc = binding.Allocator(w.num_blocks, w.block_size, w.free_order)
    for i in range(w.B):
        alloc.alloc(i, int(w.context_lens[i]))
    blocks = sum(alloc.seq_info(i)[1] for i in range(nseq))
    alloc.set_swap_pool(blocks)
    pairs = np.concatenate([alloc.swap_out(i) for i in range(nseq)])
    dev = torch.device("cuda")
    shape = (w.num_blocks, w.block_size, w.Hkv, w.d)
    pools = [torch.empty(shape, dtype=torch.float16, device=dev).normal_()
             for _ in range(2 * layers)]
    host = [torch.empty((blocks,) + shape[1:], dtype=torch.float16).pin_memory()
            for _ in range(2 * layers)]
    out_pairs = torch.from_numpy(pairs.astype(np.int32)).to(dev)
    in_pairs = torch.from_numpy(pairs[:, ::-1].copy().astype(np.int32)).to(dev)
    block_bytes = pools[0][0].numel() * 2
    moved = blocks * block_bytes * 2 * layers

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    reps = max(3, min(args.steps, 20))
    t_out = timed(lambda: binding.pa_swap_blocks(pools, host, out_pairs), reps)
    t_in = timed(lambda: binding.pa_swap_blocks(host, pools, in_pairs), reps)
    flags = binding.pa_check_device_errors()
    if flags:
        raise RuntimeError("device error flags 0x%x" % flags)
    # bit check of one pool after the round trip
    src_idx = torch.from_numpy(pairs[:, 0].astype(np.int64)).to(dev)
    ok = torch.equal(host[0].to(dev), pools[0][src_idx])
    flat_d = torch.empty(moved // 2, dtype=torch.float16, device=dev)
    flat_h = torch.empty(moved // 2, dtype=torch.float16).pin_memory()
    t_cd2h = timed(lambda: flat_h.copy_(flat_d, non_blocking=True), reps)
    t_ch2d = timed(lambda: flat_d.copy_(flat_h, non_blocking=True), reps)
    sub = pairs[: max(1, len(pairs) // 8)]          # per-block copies: an eighth of the blocks

    def per_block():
        for p, h in zip(pools, host):
            for s, d in sub:
                h[int(d)].copy_(p[int(s)], non_blocking=True)
    t_pb = timed(per_block, 2) * 8
    gbs = lambda t: round(moved / (t * 1e-3) / 1e9, 1)
    print(json.dumps({
        "metric": "KV swap GB/s (device->host; host->device in h2d)", "value": gbs(t_out),
        "unit": "GB/s", "n_gpus": 1, "steps": reps, "warmup": 3, "ms_per_step": round(t_out, 4),
        "higher_is_better": True, "dtype": "f16 (bit copies)", "data": "synthetic",
        "h2d": {"value": gbs(t_in), "ms": round(t_in, 4)},
        "bit_exact_round_trip": bool(ok),
        "contiguous_memcpy": {"d2h": gbs(t_cd2h), "h2d": gbs(t_ch2d),
                              "note": "one cudaMemcpyAsync of the same bytes, pinned host"},
        "per_block_memcpy": {"d2h": gbs(t_pb),
                             "note": "one cudaMemcpyAsync per block and pool (scaled from 1/8)"},
        "roofline": {"bound": "host link", "achieved": gbs(t_out), "peak": gbs(t_cd2h),
                     "unit": "GB/s", "frac": round(t_cd2h / t_out, 3),
                     "peak_source": "contiguous cudaMemcpyAsync device->pinned host, same run"},
        "gpu_launches": 2 * reps,
        "config": {"workload": "swap of 16 llama13b sequences x 8 layers (K and V)",
                   "blocks": int(blocks), "pools": 2 * layers, "block_bytes": int(block_bytes),
                   "bytes_per_direction": int(moved)}}))


def load_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def run_multi_query(args):
    print(json.dumps(measure_multi_query(args, with_cpu=not args.no_cpu_baseline)))


def kv8_summary(fmt, args):
    """The same llama13b decode step over an 8-bit cache (E4M3 or INT8 codes
    and fp32 scales), timed by a child run of this bench (its own pre-roll,
    clock record and traffic figure); the figures the decode line carries."""
    steps = max(20, min(args.steps, 500))
    cmd = [sys.executable, os.path.abspath(__file__), "--kv-format", fmt, "--sweep", "none",
           "--multi-query", "off", "--kv8", "off", "--no-cpu-baseline",
           "--steps", str(steps), "--warmup", str(max(3, args.warmup))]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, timeout=900)
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode != 0 or not lines:
        raise RuntimeError("the %s decode run failed:\n%s" % (fmt, r.stderr[-2000:]))
    d = json.loads(lines[-1])
    rf = d["roofline"]
    return {"kernel": rf["kernel"], "value": d["value"], "unit": d["unit"],
            "pct_of_hbm_peak": d["pct_of_hbm_peak"], "ms_per_step": d["ms_per_step"],
            "steps": d["steps"],
            "roofline": {k: rf.get(k) for k in ("achieved", "peak", "frac", "traffic",
                                                "algorithmic_bytes_per_launch", "avg_launch_us")},
            "e2e": {"value": d["e2e"]["value"], "unit": d["e2e"]["unit"]},
            "clocks": d.get("clocks"), "config": d["config"],
            "how": "bench.py --kv-format %s --sweep none --steps %d, a child process" % (fmt, steps)}


def multi_query_summary(mq):
    """The figures of a measure_multi_query result that the decode line
    carries: each kernel's rate, roofline fraction and time per launch."""
    sv = mq["speculative_verification"]
    return {
        "chunked_prefill": {
            "kernel": mq["roofline"]["kernel"], "value": mq["value"], "unit": mq["unit"],
            "frac": mq["roofline"]["frac"], "peak": mq["roofline"]["peak"],
            "us_per_launch": mq["roofline"]["avg_launch_us"],
            "mma_sync_kernel": {k: mq["roofline"]["mma_sync_kernel"][k]
                                for k in ("kernel", "value", "unit", "us_per_launch")},
            "workload": mq["config"]["workload"]},
        "speculative_verification": {
            "kernel": "pa_multi_query_tc", "value": sv["value"], "unit": sv["unit"],
            "frac": round(sv["pct_of_hbm_peak"] / 100.0, 4), "us_per_launch": sv["us_per_launch"],
            "mma_sync_kernel": {k: sv["mma_sync_kernel"][k]
                                for k in ("kernel", "value", "us_per_launch")},
            "workload": sv["config"]},
        "how": "bench.py --measure multi_query, run after the decode sweep in the same process",
    }


def measure_multi_query(args, with_cpu=True):
    """pa_multi_query on two shapes: a chunked prefill (4 sequences, a
    2048-token chunk each on top of 6144 cached tokens, 7B GQA 32 / 8 heads,
    bf16) timed against the tensor roofline, and speculative verification (the
    Qwen long-tail batch of 128 sequences, 6 query tokens each) timed against
    the HBM roofline.  CUDA events over repeated launches on one stream."""
    import numpy as np
    import torch

    from paged_kv_cache_103_gb300 import binding
    from paged_kv_cache_103_gb300 import build as pa_build

    pa_build.build()
    binding.load()
    dev = torch.device("cuda")

    def make(lens, qlens, H, Hkv, d, bs, seed):
        N = int(math.ceil(1.25 * sum(math.ceil(n / bs) for n in lens))) + 2
        alloc = binding.Allocator(N, bs, np.random.default_rng(seed).permutation(N).astype(np.int32))
        for i, n in enumerate(lens):
            alloc.alloc(i, int(n))
        mb = max(math.ceil(n / bs) for n in lens)
        tbl, ln = alloc.export(list(range(len(lens))), mb)
        qs = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
        g = torch.Generator(device=dev).manual_seed(seed)
        kc = torch.randn(N, bs, Hkv, d, generator=g, device=dev).to(torch.bfloat16)
        vc = torch.randn(N, bs, Hkv, d, generator=g, device=dev).to(torch.bfloat16)
        q = torch.randn(int(qs[-1]), H, d, generator=g, device=dev).to(torch.bfloat16)
        out = torch.empty_like(q)
        ws = torch.empty(binding.pa_multi_query_workspace_size(len(lens), H, Hkv, d,
                                                                int(max(qlens))),
                         dtype=torch.uint8, device=dev)
        binding.pa_decode_workspace_init(ws)
        ws_tc = torch.empty(binding.pa_multi_query_tc_workspace_size(len(lens), H, Hkv, d),
                            dtype=torch.uint8, device=dev)
        binding.pa_decode_workspace_init(ws_tc)
        return dict(kc=kc, vc=vc, q=q, out=out, ws=ws, ws_tc=ws_tc,
                    tbl=torch.from_numpy(tbl).to(dev),
                    ln=torch.from_numpy(ln).to(dev), qs=torch.from_numpy(qs).to(dev),
                    lens=np.asarray(lens), qlens=np.asarray(qlens), H=H, Hkv=Hkv, d=d,
                    maxq=int(max(qlens)))

    def time_it(c, reps, flush=None, tc=False):
        def run():
            if tc:
                binding.pa_multi_query_tc(c["q"], c["qs"], c["kc"], c["vc"], c["tbl"], c["ln"],
                                          c["maxq"], 1 / math.sqrt(c["d"]), c["out"], c["ws_tc"])
            else:
                binding.pa_multi_query(c["q"], c["qs"], c["kc"], c["vc"], c["tbl"], c["ln"],
                                       c["maxq"], 1 / math.sqrt(c["d"]), c["out"], c["ws"])
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            if flush is not None:
                flush.zero_()
                torch.count_nonzero(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        if binding.pa_check_device_errors():
            raise RuntimeError("device error flags set")
        return sorted(ts)[len(ts) // 2]

    reps = max(5, min(args.steps, 50))
    # chunked prefill
    pf = make([8192] * 4, [2048] * 4, 32, 8, 128, 16, 31)
    t_pf_legacy = time_it(pf, reps)
    out_legacy = pf["out"].clone()
    t_pf = time_it(pf, reps, tc=True)
    agree = float((pf["out"].float() - out_legacy.float()).abs().max())
    keys = sum(sum(n - ql + r + 1 for r in range(ql)) for n, ql in zip(pf["lens"], pf["qlens"]))
    flops = 4.0 * pf["H"] * pf["d"] * keys
    tflops = flops / (t_pf * 1e-3) / 1e12
    tflops_legacy = flops / (t_pf_legacy * 1e-3) / 1e12
    peak_t, peak_kind = load_tensor_peak()
    # the ceiling of the mma.sync m16n8k16 path itself (bf16), same process
    sink = torch.empty(binding.pa_decode_grid_size() * 4 * 256, dtype=torch.float32, device=dev)
    for _ in range(3):
        binding.pa_measure_mma_ceiling(True, 4096, sink)
    torch.cuda.synchronize()
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    m0.record()
    mma_flops = sum(binding.pa_measure_mma_ceiling(True, 4096, sink) for _ in range(5))
    m1.record()
    torch.cuda.synchronize()
    mma_ceiling = mma_flops / (m0.elapsed_time(m1) * 1e-3) / 1e12
    # speculative verification
    w = wl_mod().qwen_longtail(16)
    lens = (np.asarray(w.context_lens, np.int64) + 6).tolist()
    sv = make(lens, [6] * w.B, w.H, w.Hkv, w.d, 16, 32)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    t_sv_legacy = time_it(sv, reps, flush)
    sv_legacy = sv["out"].clone()
    t_sv = time_it(sv, reps, flush, tc=True)
    sv_agree = float((sv["out"].float() - sv_legacy.float()).abs().max())
    kv = kv_bytes(lens, w.Hkv, w.d)
    gbs = kv / (t_sv * 1e-3) / 1e9
    gbs_legacy = kv / (t_sv_legacy * 1e-3) / 1e9
    peak_h, _ = load_peak()
    # the oracle on the host cores: 256 query rows of the first prefill sequence (each over its
    # full causal context), same tables and cache contents
    cpu = None
    if with_cpu:
        import oracle
        oracle.build()
        threads = os.cpu_count() or 1
        rows = 256
        qs0 = np.array([0, rows], np.int32)
        qh = pf["q"][:rows].cpu()
        n0 = int(pf["lens"][0])
        q_off = n0 - int(pf["qlens"][0])            # these are the chunk's first rows
        kh_, vh_ = pf["kc"].cpu(), pf["vc"].cpu()
        tbl0 = pf["tbl"][:1].cpu().numpy()
        t0 = time.perf_counter()
        oracle.multi_query(wl_mod().bits(qh), qs0, wl_mod().bits(kh_), wl_mod().bits(vh_), tbl0,
                           np.array([q_off + rows], np.int32), 1 / math.sqrt(pf["d"]),
                           oracle.DTYPE_BF16, num_threads=threads)
        dt = time.perf_counter() - t0
        cflops = 4.0 * pf["H"] * pf["d"] * sum(q_off + r + 1 for r in range(rows))
        cpu = {"value": round(cflops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads,
               "kind": "oracle", "seconds": round(dt, 2),
               "sample": "%d query rows of one 2048-token prefill chunk (each over its %d+ "
                         "causal keys), fp64 C oracle" % (rows, q_off + 1)}
    return ({
        "metric": "multi-query paged attention: TFLOP/s (chunked prefill), KV GB/s "
                  "(speculative verification)",
        "cpu_baseline": cpu,
        "value": round(tflops, 1), "unit": "TFLOP/s", "n_gpus": 1, "steps": reps, "warmup": 3,
        "ms_per_step": round(t_pf, 4), "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic (N(0,1) Q/K/V, random block placement)",
        "roofline": {"kernel": "pa_multi_query_tc", "bound": "tensor",
                     "achieved": round(tflops, 1), "peak": peak_t,
                     "unit": "TFLOP/s", "frac": round(tflops / peak_t, 4),
                     "peak_source": "%s bf16_tflops (cuBLAS burst)" % peak_kind,
                     "flops_per_launch": flops, "avg_launch_us": round(t_pf * 1e3, 2),
                     "note": "tcgen05.mma (M = N = 128, accumulators in TMEM), useful flops only",
                     "mma_sync_kernel": {
                         "kernel": "pa_multi_query", "value": round(tflops_legacy, 1),
                         "unit": "TFLOP/s", "us_per_launch": round(t_pf_legacy * 1e3, 2),
                         "max_abs_diff_vs_tc": agree,
                         "note": "mma.sync m16n8k16 path (a bf16 P's residual product only "
                                 "in warps holding a row of fewer than 256 keys: none here)"},
                     "mma_sync_ceiling": {
                         "value": round(mma_ceiling, 1), "unit": "TFLOP/s",
                         "how": "pa_measure_mma_ceiling: 2 CTAs x 8 warps per SM, 8 independent "
                                "bf16 m16n8k16 MMAs per round from registers, CUDA events over 5 "
                                "launches",
                         "mma_sync_work_frac": round(tflops_legacy / mma_ceiling, 4)}},
        "e2e": None,
        "speculative_verification": {
            "kernel": "pa_multi_query_tc (one query tile per sequence and KV head, key tiles "
                      "split evenly over the CTAs)",
            "value": round(gbs, 1), "unit": "GB/s", "us_per_launch": round(t_sv * 1e3, 2),
            "pct_of_hbm_peak": round(100 * gbs / peak_h, 1), "tokens": 6 * w.B,
            "mma_sync_kernel": {"kernel": "pa_multi_query", "value": round(gbs_legacy, 1),
                                "us_per_launch": round(t_sv_legacy * 1e3, 2),
                                "pct_of_hbm_peak": round(100 * gbs_legacy / peak_h, 1),
                                "max_abs_diff_vs_tc": sv_agree},
            "config": "qwen long-tail batch, 128 sequences x 6 query tokens, 28 / 4 heads, "
                      "block 16, L2 flushed between launches"},
        "gpu_launches": 4 * (reps + 3) + 8,
        "config": {"workload": "chunked prefill: 4 sequences x 2048-token chunk on 6144 cached "
                               "tokens, 32 / 8 heads of 128, bf16, block 16",
                   "causal_keys": int(keys), "us_per_launch": round(t_pf * 1e3, 2)}})


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama13b")
    ap.add_argument("--batch", type=int, default=None, help="batch of the llama13b workload")
    ap.add_argument("--e2e-extra", type=int, default=64,
                    help="e2e steps (each appends a token to every sequence)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-step-seconds", type=float, default=1.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", default="all",
                    help="after the llama13b headline, time these decode workloads too: 'all', "
                         "'none' or a comma-separated list of workload names")
    ap.add_argument("--preroll-s", type=float, default=0.3,
                    help="seconds of untimed step replays right before the timed region")
    ap.add_argument("--sweep-preroll-s", type=float, default=0.1,
                    help="seconds of untimed replays before each sweep entry's timed replays")
    ap.add_argument("--kv-format", choices=["native", "fp8", "int8"], default="native",
                    help="cache in the workload's 16-bit dtype, or E4M3 / INT8 codes + fp32 scales")
    ap.add_argument("--kv8", choices=["on", "off"], default="on",
                    help="after the 16-bit line, time the same decode step over FP8 and INT8 "
                         "caches in child runs and add their figures (llama13b, one GPU)")
    ap.add_argument("--multi-query", choices=["on", "off"], default="on",
                    help="after the sweep, time the chunked prefill and speculative verification "
                         "kernels too and add their figures to the line (llama13b runs only)")
    ap.add_argument("--measure", choices=["decode", "swap", "multi_query"], default="decode",
                    help="swap: device<->host block swap bandwidth; multi_query: chunked prefill "
                         "and speculative verification, instead of the decode step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.measure == "swap":
        run_swap(args)
    elif args.measure == "multi_query":
        run_multi_query(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
