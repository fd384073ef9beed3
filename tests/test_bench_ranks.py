"""The bench's multi-rank host logic on CPU: two gloo ranks (replicas) agree
on the slowest rank's time and report the whole job's rate."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
        out[rank] = (ms, bench.whole_job_rate(1000, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] == pytest.approx(2 * 1000 / 15e-3)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, None, None) == 3.5
    assert bench.whole_job_rate(100, 1, 2.0) == pytest.approx(50000.0)


def test_reference_arm_under_two_ranks_prints_one_line():
    """`bench.py --impl reference` launched as two ranks: rank 0 alone times
    the oracle and prints the one JSON line; rank 1 exits 0 without work."""
    import json
    import subprocess
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--workload", "gqa7b_1x1024", "--ref-step-seconds", "0.2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle"
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["value"] == out["value"]


def test_e2e_appends_fit_the_grown_pool():
    """For every workload built on a fresh allocator, the bench's pool growth
    leaves the batch's tables as the workload has them and holds the e2e
    leg's two loops of appended tokens (the default 64 each)."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_cache_103_gb300 import binding
    extra = 64
    for name, make in sorted(bench.WORKLOADS.items()):
        w = make(None)
        if "trace" in w.extra:
            continue
        plain = binding.Allocator(w.num_blocks, w.block_size, w.free_order)
        bench.populate(plain, w)
        bench.grow_pool_for_e2e(w, extra)
        alloc = binding.Allocator(w.num_blocks, w.block_size, w.free_order)
        bench.populate(alloc, w)
        seqs = list(range(w.B))
        width = int(np.ceil((w.context_lens.max() + 2 * extra + 1) / w.block_size)) + 1
        assert np.array_equal(plain.export(seqs, width)[0], alloc.export(seqs, width)[0]), name
        for _ in range(2 * extra + 1):
            alloc.append_batch(seqs)


def test_multi_query_summary_keeps_each_kernels_figures():
    """The decode line's multi-query object carries, for each shape, the
    tcgen05 kernel's rate, fraction and time and the mma.sync kernel's beside
    it, taken unchanged from the multi-query measurement."""
    sys.path.insert(0, ROOT)
    import bench
    mq = {"value": 940.0, "unit": "TFLOP/s",
          "roofline": {"kernel": "pa_multi_query_tc", "frac": 0.5, "peak": 1880.0,
                       "avg_launch_us": 1020.0,
                       "mma_sync_kernel": {"kernel": "pa_multi_query", "value": 220.0,
                                           "unit": "TFLOP/s", "us_per_launch": 4300.0,
                                           "note": "dropped"}},
          "config": {"workload": "prefill shape"},
          "speculative_verification": {"value": 4600.0, "unit": "GB/s", "pct_of_hbm_peak": 68.1,
                                       "us_per_launch": 170.0, "config": "verify shape",
                                       "mma_sync_kernel": {"kernel": "pa_multi_query",
                                                           "value": 3400.0, "us_per_launch": 230.0,
                                                           "pct_of_hbm_peak": 50.0}}}
    s = bench.multi_query_summary(mq)
    pf, sv = s["chunked_prefill"], s["speculative_verification"]
    assert (pf["value"], pf["frac"], pf["us_per_launch"], pf["workload"]) == \
        (940.0, 0.5, 1020.0, "prefill shape")
    assert pf["mma_sync_kernel"] == {"kernel": "pa_multi_query", "value": 220.0,
                                     "unit": "TFLOP/s", "us_per_launch": 4300.0}
    assert (sv["value"], sv["frac"], sv["us_per_launch"], sv["workload"]) == \
        (4600.0, 0.681, 170.0, "verify shape")
    assert sv["mma_sync_kernel"]["us_per_launch"] == 230.0
