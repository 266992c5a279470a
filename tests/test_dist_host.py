"""The multi-rank host logic of bench.py on CPU: world-size-2 gloo ranks.

Decode sequences are independent, so N GPUs run N replicas of the per-GPU
workload (weak scaling) with no collective on the data path; the only
cross-rank steps are the barriers around the timed region and the max of the
ranks' times.  These tests run that logic with gloo on the host (no GPU).
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        local_ms = 10.0 * (rank + 1)          # rank 1 is the slowest
        value, ms = bench.job_throughput(world, 8, local_ms)
        m = bench.max_over_ranks(world, float(rank) - 5.0)
        bench.barrier(world)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"value": value, "ms": ms, "max": m}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        # 8 tokens per rank, 2 ranks, slowest rank took 20 ms
        assert r["ms"] == pytest.approx(20.0)
        assert r["value"] == pytest.approx(16 / 0.020)
        assert r["max"] == pytest.approx(-4.0)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.job_throughput(1, 8, 4.0)
    assert ms == 4.0 and value == pytest.approx(2000.0)


def test_reference_arm_prints_on_rank_zero_only():
    """Under torchrun only rank 0 runs the oracle sample and prints the line;
    the other ranks return at once without work."""
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup, gpus, workload, batch, context = 1, 0, 2, "hybrid_decode_1m", 0, 0
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A(), 2, 1)
    assert buf.getvalue() == ""


def test_reference_arm_line_on_rank_zero():
    """Rank 0 times the oracle on a bounded sample and prints one JSON line
    with the reference arm's keys: impl, the bench's metric and unit, a
    cpu_baseline describing this run, and an e2e object with no host copies."""
    import json
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup, gpus, workload, batch, context = 1, 0, 1, "hybrid_decode_1m", 0, 1 << 16
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A(), 1, 0, budget_s=2.0)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] == 1 and d["cpu_baseline"]["host"]["nproc"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["steps"] == 1 and d["dtype"] == "f64"
