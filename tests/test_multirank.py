"""Multi-rank plumbing of bench.py on CPU (gloo, world size 2).

Tokens shard across GPUs with no data-path collective: each rank runs its own
batches on a replica of the layer, and the only cross-rank step is the
reduction of the timing (the slowest rank's time defines the job's rate).
These tests run that reduction and the reference arm's rank handling on two
CPU processes.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        total = bench.max_over_ranks(times[rank], world)
        out[rank] = (total, bench.job_rate(world, 1024, 10, total))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo_world2():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    times = [31.5, 47.25]  # ms per rank: rank 1 is the slow one
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, times, out), nprocs=2, join=True, start_method="spawn")
    for rank in range(2):
        total, rate = out[rank]
        assert total == pytest.approx(47.25)
        assert rate == pytest.approx(2 * 1024 * 10 / 0.04725)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(12.0, 1) == 12.0
    assert bench.job_rate(1, 8, 50, 1000.0) == pytest.approx(400.0)


def test_reference_arm_runs_on_rank_zero_only():
    import bench

    class Args:
        workload = "tiny"
        steps = 1
        warmup = 0
        gpus = 2

    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(Args(), world=2, rank=1)
    assert buf.getvalue() == ""


@pytest.mark.parametrize("fmt,gains", [("q2", 0), ("mx4", 2), ("vq13", 1)])
def test_reference_arm_prints_the_contract_line(fmt, gains):
    """Rank 0 of the reference arm (the oracle on the host's cores) prints one
    JSON line with the keys the benchmark contract names."""
    import json

    import bench

    class Args:
        workload = "tiny"
        steps = 2
        warmup = 1
        gpus = 1
        routed_format = fmt

    Args.gains = gains
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(Args(), world=1, rank=0)
    lines = buf.getvalue().strip().splitlines()
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["unit"] == bench.UNIT and d["metric"] == bench.METRIC and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny" and ("MXFP4" in d["config"]["weights"]) == (fmt == "mx4")
    assert d["config"].get("down_gain_tables", 0) == gains
