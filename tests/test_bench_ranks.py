"""The benchmark's multi-rank logic on CPU with gloo (world size 2): the timed
region is the maximum over ranks, and the reference arm runs and prints on
rank 0 only."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        buf = io.StringIO()

        class Args:
            steps, warmup, cpu_seconds, gpus = 1, 0, 0.05, world
        if rank != 0:                    # rank 0's reference run is heavy; only the silent ranks are checked
            with contextlib.redirect_stdout(buf):
                bench.run_reference(Args, world, rank)
        out[rank] = (got, buf.getvalue())
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_silent_reference_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert res[0][0] == 15.0 and res[1][0] == 15.0
    assert res[1][1] == ""


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5


def test_clock_sampler_reports_its_source():
    """The clock sampler takes NVML when the driver library answers and falls
    back to nvidia-smi otherwise; either way stop() returns a record that says
    which source it used and keeps only samples inside the given window."""
    sys.path.insert(0, ROOT)
    import time
    import bench
    c = bench.clock_sampler("00000000:00:00.0")
    c.start()
    t0 = time.time()
    time.sleep(0.05)
    t1 = time.time()
    rec = c.stop(t0, t1)
    assert isinstance(rec, dict) and "reasons" in rec
    if isinstance(c, bench.NvmlClockSampler):
        assert rec["source"] == "nvml" and rec["samples"] >= 1
    else:
        assert getattr(c, "nvml_error", None)          # why NVML was not used
