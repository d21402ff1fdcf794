"""The multi-rank path of the benchmark on CPU: two gloo ranks on 127.0.0.1.

The fit shards by rows with no exchange, so N GPUs run N replicas of the
workload; what the ranks share is the step time (the slowest rank's) and the
whole-job throughput.  The reference arm runs on rank 0 only.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        m = bench.cross_rank_max(times[rank], torch.device("cpu"))
        v = bench.job_value(1000, world, m)
        with open(os.path.join(outdir, f"r{rank}.txt"), "w") as f:
            f.write(f"{m!r} {v!r}\n")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_share_the_slowest_step(tmp_path):
    times = [1.5, 4.0]
    mp.start_processes(_worker, args=(2, _free_port(), times, str(tmp_path)), nprocs=2,
                       join=True, start_method="spawn")
    got = [open(tmp_path / f"r{r}.txt").read().split() for r in range(2)]
    for m, v in got:
        assert float(m) == 4.0
        assert float(v) == pytest.approx(2 * 1000 / 4.0e-3)


def test_single_process_needs_no_group():
    import bench
    assert bench.cross_rank_max(2.5, torch.device("cpu")) == 2.5
    assert bench.job_value(10, 1, 1.0) == pytest.approx(1e4)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        gpus, steps, warmup = 2, 1, 3
    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""
