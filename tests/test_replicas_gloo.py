"""The N>1 bench path on CPU: replicas only, one process per rank, gloo.

The det_gemm path does not shard (each launch is one GPU's work; tensor
parallel GEMM is out of scope on the det_gemm page, section "Scope"), so
`bench.py --gpus N` runs N independent replicas. What the ranks share is
the timing protocol: a barrier around the timed region, the slowest rank's
time, and whole-job throughput = every rank's work over that time. These
tests run that protocol on two CPU processes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ranks(rank, ws, port, times, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench.dist_env() == (ws, rank, rank)
        dist.barrier()
        slowest = bench.max_over_ranks(times[rank], ws, torch.device("cpu"))
        value = bench.whole_job_tflops(1e12, ws, slowest)
        out.put((rank, slowest, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [2.0, 5.0]                    # ms per step on rank 0 and rank 1
    port = free_port()
    procs = [ctx.Process(target=_ranks, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 5.0                          # max over ranks, on every rank
        assert value == pytest.approx(2 * 1e12 / 5e-3 / 1e12)   # 400 TFLOP/s for the job


def test_single_rank_protocol_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.whole_job_tflops(2e12, 1, 4.0) == pytest.approx(500.0)


def test_reference_arm_does_no_work_on_other_ranks(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup = 1, 0
    bench.reference_arm(Args())
    assert capsys.readouterr().out == ""
