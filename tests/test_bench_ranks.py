"""bench.py's multi-rank bookkeeping on the host: replicas under torchrun (gloo, 2 ranks, CPU).

The layer needs no exchange between GPUs, so N > 1 runs N independent replicas; the only
cross-rank steps are the barrier, the max of the ranks' times and rank 0 printing the line.
"""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        worst = bench.max_over_ranks(times[rank], dist, "cpu")
        value = bench.job_tflops(world, 2.0e12, 10, worst)
        dist.barrier()
        out.put((rank, worst, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    import torch.multiprocessing as mp

    world, port = 2, _free_port()
    times = [12.5, 20.0]  # ms over the timed steps, per rank
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest rank's time; the job value counts both replicas' work over it
    for rank, worst, value in res:
        assert worst == 20.0
        assert value == pytest.approx(2 * 2.0e12 * 10 / 20.0e-3 / 1e12)


def test_single_rank_without_process_group():
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.job_tflops(1, 1e12, 4, 2.0) == pytest.approx(2000.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    # under torchrun only rank 0 runs and prints the oracle arm; the others return 0 at once
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, gpus = 2, 3, 2

    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    # rank 0 prints one JSON line with the contract's keys (a bounded oracle sample per step)
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setattr(bench, "oracle_sample", lambda max_rows_per_m=None: (None, None))
    monkeypatch.setattr(bench, "time_oracle", lambda data, xs, ms: (0.5, 1.0e9))

    class A:
        steps, warmup, gpus = 2, 3, 1

    assert bench.run_reference(A()) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["higher_is_better"]
    assert line["value"] == pytest.approx(1.0e9 * 2 / 1.0 / 1e12)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
