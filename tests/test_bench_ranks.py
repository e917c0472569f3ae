"""The benchmark's multi-rank timing on CPU (gloo, world size 2): a barrier, the max of the ranks' times, and
whole-job throughput (each rank's slice is one workload, so the job processes world_size workloads a step).
The slices' shared skip decision is tested in test_sliced_ranks.py."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier()
    local_ms = [3.0, 5.0][rank]
    ms = bench.max_over_ranks(local_ms, "cpu")
    value = bench.job_throughput(123_568_896, world, ms)
    ws, r, _ = bench.dist_env()
    out.put((rank, ms, value, ws, r))
    bench.barrier()
    tdist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ms, value, ws, r in res:
        assert ms == 5.0                       # the max over ranks
        assert ws == 2 and r == rank
        assert value == pytest.approx(2 * 123_568_896 / 5e-3 / 1e9)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, "cpu") == 7.5
    assert bench.job_throughput(10 ** 9, 1, 1000.0) == pytest.approx(1.0)


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    import synth
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, cpu_sample, gpus, sum = 1, 0, 1 << 12, 2, "compensated"
    assert bench.reference_main(A, synth.WORKLOADS["tiny"]) == 0
    assert capsys.readouterr().out == ""
