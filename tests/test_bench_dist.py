"""The multi-rank host logic of bench.py with two gloo ranks on the CPU:
process-group set-up from the torchrun environment, barrier, the max over
ranks of the timed region, the whole-job (weak-scaled) throughput, and the
reference arm's rule that only rank 0 works and prints."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(ws),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    got_ws, got_rank, _ = bench.dist_setup(None, backend="gloo")
    bench.barrier(got_ws)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, got_ws)   # this rank's "ms"
    ref = bench.run_reference(type("A", (), dict(warmup=0, steps=1))())
    bench.barrier(got_ws)
    q.put((got_rank, got_ws, slowest, ref is None))
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(ws))
    assert [r[0] for r in res] == [0, 1] and all(r[1] == ws for r in res)
    assert all(r[2] == 15.0 for r in res)          # every rank sees the slowest rank's time
    assert res[0][3] is False and res[1][3] is True  # reference arm: rank 0 only


def test_job_throughput_is_weak_scaled():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_throughput(1, 1e12, 1.0)
    assert one == pytest.approx(1000.0)
    assert bench.job_throughput(4, 1e12, 1.0) == pytest.approx(4 * one)
