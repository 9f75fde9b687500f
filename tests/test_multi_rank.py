"""The benchmark's multi-rank path on CPU (gloo, world size 2): every rank runs its own
batch (the (layer, batch, head) slices are independent, no collective on the data path);
the job's time is the slowest rank's, and its throughput all ranks' units over that time.
The reference arm prints on rank 0 only."""
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


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]  # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, world, torch.device("cpu"))
    rate = bench.job_rate(1000.0, world, worst)
    out.put((rank, worst, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, rate in got:
        assert worst == 5.0                      # every rank sees the slowest time
        assert rate == pytest.approx(2 * 1000.0 / 5e-3)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.0, 1, torch.device("cpu")) == 4.0
    assert bench.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    import fibattn_inputs as fi

    class A:
        steps, warmup, workload = 1, 3, "c1"
    assert bench.run_reference(A(), fi.WORKLOADS["c1"], 2, 1) is None
