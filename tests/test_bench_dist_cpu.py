"""The replicas path of bench.py (one process per GPU, no data exchange): its
max-over-ranks timing and whole-job throughput, run as two gloo ranks on CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 1.0 + rank                          # rank 1 is the slow one
        ms_all = bench.max_over_ranks(ms, world, "cpu")
        value = bench.job_gbps(1e6, ms_all, world)
        out.put((rank, ms_all, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest time; throughput = 2 ranks x 1e6 bytes / 2 ms
    assert [g[1] for g in got] == [2.0, 2.0]
    assert got[0][2] == pytest.approx(2 * 1e6 / 2e-3 / 1e9)
