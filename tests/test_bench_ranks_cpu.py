"""bench.py's multi-rank reduction on CPU: two gloo ranks report different step times; both must
see the slower one, and the whole-job throughput counts every rank's work over that time.  (The
forward runs as independent replicas; this reduction is the only multi-rank step.)"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + rank, world, "cpu")
        out[rank] = (ms, bench.whole_job_tflops(1e12, world, ms))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    old = os.environ.get("PYTHONPATH", "")
    os.environ["PYTHONPATH"] = root + (os.pathsep + old if old else "")
    try:
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
    finally:
        os.environ["PYTHONPATH"] = old
    for r in range(2):
        ms, value = out[r]
        assert ms == pytest.approx(2.0)
        assert value == pytest.approx(2 * 1e12 / 2e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_tflops(4e12, 1, 2.0) == pytest.approx(2000.0)
