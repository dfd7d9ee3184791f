"""The multi-GPU path is replicas: each rank runs its own streams, the bench line sums the
stream-steps of all ranks over the slowest rank's time.  Checked with two gloo ranks on CPU."""
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    # rank 1 is slower and ran more streams
    job = bench.aggregate(10.0 * (rank + 1), 100 * (2 * rank + 1), world, "cpu")
    results.put((rank, job))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_sum_stream_steps_over_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(results.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert got[r]["ms"] == 20.0
        assert got[r]["stream_steps"] == 400.0
        assert got[r]["value"] == pytest.approx(400.0 / 0.020)


def test_single_rank_is_its_own_job():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    job = bench.aggregate(5.0, 64, 1)
    assert job == {"ms": 5.0, "stream_steps": 64.0, "value": 64.0 / 0.005}
