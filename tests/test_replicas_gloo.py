"""Host logic of `bench.py --gpus N` (replicas only: no collective on the data
path): the step time is the maximum over ranks and the whole-job value counts
every replica's bytes.  Two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(1.0 + rank * 0.25)  # rank 1 is the slower replica
        q.put((rank, ms, bench.job_gbs(world, 1e9, ms)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_time_and_job_throughput():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, gbs in out:
        assert ms == pytest.approx(1.25)           # the slowest replica
        assert gbs == pytest.approx(2 * 1e9 / 1.25e-3 / 1e9)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_gbs(1, 2e9, 2.0) == pytest.approx(1000.0)
