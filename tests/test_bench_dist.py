"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the timed
region's max over ranks and the whole-job value."""
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


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [3.0, 5.5][rank]
    m = bench.max_over_ranks(local_ms, world, "cpu")
    dist.barrier()
    q.put((rank, m, bench.whole_job_gbs(1_000_000_000, world, m)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in got:
        assert m == 5.5, "every rank must see the slowest rank's time"
        assert v == pytest.approx(2 * 1e9 / 5.5e-3 / 1e9)


def test_single_rank_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.whole_job_gbs(4_000_000_000, 1, 1.0) == pytest.approx(4000.0)
