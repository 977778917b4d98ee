"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): each rank
reports its own step time, the job takes the slowest, and the job rate counts
every rank's bytes. No GPU is involved."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, world, rank)
    step_ms = 10.0 if rank == 0 else 25.0  # rank 1 is the slow one
    ms, gbs = bench.aggregate_ranks(step_ms, 1e9, world)
    dist.barrier()
    out[rank] = (ms, gbs)
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_and_count_all_bytes():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, gbs = res[rank]
        assert ms == 25.0
        assert gbs == pytest.approx(2 * 1e9 / 25e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    ms, gbs = bench.aggregate_ranks(4.0, 2e9, 1)
    assert ms == 4.0 and gbs == pytest.approx(500.0)
