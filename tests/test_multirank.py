"""The replicated multi-rank path of bench.py on CPU: two gloo ranks (no GPU).

Each rank times its own solves; the job reports the sum of all ranks' iterations over the slowest
rank's time.  The single-system solve has no exchange step, so no collective touches the data path.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r spent (r + 1) seconds on 100 * (r + 1) iterations
    secs, its = bench.aggregate_over_ranks(float(rank + 1), 100 * (rank + 1), world, "cpu")
    q.put((rank, secs, its))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_aggregate_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    expect_t = float(world)
    expect_it = float(sum(100 * (r + 1) for r in range(world)))
    for rank, secs, its in out:
        assert secs == expect_t and its == expect_it, (rank, secs, its)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_over_ranks(2.5, 7, 1) == (2.5, 7.0)
