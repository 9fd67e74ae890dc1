"""The multi-replica path of bench.py on CPU: two gloo ranks, max-over-ranks timing and
the whole-job aggregate (units of all ranks / slowest rank's time)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, l = bench.dist_env()
    sec = [0.5, 2.0][rank]
    m = bench.max_over_ranks(sec, w)
    bench.barrier(w)
    agg = bench.aggregate(64, 10, w, m)
    q.put((r, w, m, agg["value"], agg["ms_per_step"]))
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, w, m, val, ms in res:
        assert w == 2 and m == 2.0
        assert val == pytest.approx(64 * 10 * 2 / 2.0)
        assert ms == pytest.approx(200.0)


def test_single_rank_aggregate_is_identity():
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.aggregate(64, 100, 1, 0.5)["value"] == pytest.approx(12800.0)
