"""The multi-GPU path of bench.py is replicas only: every rank runs the whole
step on its own GPU and the job rate is (ranks x bytes per step) / (slowest
rank's step time).  This checks that aggregation with two gloo ranks on the
CPU (no GPU, no collective on the data path)."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms_local = [4.0, 5.0][rank]                  # rank 1 is the slower one
    gbs, ms = bench.aggregate(ms_local, 10_000_000_000, dist)
    out[rank] = (gbs, ms)
    dist.destroy_process_group()


def test_two_rank_aggregation_uses_the_slowest_rank():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        gbs, ms = out[r]
        assert ms == 5.0
        assert gbs == pytest.approx(2 * 10.0 / 5e-3)   # 2 ranks x 10 GB per 5 ms


def test_single_rank_aggregation():
    import bench

    gbs, ms = bench.aggregate(2.5, 5_000_000_000, None)
    assert ms == 2.5 and gbs == pytest.approx(2000.0)
