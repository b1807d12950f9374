"""The bench's N > 1 path (replicas only: the linear does not shard across
GPUs here, so N GPUs run N independent copies of the workload): the
whole-job value is every rank's algorithmic bytes over the slowest rank's
step time.  Runs as two gloo ranks on the CPU (no GPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: 10 + 5 r ms per step, 1 GB per step on every rank
        ms = 10.0 + 5.0 * rank
        out = {"ms_per_step": ms, "value": 1.0 / (ms * 1e-3), "n_gpus": 1, "other": rank}
        bench._barrier()
        res = bench.aggregate_replicas(out, dist, "cpu")
        q.put((rank, res))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_every_rank_bytes():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        assert res[r]["n_gpus"] == world
        assert res[r]["ms_per_step"] == pytest.approx(15.0)        # the slowest rank
        assert res[r]["value"] == pytest.approx(2 * 1.0 / 15e-3, abs=0.05)   # 2 GB per 15 ms (1 decimal)
        assert res[r]["other"] == r                                  # the rest is the rank's own line
