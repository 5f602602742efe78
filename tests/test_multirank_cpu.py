"""The benchmark's multi-rank arithmetic on CPU: two gloo ranks, replicas of the same
workload, whole-job throughput = all ranks' bytes over the slowest rank's time."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    rank_ms = [40.0, 50.0][rank]  # rank 1 is the slow one
    gbs, ms = bench.job_throughput(10 ** 9, 4, rank_ms, world, device="cpu")
    q.put((rank, gbs, ms))
    dist.destroy_process_group()


def test_two_rank_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, gbs, ms in res:
        assert ms == 50.0                       # max over ranks
        assert abs(gbs - 2 * 4 * 1.0 / 0.050) < 1e-9  # 2 ranks x 4 steps x 1 GB / 50 ms
