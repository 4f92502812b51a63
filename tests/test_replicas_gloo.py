"""The N-GPU bench path runs independent replicas; its only cross-rank steps are a
barrier and the max-reduction of times. Checked here with two gloo ranks on the CPU."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [10.0 + rank, 30.0 - rank]            # each rank's own timings
    out = bench.slowest_rank(mine, world)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, out))


def test_slowest_rank_and_whole_job_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 30.0]
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas x 3 steps x 1e9 bytes in 1.5 s
    assert abs(bench.whole_job_gbs(1e9, 3, 2, 1500.0) - 4.0) < 1e-12
