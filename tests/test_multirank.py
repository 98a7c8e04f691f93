"""The N>1 benchmark path on CPU: replicas on gloo ranks, the slowest rank's time wins.

The layer does not shard across GPUs in this scope (replicas only), so the only
cross-rank step is the barrier and the max of the timings.
"""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    vals = bench.max_over_ranks([1.0 + rank, 10.0 - rank])
    ws, r, _ = bench.dist_env()
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, vals, ws, r))


def test_two_gloo_ranks_take_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, vals, ws, r in res:
        assert vals == [2.0, 10.0]
        assert ws == 2 and r == rank


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks([3.0, 4.5]) == [3.0, 4.5]
