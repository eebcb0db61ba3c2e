"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): replicas
meet only at the barrier and at the max-over-ranks time reduction."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    bench.barrier(ws)
    t = bench.max_over_ranks(1.0 + rank * 0.5, ws)   # rank 1 is the slow one
    units = 32 * 10 * ws                              # weak scaling: per-rank work fixed
    q.put((rank, t, units / t))
    dist.destroy_process_group()


def test_two_rank_max_time_and_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [1.5, 1.5]          # every rank sees the slowest rank's time
    assert abs(res[0][2] - 640 / 1.5) < 1e-9
