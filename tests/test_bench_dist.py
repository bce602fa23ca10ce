"""bench.py's multi-rank path on CPU: two gloo ranks, each runs its own replica; the timing is
max-reduced across ranks and a barrier brackets it (no data-path collective exists)."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import bench
    r, w, _ = bench.dist_setup()
    bench.barrier(w)
    ms = bench.max_over_ranks(10.0 * (r + 1), w)   # rank 1 is the slow one
    bench.barrier(w)
    out.put((r, w, ms))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_reduce_timing():
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
    assert res == [(0, 2, 20.0), (1, 2, 20.0)]
