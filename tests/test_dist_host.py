"""The benchmark's multi-process bookkeeping (N > 1 replicas) on CPU: two
gloo ranks agree on the max time over ranks and on the whole-job
aggregate.  No GPU and no data-path collective is involved: every GPU
replica runs its own W virtual ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r = bench.init_dist("gloo")
    bench.barrier()
    t = 1.0 + rank  # rank 1 is the slow one
    tmax = bench.max_over_ranks(t)
    val = bench.aggregate_gbs(4e9, 10, ws, tmax)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, ws, tmax, val))


def test_two_gloo_ranks_take_max_time():
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
    assert [r[0] for r in res] == [0, 1]
    for _, ws, tmax, val in res:
        assert ws == 2 and tmax == 2.0
        assert val == pytest.approx(4e9 * 10 * 2 / 2.0 / 1e9)


def test_single_process_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate_gbs(1e9, 4, 1, 2.0) == pytest.approx(2.0)
