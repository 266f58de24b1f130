"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks on 127.0.0.1.  Each rank runs its own
independent batch (distinct seeds), and the job's time is the slowest rank's (max over ranks)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    t = bench.max_over_ranks(10.0 + 5.0 * rank, ws)
    bench.barrier(ws)
    out[rank] = (ws, r, local, t, bench.rank_seed(2, r))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_distinct_batches():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][:3] == (2, 0, 0) and out[1][:3] == (2, 1, 1)
    assert out[0][3] == out[1][3] == 15.0          # both see the slowest rank's time
    assert out[0][4] != out[1][4]                  # independent batches per rank (weak scaling)
