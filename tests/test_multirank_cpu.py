"""Host logic of the multi-rank benchmark path on CPU (gloo, world size 2):
replicas, timing reduced as the max over ranks, whole-job rate aggregated
over ranks. No GPU and no collective on the data path."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, local = bench.dist_env()
    secs = 1.0 + rank  # rank 1 is the slow one
    m = bench.max_over_ranks(secs, w)
    rate = bench.whole_job_rate(100.0, w, m)
    out.put((r, w, local, m, rate))
    dist.destroy_process_group()


def test_two_rank_max_and_rate():
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
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[3] == pytest.approx(2.0) for r in res)       # slowest rank's time
    assert all(r[4] == pytest.approx(100.0) for r in res)     # 2 ranks x 100 units / 2 s
