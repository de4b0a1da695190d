"""The multi-rank path of bench.py on CPU: two gloo ranks, barrier, max/sum
over ranks, one replica per rank on its own seed (no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from paged_kv_cache_170_gb300 import workloads

    r, w, local, dist = bench.dist_setup(world)
    assert (r, w) == (rank, world) and dist is not None
    bench.barrier(dist)
    mx = bench.max_over_ranks(float(rank + 1), dist)
    total = bench.sum_over_ranks(float(10 * (rank + 1)), dist)
    # each rank builds its own replica from seed + rank: different data, same shape
    inp = workloads.make_inputs(workloads.TINY, seed=rank)
    q_sum = bench.sum_over_ranks(float(inp.q.double().sum()), dist)
    dist.destroy_process_group()
    q.put((rank, mx, total, float(inp.q.double().sum()), q_sum))


@pytest.mark.timeout(120)
def test_two_rank_gloo_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(30)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]
    assert [r[2] for r in res] == [30.0, 30.0]
    assert res[0][3] != res[1][3]                      # different replicas
    assert abs(res[0][4] - (res[0][3] + res[1][3])) < 1e-9
