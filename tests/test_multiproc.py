"""The N>1 bench path on CPU: two gloo ranks, max-over-ranks timing, barrier.

The decode path shards by replica (each rank runs its own batch, no data-path
collective); what crosses ranks is only the barrier around the timed region
and the max of the elapsed times, which these tests exercise.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method="env://")
    w, r, l = bench._dist()
    bench.barrier(w)
    got = bench.reduce_max(1.5 + rank, w)
    from paged_kv_decode_05_gb300.workloads import CONFIGS, make_workload
    cfg = CONFIGS["tiny"]
    lens_sum = int(make_workload(cfg, seed=cfg.seed + r).q.astype("float64").sum())
    q.put((r, w, got, lens_sum))
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_max_and_replica_seeds():
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
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[2] == 2.5 for r in res)          # max over ranks seen by every rank
    assert res[0][3] != res[1][3]                 # each replica draws its own data


def test_single_rank_helpers_are_identity():
    import bench
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)
    assert bench._dist()[0] in (1, int(os.environ.get("WORLD_SIZE", "1")))
