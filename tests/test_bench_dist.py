"""The multi-GPU bench path is replicas only: ranks exchange nothing but the
timing scalars.  Check the rank aggregation (barrier, max of step time, sum of
bytes) with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, local, w, dist = bench.dist_setup(world)
    assert (r, local, w) == (rank, rank, world)
    bench.barrier(dist)
    ms = bench.max_over_ranks(dist, 1.0 + rank)       # rank 1 is the slowest
    total = bench.sum_over_ranks(dist, 100.0 * (rank + 1))
    out.put((rank, ms, total))
    dist.destroy_process_group()


def test_rank_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 2.0, 300.0), (1, 2.0, 300.0)]


def test_bytes_formula_matches_survey_units():
    import bench
    from combine_get_dispatch_notify_gb300.workloads import CONFIGS
    w = CONFIGS["low_latency"]
    b = bench.algorithmic_bytes(w, 13456)
    tok = 16 * 128
    assert b["dispatch"] == tok * (2 * 7168 + 96) + 13456 * (2 * 7168 + 96 + 8)
    assert b["combine"] == 13456 * (2 * 7168 + 32 + 4) + tok * (2 * 7168 + 32)
    assert b["layout"] == tok * 64 + tok * 16 and b["notify"] == tok * 16 * 5
