"""The N > 1 path of the benchmark on CPU: gloo, world size 2.  Each rank runs
its own batch (weak scaling, no data exchange); the only collectives are the
timing max and the byte/sequence sums."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from paged_kv_cache_11_gb300 import workload as W
    dist = bench.init_dist(world, "gloo")
    ws, r, local = bench.dist_env()
    spec = W.SPECS["tiny"]
    wl = W.make_workload("tiny", seed=bench.rank_seed(W.default_seed(spec), r))
    mx = bench.max_over_ranks(dist, 10.0 + r)
    sm = bench.sum_over_ranks(dist, float(wl.kv_bytes()))
    q.put((r, ws, mx, sm, int(wl.q[0, 0, 0]), bench.rank_seed(W.default_seed(spec), r)))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
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
    (r0, ws0, mx0, sm0, q0, s0), (r1, ws1, mx1, sm1, q1, s1) = res
    assert ws0 == ws1 == 2
    assert mx0 == mx1 == 11.0                    # max over ranks
    assert sm0 == sm1                             # same total on every rank
    assert s0 != s1                               # each rank its own batch
