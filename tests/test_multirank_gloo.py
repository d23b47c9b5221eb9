"""Multi-rank logic on the CPU (gloo, world size 2).

Requests are independent in verify, accept and commit, so a batch shards
across ranks by request with no collective on the data path; bench.py runs one
batch per rank (weak scaling) and only reduces its timings and unit counts.
These tests run the rank logic as two gloo processes: each rank evaluates its
shard (with the CPU oracle standing in for the GPU), the shards together
reproduce the single-process result, and the max/sum reductions bench.py uses
produce the whole-job throughput.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist

    import bench
    import oracle
    import workloads

    try:
        w, r, _ = bench.dist_setup(None)
        assert (w, r) == (world, rank)
        # shard one batch by request: rank r takes a contiguous slice of requests
        full = workloads.config2(seed=5, B=6, H=2)
        lo, hi = bench.shard_requests(full.B, world, rank)
        part = workloads.config2(seed=5, B=6, H=2)
        units = [u for u in range(full.B * full.H) if lo <= u // full.H < hi]
        res = oracle.verify(part, units=units)
        ln, path, bonus = oracle.accept_batch(part)
        mine = {u: o.tolist() for u, o in res.items()}
        gathered = [None] * world
        dist.all_gather_object(gathered, (mine, ln[lo:hi].tolist(), lo, hi))
        # the reductions bench.py applies to per-rank timings and unit counts
        t = 0.5 + rank
        tmax = bench.max_over_ranks(t, world)
        total = bench.sum_over_ranks(1000.0 * (rank + 1), world)
        bench.barrier(world)
        q.put((rank, gathered, tmax, total))
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put((rank, repr(e), None, None))


@pytest.mark.timeout(300)
def test_two_rank_sharding_and_reductions():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort(key=lambda x: x[0])
    for rank, gathered, tmax, total in out:
        assert not isinstance(gathered, str), gathered
        assert tmax == 1.5 and total == 3000.0

    import oracle
    import workloads
    full = workloads.config2(seed=5, B=6, H=2)
    ref = oracle.verify(full)
    ln_ref, _, _ = oracle.accept_batch(full)
    gathered = out[0][1]
    covered = set()
    for mine, lens, lo, hi in gathered:
        assert lens == ln_ref[lo:hi].tolist()
        for u, o in mine.items():
            assert np.array_equal(np.array(o), ref[int(u)])
            covered.add(int(u))
    assert covered == set(range(full.B * full.H))


def test_shard_requests_partitions_the_batch():
    import bench
    for B in (0, 1, 5, 16, 17):
        for world in (1, 2, 3, 8):
            spans = [bench.shard_requests(B, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == B
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c and a <= b
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
