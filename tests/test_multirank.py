"""The N > 1 bookkeeping of bench.py on CPU with the gloo backend (world size 2): every rank
runs its own replica, the job time is the slowest rank's, the job value counts every rank's work."""
import os
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(1.0 + rank, dist, "cpu")
    q.put((rank, t, bench.job_value(world, 1e12, 4, t)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [2.0, 2.0]
    assert all(abs(g[2] - 2 * 1e12 * 4 / 2.0 / 1e12) < 1e-9 for g in got)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_value(1, 2e12, 10, 2.0) == pytest.approx(10.0)


def _shard_rank(rank, world, port, q):
    """One rank: the oracle's mask and attention on this rank's (batch, key/value head) units only."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import oracle
    import workloads as W
    from free_block_sparse_gb300 import shards
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.make_config("llama32k", B=2, Hq=4, Hkv=2, N=700)
    qf, kf, vf = (W.bf16_to_f64(x) for x in (w.q, w.k, w.v))
    mine = {}
    for unit in shards.shard_units(w.B, w.Hkv, world, rank):
        b, hs, kvh = shards.unit_heads(unit, w.Hq, w.Hkv)
        qs, ks, vs = qf[b:b + 1, hs], kf[b:b + 1, kvh:kvh + 1], vf[b:b + 1, kvh:kvh + 1]
        pred = oracle.predict_mask(qs, ks, w.topk, w.theta, w.causal)
        out = oracle.block_sparse_attn(qs, ks, vs, pred["mask"], w.lam, w.causal)
        mine[unit] = (pred["mask"], out)
    parts = [None] * world
    dist.all_gather_object(parts, mine)
    if rank == 0:
        q.put(parts)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_partition_units_exactly():
    """Two ranks each take a disjoint share of the (batch, key/value head) units of a small
    Llama-like workload (B 2, 4 query heads over 2 key/value heads, causal, ragged tail) and run
    the oracle on their views only; the gathered masks and outputs equal the whole-tensor
    oracle's, every unit covered exactly once."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import oracle
    import workloads as W
    from free_block_sparse_gb300 import shards
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + os.getpid() % 1000
    procs = [ctx.Process(target=_shard_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    parts = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    w = W.make_config("llama32k", B=2, Hq=4, Hkv=2, N=700)
    qf, kf, vf = (W.bf16_to_f64(x) for x in (w.q, w.k, w.v))
    pred = oracle.predict_mask(qf, kf, w.topk, w.theta, w.causal)
    out = oracle.block_sparse_attn(qf, kf, vf, pred["mask"], w.lam, w.causal)
    seen = [u for part in parts for u in part]
    assert sorted(seen) == shards.units(w.B, w.Hkv)  # disjoint and complete
    assert all(len(part) == 2 for part in parts)
    for part in parts:
        for unit, (m, o) in part.items():
            b, hs, _ = shards.unit_heads(unit, w.Hq, w.Hkv)
            assert np.array_equal(m[0], pred["mask"][b, hs])
            assert np.array_equal(o[0], out[b, hs])


@pytest.mark.parametrize("B,Hkv,world", [(1, 8, 3), (2, 2, 4), (3, 5, 2), (1, 1, 1)])
def test_shard_units_cover_every_unit_once(B, Hkv, world):
    sys.path.insert(0, ROOT)
    from free_block_sparse_gb300 import shards
    got = [shards.shard_units(B, Hkv, world, r) for r in range(world)]
    flat = [u for g in got for u in g]
    assert flat == shards.units(B, Hkv)
    sizes = [len(g) for g in got]
    assert max(sizes) - min(sizes) <= 1
