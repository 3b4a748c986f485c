"""The multi-rank host logic on CPU with world size 2 over gloo: the skip
decision is the OR of the ranks' overflow flags, timing takes the slowest
rank, and replicas take consecutive shards.  With the oracle as each rank's
local step (test infrastructure), two ranks that OR their flags and commit
or skip together end with the state an unsharded step would give."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from zero_partitioned_mixed_partition_gb300 import dist as zdist


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        oracle.build()
        out = {}
        out["or_none"] = zdist.agree_overflow(0)
        out["or_one"] = zdist.agree_overflow(1 if rank == 1 else 0)
        out["max"] = zdist.max_over_ranks(10.0 + rank)
        out["shard"] = zdist.replica_shard(3, rank, 4)

        # two ranks of a 2-way partition of one 1000-element buffer; rank 1's
        # contribution carries an inf at step 2 only
        n_d, psi = 2, 1000
        lay = oracle.layout([psi], n_d, 8)
        s = lay["shard_numel"]
        lo, hi = rank * s, min(psi, (rank + 1) * s)
        rng = np.random.Generator(np.random.PCG64(5))
        theta = rng.standard_normal(psi).astype(np.float32)
        contrib = [[(rng.standard_normal(psi) * 64).astype(np.float16) for _ in range(n_d)] for _ in range(3)]
        contrib[1][1][700] = np.inf
        master, m, v = theta[lo:hi].copy(), np.zeros(hi - lo, np.float32), np.zeros(hi - lo, np.float32)
        params = np.zeros(hi - lo, np.uint16)
        ls, applied, flags = 256.0, 0, []
        for step in range(3):
            parts = [c[lo:hi].view(np.uint16) for c in contrib[step]]
            g, bad = oracle.grad_reduce(parts, ls)
            ovf = zdist.agree_overflow(bad)
            flags.append(ovf)
            if not ovf:
                oracle.adam_apply(g, master, m, v, params, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                  weight_decay=0.0, step=applied + 1)
            ls, applied = oracle.commit(ovf, ls, applied)
        out["flags"] = flags
        out["master"] = (lo, master)
        out["ls"], out["applied"] = ls, applied

        # global gradient clipping: each rank adds its shard's sum of squares,
        # the ranks sum them, and every rank clips with the same factor
        cm, cmm, cv = theta[lo:hi].copy(), np.zeros(hi - lo, np.float32), np.zeros(hi - lo, np.float32)
        for step in range(2):
            parts = [c[lo:hi].view(np.uint16) for c in contrib[2 * step]]
            g, bad = oracle.grad_reduce(parts, 256.0)
            sq = torch.tensor([oracle.grad_sqnorm(g)], dtype=torch.float64)
            zdist.allreduce_sqnorm(sq)
            c = oracle.clip_factor(float(sq.item()), 5.0)
            oracle.scale(g, c)
            oracle.adam_apply(g, cm, cmm, cv, None, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                              weight_decay=0.0, step=step + 1)
        out["clip_sq"], out["clip_c"], out["clip_master"] = float(sq.item()), c, (lo, cm)
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_skip_and_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        o = res[r]
        assert o["or_none"] == 0 and o["or_one"] == 1 and o["max"] == 11.0
        assert o["shard"] == (3 + r) % 4
        assert o["flags"] == [0, 1, 0]           # rank 1's inf skips the step on both ranks
        assert o["ls"] == 128.0 and o["applied"] == 2

    # the union of the two ranks' shards equals one unsharded oracle run
    import oracle
    psi = 1000
    rng = np.random.Generator(np.random.PCG64(5))
    theta = rng.standard_normal(psi).astype(np.float32)
    contrib = [[(rng.standard_normal(psi) * 64).astype(np.float16) for _ in range(2)] for _ in range(3)]
    contrib[1][1][700] = np.inf
    master, m, v = theta.copy(), np.zeros(psi, np.float32), np.zeros(psi, np.float32)
    ls, applied = 256.0, 0
    for step in range(3):
        ovf = oracle.shard_step([c.view(np.uint16) for c in contrib[step]], master, m, v, None, lr=1e-3,
                                beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, loss_scale=ls,
                                step=applied + 1)
        ls, applied = oracle.commit(ovf, ls, applied)
    joined = np.zeros(psi, np.float32)
    for r in range(world):
        lo, part = res[r]["master"]
        joined[lo:lo + part.size] = part
    assert np.array_equal(joined, master)

    # clipped steps: the summed norm and the joined shards match one unsharded run
    cm, cmm, cv = theta.copy(), np.zeros(psi, np.float32), np.zeros(psi, np.float32)
    for step in range(2):
        g, _ = oracle.grad_reduce([c.view(np.uint16) for c in contrib[2 * step]], 256.0)
        sq = oracle.grad_sqnorm(g)
        c = oracle.clip_factor(sq, 5.0)
        oracle.scale(g, c)
        oracle.adam_apply(g, cm, cmm, cv, None, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                          step=step + 1)
    assert res[0]["clip_sq"] == res[1]["clip_sq"] and abs(res[0]["clip_sq"] - sq) <= 1e-12 * sq
    assert res[0]["clip_c"] == res[1]["clip_c"] == c and c < 1.0
    joined = np.zeros(psi, np.float32)
    for r in range(world):
        lo, part = res[r]["clip_master"]
        joined[lo:lo + part.size] = part
    np.testing.assert_allclose(joined, cm, rtol=2e-6, atol=1e-9)
