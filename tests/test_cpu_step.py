"""The shard step on the host cores (ZeRO-Offload's CPU Adam, "DeepSpeed ZeRO
Stages" sec. 5.1) against the oracle: same arithmetic, so bit-exact, for
ragged sizes, N_d = 1 / non-powers of two / 64, one to eight threads,
in-place state, overflow skip with restore, and a multi-shard step.  Runs on
the CPU (no CUDA call)."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from parity_util import OracleShard, oracle_group_step


def _w(n, n_d, **kw):
    base = dict(name="cpu", numels=(n,), n_d=n_d, rank=0, align=1, steps=3, lr=1e-3, beta1=0.9, beta2=0.999,
                eps=1e-8, weight_decay=0.05, loss_scale=512.0, grad_dist="normal", grad_std=1e-2, grad_mult=512.0,
                grads_fresh_per_step=True, master_dist="normal", master_param=0.02, seed=n + 13 * n_d)
    base.update(kw)
    return synth.Workload(**base)


def _host_shard(zs, w, n, inplace=False):
    grads = [torch.zeros(n, dtype=torch.float16) for _ in range(w.n_d)]
    master0 = synth.master_init(w, n)
    mk = lambda: torch.zeros(n, dtype=torch.float32)
    a = master0.clone()
    master = (a, a if inplace else mk())
    m0 = mk()
    m = (m0, m0 if inplace else mk())
    v0 = mk()
    v = (v0, v0 if inplace else mk())
    params = torch.zeros(n, dtype=torch.float16)
    view = zs.CpuShardView(grads, master, m, v, params, n)
    return view, master0


@pytest.mark.parametrize("n", [1, 7, 2049, 70001])
@pytest.mark.parametrize("n_d", [1, 3, 4, 64])
@pytest.mark.parametrize("threads", [1, 3, 8])
def test_cpu_step_bit_exact(zs, oracle, n, n_d, threads):
    w = _w(n, n_d)
    view, master0 = _host_shard(zs, w, n)
    ref = OracleShard(oracle, master0.numpy())
    cur, ls, applied = 0, w.loss_scale, 0
    for step in range(1, 4):
        contribs = [synth.grad_contribution(w, n, k, step) for k in range(n_d)]
        if step == 2 and n > 5:
            contribs[n_d - 1][n - 1] = float("inf")
        for g, c in zip(view.grads, contribs):
            g.copy_(c)
        ovf = zs.zero_shard_step_cpu([view], n_d, zs.adam(w.lr, weight_decay=w.weight_decay), ls, applied + 1,
                                     cur, n_threads=threads)
        rovf, ls, applied = oracle_group_step(oracle, [ref], [[synth.fp16_bits(c) for c in contribs]], w, ls,
                                              applied)
        assert ovf == rovf
        if not ovf:
            cur ^= 1
        for got, want in ((view.master[cur], ref.master), (view.m[cur], ref.m), (view.v[cur], ref.v)):
            assert np.array_equal(got.numpy().view(np.uint32), want.view(np.uint32))
        assert np.array_equal(view.params.view(torch.int16).numpy().view(np.uint16), ref.params)


def test_cpu_step_in_place_and_multi_shard(zs, oracle):
    n_d = 4
    sizes = [5000, 33, 12288]
    views, refs = [], []
    for i, n in enumerate(sizes):
        w = _w(n, n_d, seed=100 + i)
        v, m0 = _host_shard(zs, w, n, inplace=(i == 1))
        views.append(v)
        refs.append(OracleShard(oracle, m0.numpy()))
    w = _w(sizes[0], n_d)
    ls, applied = w.loss_scale, 0
    for step in range(1, 3):
        contribs = []
        for i, (v, n) in enumerate(zip(views, sizes)):
            c = [synth.random_fp16(n, 1000 * step + 10 * i + k, scale=100.0) for k in range(n_d)]
            for g, x in zip(v.grads, c):
                g.copy_(x)
            contribs.append([synth.fp16_bits(x) for x in c])
        ovf = zs.zero_shard_step_cpu(views, n_d, zs.adam(w.lr, weight_decay=w.weight_decay), ls, applied + 1,
                                     (applied % 2), n_threads=4)
        rovf, ls, applied = oracle_group_step(oracle, refs, contribs, w, ls, applied)
        assert ovf == rovf == 0
        for i, (v, ref) in enumerate(zip(views, refs)):
            cur = 0 if i == 1 else applied % 2
            assert np.array_equal(v.master[cur].numpy(), ref.master)
            assert np.array_equal(v.params.view(torch.int16).numpy().view(np.uint16), ref.params)


def test_cpu_step_rejects_bad_arguments(zs):
    import ctypes
    L = zs.lib()
    ovf = ctypes.c_int32()
    hp = zs.adam(1e-3)
    assert L.zero_shard_step_cpu(None, 1, 2, ctypes.byref(hp), 1.0, 1, 0, 1, ctypes.byref(ovf)) == zs.ZS_ERR_ARG
    n = 16
    w = _w(n, 2)
    view, _ = _host_shard(zs, w, n)
    arr = (zs.Shard * 1)(view.struct)
    assert L.zero_shard_step_cpu(arr, 1, 2, ctypes.byref(hp), 0.0, 1, 0, 1, ctypes.byref(ovf)) == zs.ZS_ERR_ARG
    assert L.zero_shard_step_cpu(arr, 1, 2, ctypes.byref(hp), 1.0, 0, 0, 1, ctypes.byref(ovf)) == zs.ZS_ERR_ARG
    arr[0].qcodes = 64
    arr[0].qscales = 64
    assert L.zero_shard_step_cpu(arr, 1, 2, ctypes.byref(hp), 1.0, 1, 0, 1, ctypes.byref(ovf)) == zs.ZS_ERR_ARG
