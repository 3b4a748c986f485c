"""ZeRO-Offload on a GB300 machine ("DeepSpeed ZeRO Stages" sec. 5.1; "DeepSpeed
ZeRO: Extreme Memory Efficiency", the ZeRO-Offload section): the host-core
step and the full offload step with its transfers, against the oracle, bit
for bit.

  - the host-core step (zero_shard_step_cpu) on the GPU machine's own host
    CPU (aarch64 on Grace; the CPU tests run it on x86_64 too): ragged sizes,
    N_d = 1, 4, 64, one thread and every core, an overflow step;
  - zero_shard_step_offload: contributions copied from the device to
    page-locked staging, the step on the host cores, fp16 parameters copied
    back, overlapped by chunks; several chunk sizes and thread counts, an
    overflow step in the middle (the device slice must hold the kept
    parameters afterwards), and the device slice compared with the oracle's
    fp16 parameters after every step;
  - staging memory that is not page-locked is refused.
"""
import ctypes

import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from parity_util import OracleShard, oracle_group_step
from test_cpu_step import _host_shard, _w

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,n_d,threads", [(2049, 1, 1), (70001, 4, 0), (70001, 64, 3), (1_000_003, 4, 0),
                                           (4_000_037, 8, 0)])
def test_host_step_bit_exact_on_this_host(zs, oracle, cuda_device, n, n_d, threads):
    w = _w(n, n_d)
    view, master0 = _host_shard(zs, w, n)
    ref = OracleShard(oracle, master0.numpy())
    cur, ls, applied = 0, w.loss_scale, 0
    for step in range(1, 4):
        contribs = [synth.grad_contribution(w, n, k, step) for k in range(n_d)]
        if step == 2:
            contribs[n_d - 1][n - 1] = float("inf")
        for g, c in zip(view.grads, contribs):
            g.copy_(c)
        ovf = zs.zero_shard_step_cpu([view], n_d, zs.adam(w.lr, weight_decay=w.weight_decay), ls, applied + 1,
                                     cur, n_threads=threads)
        rovf, ls, applied = oracle_group_step(oracle, [ref], [[synth.fp16_bits(c) for c in contribs]], w, ls,
                                              applied)
        assert ovf == rovf == int(step == 2)
        if not ovf:
            cur ^= 1
        for got, want in ((view.master[cur], ref.master), (view.m[cur], ref.m), (view.v[cur], ref.v)):
            assert np.array_equal(got.numpy().view(np.uint32), want.view(np.uint32))
        assert np.array_equal(view.params.view(torch.int16).numpy().view(np.uint16), ref.params)


def _offload_shard(zs, dev, w, n):
    grads_dev = [torch.zeros(n, dtype=torch.float16, device=dev) for _ in range(w.n_d)]
    grads_host = [torch.zeros(n, dtype=torch.float16).pin_memory() for _ in range(w.n_d)]
    params_host = torch.zeros(n, dtype=torch.float16).pin_memory()
    master0 = synth.master_init(w, n)
    mk = lambda: torch.zeros(n, dtype=torch.float32)
    master = (master0.clone(), mk())
    m = (mk(), mk())
    v = (mk(), mk())
    params_dev = master0.to(torch.float16).to(dev)        # fp16(master): RNE on both sides
    view = zs.OffloadShardView(grads_dev, params_dev, grads_host, params_host, master, m, v, n)
    return view, master0


@pytest.mark.parametrize("n,n_d,threads,chunk", [(70001, 4, 4, 4096), (1_000_003, 4, 0, 0),
                                                 (2_500_013, 8, 0, 65536), (300_007, 64, 0, 1 << 16),
                                                 (17, 2, 0, 16)])
def test_offload_step_matches_oracle(zs, oracle, cuda_device, n, n_d, threads, chunk):
    w = _w(n, n_d)
    view, master0 = _offload_shard(zs, cuda_device, w, n)
    ref = OracleShard(oracle, master0.numpy())
    assert np.array_equal(synth.fp16_bits(view.params_dev), ref.params)
    hp = zs.adam(w.lr, weight_decay=w.weight_decay)
    d2h, h2d = torch.cuda.Stream(device=cuda_device), torch.cuda.Stream(device=cuda_device)
    cur, ls, applied = 0, w.loss_scale, 0
    for step in range(1, 5):
        contribs = [synth.grad_contribution(w, n, k, step) for k in range(n_d)]
        if step == 2:
            contribs[0][n // 2] = float("nan")
        for g, c in zip(view.grads_dev, contribs):
            g.copy_(c.to(cuda_device))
        torch.cuda.synchronize()
        ovf = zs.zero_shard_step_offload(view, n_d, hp, ls, applied + 1, cur, n_threads=threads, chunk=chunk,
                                         d2h_stream=d2h, h2d_stream=h2d)
        rovf, ls, applied = oracle_group_step(oracle, [ref], [[synth.fp16_bits(c) for c in contribs]], w, ls,
                                              applied)
        assert ovf == rovf == int(step == 2), step
        if not ovf:
            cur ^= 1
        for got, want in ((view.master[cur], ref.master), (view.m[cur], ref.m), (view.v[cur], ref.v)):
            assert np.array_equal(got.numpy().view(np.uint32), want.view(np.uint32)), step
        # the call is synchronous: the device slice already holds the result
        assert np.array_equal(synth.fp16_bits(view.params_dev), ref.params), step
        assert np.array_equal(synth.fp16_bits(view.params_host), ref.params), step


def test_offload_refuses_pageable_staging(zs, cuda_device):
    n, n_d = 64, 2
    w = _w(n, n_d)
    view, _ = _offload_shard(zs, cuda_device, w, n)
    pageable = torch.zeros(n, dtype=torch.float16)
    s = zs.OffloadShard.from_buffer_copy(view.struct)
    s.params_host = pageable.data_ptr()
    ovf = ctypes.c_int32(-1)
    launches = zs.zero_kernel_launches()
    rc = zs.lib().zero_shard_step_offload(ctypes.byref(s), n_d, ctypes.byref(zs.adam(1e-3)), 1.0, 1, 0, 0, 0,
                                          None, None, ctypes.byref(ovf))
    assert rc == zs.ZS_ERR_ARG and b"page-locked" in zs.lib().zero_last_error()
    assert zs.zero_kernel_launches() == launches
    with pytest.raises(TypeError):
        zs.OffloadShardView(view.grads_dev, view.params_dev, view.grads_host, pageable, view.master, view.m, view.v,
                            n)
