"""Parity of the CUDA shard step with the oracle, element by element, at sizes
the oracle finishes in seconds (several tiles plus ragged tails), and the edge
cases of the method: empty shards, tails shorter than a vector, N_d = 1 and
non-powers of two, misaligned buffers (scalar kernel), in-place state,
+inf / -inf / NaN / (+inf, -inf) contributions at the first, last and tail
elements, multi-shard steps that skip together, and a captured CUDA graph."""
import dataclasses

import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner
from parity_util import (OracleShard, assert_f16_close, assert_f32_close, f16_bits, oracle_group_step,
                         to_np, MAX_ULP)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _fresh_ulp_record():
    """test_report_max_ulp summarises this module's comparisons only."""
    MAX_ULP["f32"] = MAX_ULP["f16"] = 0
    yield


def _workload(n, n_d, **kw):
    base = dict(name="case", numels=(n,), n_d=n_d, rank=0, align=1, steps=3, lr=1e-3, beta1=0.9,
                beta2=0.999, eps=1e-8, weight_decay=0.0, loss_scale=1024.0, grad_dist="normal",
                grad_std=1e-2, grad_mult=1024.0, grads_fresh_per_step=True, master_dist="normal",
                master_param=0.02, seed=n * 31 + n_d)
    base.update(kw)
    return synth.Workload(**base)


class SyncShard:
    """Device buffers of one shard for the synchronous entry point, built from
    host arrays, with the host-side commit bookkeeping."""

    def __init__(self, zs, dev, contribs, master0, n, offset=0, inplace=False, off_h=None, off_f=None):
        self.zs = zs
        oh = offset if off_h is None else off_h
        of = offset if off_f is None else off_f
        self.g = [torch.zeros(n + oh + 16, dtype=torch.float16, device=dev)[oh:oh + n] for _ in contribs]
        for t, c in zip(self.g, contribs):
            t.copy_(c.to(dev))
        mk = lambda: torch.zeros(n + of + 16, dtype=torch.float32, device=dev)[of:of + n]
        self.master = (mk(), None)
        self.master[0].copy_(master0.to(dev))
        self.master = (self.master[0], self.master[0] if inplace else mk())
        a = mk()
        self.m = (a, a if inplace else mk())
        b = mk()
        self.v = (b, b if inplace else mk())
        self.params = torch.zeros(n + oh + 16, dtype=torch.float16, device=dev)[oh:oh + n]
        zs.zero_params_from_master(self.master[0], self.params, n)
        self.view = zs.ShardView(self.g, self.master, self.m, self.v, self.params, n)
        self.cur = 0

    def set_grads(self, contribs):
        for t, c in zip(self.g, contribs):
            t.copy_(c.to(t.device))

    def state(self):
        c = self.cur
        return (to_np(self.master[c]), to_np(self.m[c]), to_np(self.v[c]), f16_bits(self.params))


def _contribs(w, n, step):
    return [synth.grad_contribution(w, n, k, step) for k in range(w.n_d)]


def _bits(ts):
    return [synth.fp16_bits(t) for t in ts]


# ------------------------------------------------------------ sync path ---

SIZES = [1, 7, 8, 9, 2047, 2048 * 3 + 5, 65536 + 3, 262144]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("n_d", [1, 3, 4, 8])
def test_sync_step_matches_oracle(zs, oracle, cuda_device, n, n_d):
    w = _workload(n, n_d, weight_decay=0.1 if n % 2 else 0.0)
    master0 = synth.master_init(w, n)
    sh = SyncShard(zs, cuda_device, _contribs(w, n, 1), master0, n)
    ref = OracleShard(oracle, master0.numpy())
    assert_f16_close(f16_bits(sh.params), ref.params, "initial cast")
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ls, applied = w.loss_scale, 0
    for step in range(1, 4):
        contribs = _contribs(w, n, step)
        sh.set_grads(contribs)
        ovf = zs.zero_shard_step([sh.view], n_d, zs.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay),
                                 ls, applied + 1, sh.cur, flag)
        rovf, ls_ref, applied_ref = oracle_group_step(oracle, [ref], [_bits(contribs)], w, ls, applied)
        assert ovf == rovf == 0
        sh.cur ^= 1
        ls, applied = ls_ref, applied_ref
        ref.compare(*sh.state(), what=f"n={n} n_d={n_d} step={step}")


@pytest.mark.parametrize("n_d", [2, 5, 16, 17, 32, 64, 65, 100])
def test_sync_step_many_contributions(zs, oracle, cuda_device, n_d):
    n = 4099
    w = _workload(n, n_d, loss_scale=float(2 ** 14), grad_mult=float(2 ** 14))
    master0 = synth.master_init(w, n)
    sh = SyncShard(zs, cuda_device, _contribs(w, n, 1), master0, n)
    ref = OracleShard(oracle, master0.numpy())
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for step in (1, 2):
        contribs = _contribs(w, n, step)
        sh.set_grads(contribs)
        ovf = zs.zero_shard_step([sh.view], n_d, zs.adam(w.lr), w.loss_scale, step, sh.cur, flag)
        assert ovf == 0
        oracle_group_step(oracle, [ref], [_bits(contribs)], w, w.loss_scale, step - 1)
        sh.cur ^= 1
        ref.compare(*sh.state(), what=f"n_d={n_d} step={step}")


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_misaligned_buffers_take_scalar_kernel(zs, oracle, cuda_device, offset):
    n, n_d = 5000, 3
    w = _workload(n, n_d)
    master0 = synth.master_init(w, n)
    sh = SyncShard(zs, cuda_device, _contribs(w, n, 1), master0, n, offset=offset)
    assert sh.params.data_ptr() % 16 != 0
    ref = OracleShard(oracle, master0.numpy())
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ovf = zs.zero_shard_step([sh.view], n_d, zs.adam(w.lr), w.loss_scale, 1, 0, flag)
    oracle_group_step(oracle, [ref], [_bits(_contribs(w, n, 1))], w, w.loss_scale, 0)
    assert ovf == 0
    sh.cur = 1
    ref.compare(*sh.state(), what=f"offset={offset}")


def test_in_place_state(zs, oracle, cuda_device):
    n, n_d = 10001, 4
    w = _workload(n, n_d, weight_decay=0.05)
    master0 = synth.master_init(w, n)
    sh = SyncShard(zs, cuda_device, _contribs(w, n, 1), master0, n, inplace=True)
    ref = OracleShard(oracle, master0.numpy())
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for step in (1, 2, 3):
        contribs = _contribs(w, n, step)
        sh.set_grads(contribs)
        assert zs.zero_shard_step([sh.view], n_d, zs.adam(w.lr, weight_decay=w.weight_decay), w.loss_scale,
                                  step, 0, flag) == 0
        oracle_group_step(oracle, [ref], [_bits(contribs)], w, w.loss_scale, step - 1)
        ref.compare(*sh.state(), what=f"in-place step={step}")


def test_empty_shard(zs, cuda_device):
    w = _workload(16, 2)
    sh = SyncShard(zs, cuda_device, _contribs(w, 16, 1), synth.master_init(w, 16), 16)
    empty = zs.ShardView(sh.g, sh.master, sh.m, sh.v, sh.params, 0)
    flag = torch.ones(1, dtype=torch.int32, device=cuda_device)
    before = sh.state()
    assert zs.zero_shard_step([empty], 2, zs.adam(1e-3), 1.0, 1, 0, flag) == 0
    for a, b in zip(before, sh.state()):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("n_d", [4, 8, 64])
@pytest.mark.parametrize("off_h,off_f,width", [(0, 0, "wide"), (8, 4, "narrow"), (0, 4, "narrow"),
                                               (1, 0, "scalar"), (0, 1, "scalar")])
def test_alignment_paths(zs, oracle, cuda_device, n_d, off_h, off_f, width):
    """The three access widths (16 / 8 elements per thread, scalar) give the
    oracle's results; offsets pick the width through buffer alignment."""
    n = 2048 * 9 + 13
    w = _workload(n, n_d)
    master0 = synth.master_init(w, n)
    sh = SyncShard(zs, cuda_device, _contribs(w, n, 1), master0, n, off_h=off_h, off_f=off_f)
    assert (sh.master[0].data_ptr() % 32 == 0) == (off_f == 0)
    ref = OracleShard(oracle, master0.numpy())
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    for step in (1, 2):
        contribs = _contribs(w, n, step)
        sh.set_grads(contribs)
        assert zs.zero_shard_step([sh.view], n_d, zs.adam(w.lr), w.loss_scale, step, sh.cur, flag) == 0
        oracle_group_step(oracle, [ref], [_bits(contribs)], w, w.loss_scale, step - 1)
        sh.cur ^= 1
        ref.compare(*sh.state(), what=f"{width} n_d={n_d} step={step}")


# ----------------------------------------------------- overflow and skip ---

def _place(kind, contribs, j):
    if kind == "inf":
        contribs[1][j] = float("inf")
    elif kind == "-inf":
        contribs[0][j] = float("-inf")
    elif kind == "nan":
        contribs[-1][j] = float("nan")
    else:
        contribs[0][j] = float("inf")
        contribs[-1][j] = float("-inf")


@pytest.mark.parametrize("kind", ["inf", "-inf", "nan", "inf-inf"])
@pytest.mark.parametrize("where", ["first", "last", "tail", "middle"])
def test_overflow_skips_async(zs, oracle, cuda_device, kind, where):
    n, n_d = 2048 * 5 + 6, 3
    w = _workload(n, n_d, numels=(n * n_d,), loss_scale=2.0 ** 16, grad_mult=2.0 ** 16,
                  grads_fresh_per_step=False)
    j = {"first": 0, "last": n - 1, "tail": n - 4, "middle": 4097}[where]
    run = WorkloadRunner(w, cuda_device)
    r = run.shard_ids[0]
    refs = [OracleShard(oracle, to_np(run.state[r][0][0]))]
    host = [_bits(run.grads[r])]
    ls, applied = w.loss_scale, 0
    for step in range(1, 5):
        inject = step == 2
        if inject:
            saved = [g.clone() for g in run.grads[r]]
            _place(kind, run.grads[r], j)
            host_step = [_bits(run.grads[r])]
        else:
            host_step = host
        before = [t.clone() for t in run.current(r)]
        run.step()
        torch.cuda.synchronize()
        ovf, ls, applied = oracle_group_step(oracle, refs, host_step, w, ls, applied)
        c = run.ctrl_host()
        assert c["last_overflow"] == ovf == (1 if inject else 0)
        assert c["loss_scale"] == ls and c["step"] == applied and c["overflow"] == 0 and c["arrivals"] == 0
        if inject:
            assert c["skipped"] == 1
            for a, b in zip(before, run.current(r)):
                assert torch.equal(a, b)            # state and fp16 slice as before the step
            for g, s in zip(run.grads[r], saved):
                g.copy_(s)
        master, m, v, params = run.current(r)
        refs[0].compare(to_np(master), to_np(m), to_np(v), f16_bits(params), what=f"step {step}")


def test_overflow_skips_sync_restores_params(zs, oracle, cuda_device):
    n, n_d = 3000, 4
    w = _workload(n, n_d)
    master0 = synth.master_init(w, n)
    sh = SyncShard(zs, cuda_device, _contribs(w, n, 1), master0, n)
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    assert zs.zero_shard_step([sh.view], n_d, zs.adam(w.lr), w.loss_scale, 1, 0, flag) == 0
    sh.cur = 1
    before = sh.state()
    contribs = _contribs(w, n, 2)
    contribs[2][n - 1] = float("inf")
    sh.set_grads(contribs)
    assert zs.zero_shard_step([sh.view], n_d, zs.adam(w.lr), w.loss_scale, 2, 1, flag) == 1
    for a, b in zip(before, sh.state()):
        assert np.array_equal(a, b)


def test_multi_shard_step_skips_together(zs, oracle, cuda_device):
    """Every shard of a small ragged tensor list stepped in one step; an
    overflow in one shard's contributions skips all of them."""
    numels = tuple(synth.ragged_numels(96, seed=3, max_exp=12))
    w = _workload(0, 16, numels=numels, rank=None, align=128, grads_fresh_per_step=False,
                  grad_dist="laplace", grad_std=5e-4, grad_mult=2.0 ** 14, loss_scale=2.0 ** 14,
                  master_dist="uniform", master_param=0.05, seed=7)
    run = WorkloadRunner(w, cuda_device)
    assert len(run.shard_ids) == 16
    refs = [OracleShard(oracle, to_np(run.state[r][0][0][: run.n_valid[r]])) for r in run.shard_ids]
    ls, applied = w.loss_scale, 0
    victim = run.shard_ids[5]
    for step in range(1, 5):
        inject = step == 3
        if inject:
            run.grads[victim][7][run.n_valid[victim] // 2] = float("nan")
        host_step = [[synth.fp16_bits(g[: run.n_valid[r]]) for g in run.grads[r]] for r in run.shard_ids]
        run.step()
        torch.cuda.synchronize()
        ovf, ls, applied = oracle_group_step(oracle, refs, host_step, w, ls, applied)
        c = run.ctrl_host()
        assert c["last_overflow"] == ovf == int(inject)
        assert c["step"] == applied and c["loss_scale"] == ls
        if inject:
            run.grads[victim][7][run.n_valid[victim] // 2] = 0.0
        for ref, r in zip(refs, run.shard_ids):
            n = run.n_valid[r]
            master, m, v, params = run.current(r)
            ref.compare(to_np(master[:n]), to_np(m[:n]), to_np(v[:n]), f16_bits(params[:n]),
                        what=f"shard {r} step {step}")
            assert not to_np(master[n:]).any()       # padding never written
    # the union of the shards' fp16 slices is the whole updated parameter buffer
    full = f16_bits(run.params_full)
    for ref, r in zip(refs, run.shard_ids):
        lo = r * run.S
        assert np.array_equal(full[lo:lo + run.n_valid[r]], ref.params)


def test_loss_scale_floor_and_counts(zs, cuda_device):
    n, n_d = 64, 2
    w = _workload(n, n_d, numels=(n * n_d,), loss_scale=2.0, grads_fresh_per_step=False)
    run = WorkloadRunner(w, cuda_device)
    r = run.shard_ids[0]
    run.grads[r][0][3] = float("inf")
    launches = zs.zero_kernel_launches()
    for _ in range(3):
        run.step()
    torch.cuda.synchronize()
    assert zs.zero_kernel_launches() - launches == 6        # fused + commit per step
    c = run.ctrl_host()
    assert c["loss_scale"] == 1.0 and c["skipped"] == 3 and c["step"] == 0 and c["cur"] == 0


def test_graph_captured_steps(zs, oracle, cuda_device):
    n, n_d = 2048 * 7 + 1, 4
    w = _workload(n, n_d, numels=(n * n_d,), grads_fresh_per_step=False)
    run = WorkloadRunner(w, cuda_device)
    r = run.shard_ids[0]
    ref = OracleShard(oracle, to_np(run.state[r][0][0]))
    host = [_bits(run.grads[r])]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run.step()                                 # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ls, applied = oracle_group_step(oracle, [ref], host, w, w.loss_scale, 0)[1:]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run.step()
    for _ in range(3):
        g.replay()
        _, ls, applied = oracle_group_step(oracle, [ref], host, w, ls, applied)
    torch.cuda.synchronize()
    c = run.ctrl_host()
    assert c["step"] == applied == 4
    master, m, v, params = run.current(r)
    ref.compare(to_np(master), to_np(m), to_np(v), f16_bits(params), what="graph")


def test_host_memory_path(zs, oracle, cuda_device):
    """zero_shard_step_host: contributions read from, and the fp16 shard
    written to, page-locked host memory by the fused kernel."""
    import ctypes
    n, n_d = 2048 * 11 + 5, 4
    w = _workload(n, n_d, numels=(n * n_d,), grads_fresh_per_step=False)
    run = WorkloadRunner(w, cuda_device)
    r = run.shard_ids[0]
    host_grads = [g[:n].cpu().pin_memory() for g in run.grads[r]]
    host_params = torch.zeros(n, dtype=torch.float16).pin_memory()
    master, m, v, _ = run.state[r]
    view = zs.HostShardView(host_grads, master, m, v, host_params, n)
    ref = OracleShard(oracle, to_np(master[0]))
    ls, applied = w.loss_scale, 0
    for step in range(1, 5):
        if step == 2:
            saved = host_grads[1][17].clone()
            host_grads[1][17] = float("inf")
        host_step = [_bits(host_grads)]
        ovf = zs.zero_shard_step_host(view, n_d, run.hp, run.ctrl)
        rovf, ls, applied = oracle_group_step(oracle, [ref], host_step, w, ls, applied)
        assert ovf == rovf == int(step == 2)
        if step == 2:
            host_grads[1][17] = saved
        c = run.ctrl_host()
        assert c["step"] == applied and c["loss_scale"] == ls
        cur = c["cur"]
        ref.compare(to_np(master[cur]), to_np(m[cur]), to_np(v[cur]), f16_bits(host_params),
                    what=f"host path step {step}")
    # pageable host memory is refused before any launch
    pageable = torch.zeros(n, dtype=torch.float16)
    bad = zs.Shard.from_buffer_copy(view.struct)
    bad.params = pageable.data_ptr()
    out = ctypes.c_int32(-7)
    launches = zs.zero_kernel_launches()
    rc = zs.lib().zero_shard_step_host(ctypes.byref(bad), n_d, ctypes.byref(run.hp), run.ctrl.data_ptr(), None,
                                       ctypes.byref(out))
    assert rc == zs.ZS_ERR_ARG and zs.zero_kernel_launches() == launches


def test_params_from_master_cast(zs, oracle, cuda_device):
    vals = np.concatenate([
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, -1e9, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -25,
                  1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 5.96e-8, 6.1e-5], np.float32),
        np.random.Generator(np.random.PCG64(2)).standard_normal(100003).astype(np.float32)
        * np.float32(10.0) ** np.random.Generator(np.random.PCG64(3)).uniform(-8, 4, 100003).astype(np.float32)])
    for off in (0, 1):
        master = torch.tensor(vals, device=cuda_device)
        buf = torch.zeros(vals.size + 8, dtype=torch.float16, device=cuda_device)
        params = buf[off:off + vals.size - off]
        zs.zero_params_from_master(master[off:], params, vals.size - off)
        assert np.array_equal(f16_bits(params), oracle.f32_to_f16(vals[off:]))


def test_report_max_ulp():
    """The kernel does the oracle's fp32 operations in the oracle's order with
    one rounding each, so every comparison above is expected to be exact: the
    largest ulp distance seen must be 0 (the stated bar, 1 ulp for fp16 and
    2e-6 relative for fp32, is checked element by element in each test)."""
    print("max ulp seen:", MAX_ULP)
    assert MAX_ULP["f16"] == 0 and MAX_ULP["f32"] == 0, MAX_ULP
