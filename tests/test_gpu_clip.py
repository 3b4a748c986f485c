"""Parity of the clipped step (global gradient-norm clipping, two passes
around the squared norm) with the oracle: both pass-2 variants (re-reduce and
kept g), the three access widths, clipping active / inactive / disabled, a
multi-shard step whose norm spans every shard, an overflow during a clipped
step, and two full-size workloads checked on sampled elements."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner
from parity_util import OracleShard, f16_bits, to_np

pytestmark = pytest.mark.gpu


def _workload(n, n_d, **kw):
    base = dict(name="clip", numels=(n * n_d,), n_d=n_d, rank=0, align=1, steps=3, lr=1e-3, beta1=0.9,
                beta2=0.999, eps=1e-8, weight_decay=0.05, loss_scale=1024.0, grad_dist="normal",
                grad_std=1e-2, grad_mult=1024.0, grads_fresh_per_step=True, master_dist="normal",
                master_param=0.02, seed=n + 7 * n_d)
    base.update(kw)
    return synth.Workload(**base)


def _oracle_clipped_group(oracle, refs, host, w, loss_scale, applied, max_norm):
    """One oracle step of several shards that share one norm and one commit."""
    reduced, ovf, sq = [], 0, 0.0
    for ref, contribs in zip(refs, host):
        g, bad = ref.reduce(contribs, loss_scale)
        reduced.append(g)
        ovf |= bad
        sq = oracle.grad_sqnorm(g, sq)
    c = oracle.clip_factor(sq, max_norm)
    if not ovf:
        for ref, g in zip(refs, reduced):
            oracle.scale(g, c)
            ref.apply(g, w, applied + 1)
    loss_scale, applied = oracle.commit(ovf, loss_scale, applied)
    return ovf, loss_scale, applied, sq, c


def _sq_close(got, want, n):
    """The oracle sums n squares one after another in double: its own error is
    at most (n - 1) 2^-53 of the sum; the kernel's compensated sum is far
    tighter.  So they agree within 2 n 2^-53 relative (floor 1e-13)."""
    tol = max(1e-13, 2.0 * n * 2.0 ** -53)
    assert abs(got - want) <= tol * want, (got, want, tol)


def _bits(run, r):
    n = run.n_valid[r]
    return [synth.fp16_bits(g[:n]) for g in run.grads[r]]


def _compare(run, refs, what):
    for ref, r in zip(refs, run.shard_ids):
        n = run.n_valid[r]
        master, m, v, params = run.current(r)
        ref.compare(to_np(master[:n]), to_np(m[:n]), to_np(v[:n]), f16_bits(params[:n]), what=f"{what} shard {r}")


@pytest.mark.parametrize("n,n_d", [(2048 * 5 + 3, 4), (4099, 8), (20000, 16), (777, 64), (5000, 3)])
@pytest.mark.parametrize("keep_g", [False, True])
@pytest.mark.parametrize("max_norm_kind", ["active", "inactive", "off"])
@pytest.mark.parametrize("math", ["ieee", "fast"])
def test_clipped_step_matches_oracle(zs, oracle, cuda_device, n, n_d, keep_g, max_norm_kind, math):
    """math = fast: ZS_MATH_FAST, the same tolerance; m and v stay bit-exact."""
    w = _workload(n, n_d)
    run = WorkloadRunner(w, cuda_device, math=zs.ZS_MATH_FAST if math == "fast" else zs.ZS_MATH_IEEE)
    run.enable_clipping(keep_g)
    r = run.shard_ids[0]
    refs = [OracleShard(oracle, to_np(run.state[r][0][0]))]
    # the scaled-out gradient has norm ~ 1e-2 * sqrt(n * n_d) / sqrt(n_d)
    g0, _ = oracle.grad_reduce(_bits(run, r), w.loss_scale)
    norm0 = float(np.sqrt(oracle.grad_sqnorm(g0)))
    max_norm = {"active": 0.3 * norm0, "inactive": 10.0 * norm0, "off": 0.0}[max_norm_kind]
    ls, applied = w.loss_scale, 0
    for step in range(1, 4):
        if step > 1:
            run.refresh_grads(step)
        host = [_bits(run, r)]
        run.step_clipped(max_norm)
        torch.cuda.synchronize()
        ovf, ls, applied, sq, c = _oracle_clipped_group(oracle, refs, host, w, ls, applied, max_norm)
        assert ovf == 0
        _sq_close(float(run.sqnorm.item()), sq, n)
        if max_norm_kind == "active":
            assert c < 1.0
        else:
            assert c == 1.0
        assert run.ctrl_host()["step"] == applied
        _compare(run, refs, f"{math} step {step}")
        _, m, v, _ = run.current(r)
        assert np.array_equal(to_np(m[:n]).view(np.uint32), refs[0].m.view(np.uint32))
        assert np.array_equal(to_np(v[:n]).view(np.uint32), refs[0].v.view(np.uint32))


@pytest.mark.parametrize("n_d,math", [(8, "ieee"), (4, "ieee"), (4, "fast"), (16, "fast")])
def test_clip_off_equals_unclipped_step(zs, cuda_device, n_d, math):
    """max_norm <= 0: the clipped step is the plain step, bit for bit, in
    either arithmetic mode."""
    n = 2048 * 3 + 1
    w = _workload(n, n_d, grads_fresh_per_step=False)
    mode = zs.ZS_MATH_FAST if math == "fast" else zs.ZS_MATH_IEEE
    a, b = WorkloadRunner(w, cuda_device, math=mode), WorkloadRunner(w, cuda_device, math=mode)
    b.enable_clipping(True)
    for _ in range(3):
        a.step()
        b.step_clipped(0.0)
    torch.cuda.synchronize()
    for x, y in zip(a.current(0), b.current(0)):
        assert torch.equal(x, y)


@pytest.mark.parametrize("keep_g", [False, True])
def test_clipped_multi_shard_norm_spans_all_shards(zs, oracle, cuda_device, keep_g):
    numels = tuple(synth.ragged_numels(80, seed=11, max_exp=12))
    w = _workload(0, 16, numels=numels, rank=None, align=128, grads_fresh_per_step=False, grad_dist="laplace",
                  grad_std=5e-4, grad_mult=2.0 ** 14, loss_scale=2.0 ** 14, master_dist="uniform",
                  master_param=0.05, seed=3)
    run = WorkloadRunner(w, cuda_device)
    run.enable_clipping(keep_g)
    refs = [OracleShard(oracle, to_np(run.state[r][0][0][: run.n_valid[r]])) for r in run.shard_ids]
    host = [_bits(run, r) for r in run.shard_ids]
    sq0 = 0.0
    for ref, h in zip(refs, host):
        g, _ = ref.reduce(h, w.loss_scale)
        sq0 = oracle.grad_sqnorm(g, sq0)
    max_norm = 0.5 * float(np.sqrt(sq0))
    ls, applied = w.loss_scale, 0
    victim = run.shard_ids[4]
    for step in range(1, 5):
        inject = step == 2
        if inject:
            run.grads[victim][3][1] = float("inf")
        host = [_bits(run, r) for r in run.shard_ids]
        run.step_clipped(max_norm)
        torch.cuda.synchronize()
        ovf, ls, applied, sq, c = _oracle_clipped_group(oracle, refs, host, w, ls, applied, max_norm)
        assert ovf == int(inject) == run.ctrl_host()["last_overflow"]
        if inject:
            run.grads[victim][3][1] = 0.0
        else:
            _sq_close(float(run.sqnorm.item()), sq, sum(run.n_valid.values()))
            assert c < 1.0
        assert run.ctrl_host()["step"] == applied
        _compare(run, refs, f"step {step}")


def test_clip_passes_called_separately(zs, oracle, cuda_device):
    """The two passes through their own entry points (as a multi-rank caller
    uses them, with its all-reduce in between) equal the composite call."""
    n, n_d = 3001, 4
    w = _workload(n, n_d, grads_fresh_per_step=False)
    a, b = WorkloadRunner(w, cuda_device), WorkloadRunner(w, cuda_device)
    a.enable_clipping(False)
    b.enable_clipping(False)
    g_keep = torch.zeros(a.S, dtype=torch.float32, device=cuda_device)
    for _ in range(2):
        a.step_clipped(0.01)
        b.sqnorm.zero_()
        zs.zero_shard_grad_sqnorm_async(b.views[0], n_d, b.sqnorm, b.ctrl, g_dev=g_keep)
        zs.zero_shard_clipped_adam_async(b.views[0], n_d, b.hp, 0.01, b.sqnorm, b.ctrl, g_dev=g_keep)
        zs.zero_step_commit_async(b.views, b.hp, b.ctrl)
    torch.cuda.synchronize()
    for x, y in zip(a.current(0), b.current(0)):
        assert torch.equal(x, y)


@pytest.mark.parametrize("name,keep_g", [("gpt2s", True), ("xl", False)])
def test_clipped_full_size_sampled(zs, oracle, cuda_device, name, keep_g):
    w = synth.WORKLOADS[name]
    run = WorkloadRunner(w, cuda_device)
    run.enable_clipping(keep_g)
    r = run.shard_ids[0]
    n = run.n_valid[r]
    idx = torch.tensor(synth.sample_indices(n, 40000, seed=77), device=cuda_device)
    ref = OracleShard(oracle, to_np(run.state[r][0][0][idx]))
    ls, applied = w.loss_scale, 0
    g_full = None
    for step in range(1, 4):
        if w.grads_fresh_per_step and step > 1:
            run.refresh_grads(step)
        if g_full is None or w.grads_fresh_per_step:
            full = _bits(run, r)                   # the norm needs every element
            g_full, bad = oracle.grad_reduce(full, ls)
            del full
            sq = oracle.grad_sqnorm(g_full)
        max_norm = 0.5 * float(np.sqrt(sq))
        c = oracle.clip_factor(sq, max_norm)
        run.step_clipped(max_norm)
        torch.cuda.synchronize()
        assert bad == 0
        _sq_close(float(run.sqnorm.item()), sq, n)
        g = g_full[idx.cpu().numpy()].copy()
        oracle.scale(g, c)
        ref.apply(g, w, applied + 1)
        applied += 1
        master, m, v, params = run.current(r)
        ref.compare(to_np(master[idx]), to_np(m[idx]), to_np(v[idx]), f16_bits(params[idx]),
                    what=f"{name} clipped step {step}")
