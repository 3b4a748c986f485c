"""ZS_MATH_FAST against the oracle (which does every division in IEEE fp32).

The fast mode changes only how u = mh / (sqrt(vh) + eps) is divided (a
corrected hardware reciprocal instead of the IEEE divide; "DeepSpeed ZeRO
Stages", sec. 2.1, Fact 1 gives the update without fixing its rounding), so:
  - the overflow flag, the skip and the bookkeeping are bit-exact;
  - m and v involve no division and stay bit-exact;
  - master is within |a - b| <= 1e-9 + 2e-6 |b| after every step, params
    within 1 fp16 ulp (the stated bar);
  - the host-resolved (synchronous) and device-resolved (asynchronous)
    coefficients give the same bits;
  - kernels that do not take the permission (run-time N_d 16-element layout,
    scalar layout) stay bit-exact.
Sizes span several tiles and ragged tails; N_d covers the 8-element layout
(1, 3, 4), the compiled-N_d 16-element layout (16, 64) and the run-time one
(8)."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner
from parity_util import ATOL, RTOL, OracleShard, f16_bits, oracle_group_step, to_np

pytestmark = pytest.mark.gpu

WORST = {"ratio": 0.0}   # largest |got - want| / (ATOL + RTOL |want|) seen on master


def _workload(n, n_d, **kw):
    base = dict(name="case", numels=(n * n_d,), n_d=n_d, rank=0, align=1, steps=3, lr=1e-3, beta1=0.9,
                beta2=0.999, eps=1e-8, weight_decay=0.0, loss_scale=1024.0, grad_dist="normal",
                grad_std=1e-2, grad_mult=1024.0, grads_fresh_per_step=True, master_dist="normal",
                master_param=0.02, seed=n * 17 + n_d)
    base.update(kw)
    return synth.Workload(**base)


def _bits(ts):
    return [synth.fp16_bits(t) for t in ts]


def _check(ref, master, m, v, params, what, exact):
    got = to_np(master)
    ref.compare(got, to_np(m), to_np(v), f16_bits(params), what=what)
    assert np.array_equal(to_np(m).view(np.uint32), ref.m.view(np.uint32)), f"{what}: m not bit-exact"
    assert np.array_equal(to_np(v).view(np.uint32), ref.v.view(np.uint32)), f"{what}: v not bit-exact"
    if exact:
        assert np.array_equal(got.view(np.uint32), ref.master.view(np.uint32)), f"{what}: master not bit-exact"
        assert np.array_equal(f16_bits(params), ref.params), f"{what}: params not bit-exact"
    want = ref.master.astype(np.float64)
    ratio = np.abs(got.astype(np.float64) - want) / (ATOL + RTOL * np.abs(want))
    WORST["ratio"] = max(WORST["ratio"], float(ratio.max()) if ratio.size else 0.0)


def _run_fast(zs, oracle, dev, w, steps=3, exact=False):
    run = WorkloadRunner(w, dev, math=zs.ZS_MATH_FAST)
    r = run.shard_ids[0]
    ref = OracleShard(oracle, to_np(run.state[r][0][0][:run.n_valid[r]]))
    ls, applied = w.loss_scale, 0
    for step in range(1, steps + 1):
        if step > 1:
            run.refresh_grads(step)
        host = [_bits([g[:run.n_valid[r]] for g in run.grads[r]])]
        run.step()
        torch.cuda.synchronize()
        ovf, ls, applied = oracle_group_step(oracle, [ref], host, w, ls, applied)
        assert ovf == 0
        n = run.n_valid[r]
        master, m, v, params = run.current(r)
        _check(ref, master[:n], m[:n], v[:n], params[:n], f"n={n} n_d={w.n_d} step={step}", exact)
    return run


@pytest.mark.parametrize("n", [1, 7, 9, 2047, 2048 * 3 + 5, 65536 + 3, 262144])
@pytest.mark.parametrize("n_d", [1, 3, 4, 16, 64])
def test_fast_mode_within_tolerance(zs, oracle, cuda_device, n, n_d):
    w = _workload(n, n_d, weight_decay=0.1 if n % 2 else 0.0,
                  loss_scale=float(2 ** 10) if n_d <= 4 else float(2 ** 14),
                  grad_mult=float(2 ** 10) if n_d <= 4 else float(2 ** 14))
    _run_fast(zs, oracle, cuda_device, w)


def test_fast_mode_not_taken_is_bit_exact(zs, oracle, cuda_device):
    """N_d = 8 runs the run-time-N_d 16-element kernel, which keeps the IEEE
    divisions: bit-exact although the permission is given."""
    w = _workload(4096 * 3 + 7, 8, loss_scale=float(2 ** 14), grad_mult=float(2 ** 14))
    _run_fast(zs, oracle, cuda_device, w, exact=True)


def test_fast_sync_equals_async(zs, cuda_device):
    """Host-resolved coefficients (zero_shard_step) and device-resolved ones
    (zero_shard_step_async) give the same bits in the fast mode."""
    n, n_d = 2048 * 9 + 3, 4
    w = _workload(n, n_d, grads_fresh_per_step=False)
    a = WorkloadRunner(w, cuda_device, math=zs.ZS_MATH_FAST)
    b = WorkloadRunner(w, cuda_device, math=zs.ZS_MATH_FAST)
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    cur = 0
    for step in range(1, 5):
        a.step()
        ovf = zs.zero_shard_step(b.views, n_d, b.hp, w.loss_scale, step, cur, flag)
        assert ovf == 0
        cur ^= 1
    torch.cuda.synchronize()
    r = a.shard_ids[0]
    ma, mb = a.current(r), b.state[r]
    for x, y in zip(ma[:3], (mb[0][cur], mb[1][cur], mb[2][cur])):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert torch.equal(ma[3].view(torch.int16), mb[3].view(torch.int16))


def test_fast_overflow_skips(zs, oracle, cuda_device):
    n, n_d = 2048 * 5 + 6, 4
    w = _workload(n, n_d, loss_scale=2.0 ** 16, grad_mult=2.0 ** 16, grads_fresh_per_step=False)
    run = WorkloadRunner(w, cuda_device, math=zs.ZS_MATH_FAST)
    r = run.shard_ids[0]
    ref = OracleShard(oracle, to_np(run.state[r][0][0]))
    host = [_bits(run.grads[r])]
    ls, applied = w.loss_scale, 0
    for step in range(1, 5):
        inject = step == 2
        if inject:
            saved = run.grads[r][1][n - 3].clone()
            run.grads[r][1][n - 3] = float("inf")
            host_step = [_bits(run.grads[r])]
        else:
            host_step = host
        before = [t.clone() for t in run.current(r)]
        run.step()
        torch.cuda.synchronize()
        ovf, ls, applied = oracle_group_step(oracle, [ref], host_step, w, ls, applied)
        c = run.ctrl_host()
        assert c["last_overflow"] == ovf == int(inject) and c["loss_scale"] == ls and c["step"] == applied
        if inject:
            for x, y in zip(before, run.current(r)):
                assert torch.equal(x, y)
            run.grads[r][1][n - 3] = saved
        _check(ref, *run.current(r), what=f"step {step}", exact=False)


def test_fast_mode_ignored_by_scalar_layout(zs, oracle, cuda_device):
    """The scalar layout (misaligned buffers) keeps the IEEE divisions:
    bit-exact with the permission given."""
    n, n_d = 5000, 3
    w = _workload(n, n_d)
    contribs = [synth.grad_contribution(w, n, k, 1) for k in range(n_d)]
    master0 = synth.master_init(w, n)
    ref = OracleShard(oracle, master0.numpy())
    oracle_group_step(oracle, [ref], [_bits(contribs)], w, w.loss_scale, 0)
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    hp = zs.adam(w.lr, math=zs.ZS_MATH_FAST)
    off = 1   # every buffer one element off its 16-byte boundary
    g = [torch.zeros(n + 16, dtype=torch.float16, device=cuda_device)[off:off + n].copy_(c.to(cuda_device))
         for c in contribs]
    mk = lambda: torch.zeros(n + 16, dtype=torch.float32, device=cuda_device)[off:off + n]
    master = (mk().copy_(master0.to(cuda_device)), mk())
    m, v = (mk(), mk()), (mk(), mk())
    params = torch.zeros(n + 16, dtype=torch.float16, device=cuda_device)[off:off + n]
    view = zs.ShardView(g, master, m, v, params, n)
    assert zs.zero_shard_step([view], n_d, hp, w.loss_scale, 1, 0, flag) == 0
    _check(ref, master[1], m[1], v[1], params, "scalar", exact=True)


def test_report_worst_ratio():
    """Prints the largest error seen on master as a fraction of the tolerance."""
    print(f"\nZS_MATH_FAST: largest |master - oracle| / (1e-9 + 2e-6 |oracle|) = {WORST['ratio']:.4f}")
    assert WORST["ratio"] <= 1.0
