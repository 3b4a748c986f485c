"""Element-by-element parity with the oracle past one sweep of the persistent
grid, in both arithmetic modes, with an overflow step in the middle.

The fused kernels run a persistent grid: one pass of the grid covers
blocks x 256 threads x VEC elements, at most 152 SMs x 2048 resident threads
x 8 = 2.49M elements for the 8-element kernel and, with its two resident
blocks per SM, 152 x 512 x 16 = 1.25M for the 16-element ones.  The shards
here hold 4-8M elements, so every thread walks the grid-stride loop several
times, and every element of every state array is compared (m and v bit for
bit in both modes; master within the stated tolerance, params within one fp16
ulp, both exact in the IEEE mode):

  - the 8-element kernel with a run-time N_d (N_d = 4, the 1.5B workload's);
  - the 16-element kernels compiled for N_d = 16, 32 and 64;
  - the 16-element kernel with a run-time N_d (N_d = 17);
  - the grouped kernel over the four shards of a ragged tensor list
    (shard boundaries inside tensors, one launch walking all of them);
  - the GPT-2-small workload at full size (15.5M elements, N_d = 8, fresh
    gradients every step) for its 10 steps.
"""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner
from parity_util import OracleShard, f16_bits, oracle_group_step, to_np

pytestmark = pytest.mark.gpu


def _workload(n, n_d, **kw):
    base = dict(name="sweep", numels=(n * n_d,), n_d=n_d, rank=0, align=1, steps=4, lr=1e-3, beta1=0.9,
                beta2=0.999, eps=1e-8, weight_decay=0.05, loss_scale=2048.0, grad_dist="normal",
                grad_std=1e-3, grad_mult=2048.0, grads_fresh_per_step=True, master_dist="normal",
                master_param=0.02, seed=7 * n + n_d)
    base.update(kw)
    return synth.Workload(**base)


def _run_and_compare(zs, oracle, dev, w, math, inject_at, what):
    """Step every stepped shard of w for w.steps steps through
    zero_shard_step_async; at step inject_at[0] put +inf into contribution
    inject_at[1] of the first stepped shard at element inject_at[2] (for that
    step only); compare every element with the oracle after every step."""
    run = WorkloadRunner(w, dev, math=zs.ZS_MATH_FAST if math == "fast" else zs.ZS_MATH_IEEE)
    refs = [OracleShard(oracle, to_np(run.state[r][0][0][:run.n_valid[r]])) for r in run.shard_ids]
    ls, applied = w.loss_scale, 0
    r0 = run.shard_ids[0]
    for step in range(1, w.steps + 1):
        if w.grads_fresh_per_step and step > 1:
            run.refresh_grads(step)
        inject = inject_at is not None and step == inject_at[0]
        if inject:
            saved = run.grads[r0][inject_at[1]][inject_at[2]].clone()
            run.grads[r0][inject_at[1]][inject_at[2]] = float("inf")
        host = [[synth.fp16_bits(g[:run.n_valid[r]]) for g in run.grads[r]] for r in run.shard_ids]
        run.step()
        torch.cuda.synchronize()
        if inject:                     # gradients drawn once stay in place for the next step
            run.grads[r0][inject_at[1]][inject_at[2]] = saved
        ovf, ls, applied = oracle_group_step(oracle, refs, host, w, ls, applied)
        assert ovf == int(inject), (what, step)
        c = run.ctrl_host()
        assert c["last_overflow"] == ovf and c["loss_scale"] == ls and c["step"] == applied, (what, step, c)
        for ref, r in zip(refs, run.shard_ids):
            n = run.n_valid[r]
            master, m, v, params = run.current(r)
            gm, gv = to_np(m[:n]), to_np(v[:n])
            ref.compare(to_np(master[:n]), gm, gv, f16_bits(params[:n]), what=f"{what} shard {r} step {step}")
            assert np.array_equal(gm.view(np.uint32), ref.m.view(np.uint32)), (what, r, step)
            assert np.array_equal(gv.view(np.uint32), ref.v.view(np.uint32)), (what, r, step)
            if math == "ieee":
                assert np.array_equal(to_np(master[:n]).view(np.uint32), ref.master.view(np.uint32))
                assert np.array_equal(f16_bits(params[:n]), ref.params)
    if inject_at is not None:
        assert run.ctrl_host()["skipped"] == 1


@pytest.mark.parametrize("math", ["ieee", "fast"])
@pytest.mark.parametrize("n_d,n", [(4, 8_000_013), (16, 8_000_011), (32, 6_000_007), (64, 4_000_037),
                                   (17, 8_000_019)])
def test_every_element_past_grid_sweeps(zs, oracle, cuda_device, n_d, n, math):
    w = _workload(n, n_d)
    _run_and_compare(zs, oracle, cuda_device, w, math, (2, n_d // 2, n - 3), f"n_d={n_d} n={n} {math}")


@pytest.mark.parametrize("math", ["ieee", "fast"])
def test_grouped_ragged_shards_every_element(zs, oracle, cuda_device, math):
    """A ragged tensor list cut into four 128-aligned shards, all stepped in
    one grouped launch (shard boundaries fall inside tensors); the +inf goes
    into the middle of shard 0 and skips the step of all four."""
    numels = synth.ragged_numels(n=140, seed=11)
    w = _workload(1, 4, name="ragged-sweep", numels=tuple(numels), rank=None, align=128, steps=4,
                  grads_fresh_per_step=False, grad_dist="laplace", grad_std=5e-4, seed=11)
    lay = zs.zero_partition_layout(w.numels, w.n_d, w.align)
    s = int(lay["shard_numel"])
    assert s > 2_000_000 and int(lay["psi"]) > 3 * s        # four shards, each past a grid sweep
    _run_and_compare(zs, oracle, cuda_device, w, math, (3, 1, s // 2 + 1), f"ragged 4 shards {math}")


@pytest.mark.parametrize("math", ["fast", "ieee"])
def test_gpt2s_full_size_every_element(zs, oracle, cuda_device, math):
    w = synth.WORKLOADS["gpt2s"]
    _run_and_compare(zs, oracle, cuda_device, w, math, None, f"gpt2s {math}")
