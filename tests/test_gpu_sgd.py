"""Parity of the SGD-with-momentum shard step with the oracle (bit-exact):
narrow / wide / compile-time-N_d layouts, ragged tails, an overflow step
that is skipped (state, momentum and fp16 slice unchanged, loss scale
halved), a multi-shard step, and a full-size workload on sampled elements."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner
from parity_util import assert_f16_close, assert_f32_close, f16_bits, to_np

pytestmark = pytest.mark.gpu

MU, LR, WD = 0.9, 0.01, 1e-3


def _workload(n, n_d, **kw):
    base = dict(name="sgd", numels=(n * n_d,), n_d=n_d, rank=0, align=1, steps=3, lr=LR, beta1=0.9, beta2=0.999,
                eps=1e-8, weight_decay=WD, loss_scale=1024.0, grad_dist="normal", grad_std=1e-2, grad_mult=1024.0,
                grads_fresh_per_step=True, master_dist="normal", master_param=0.02, seed=n + 5 * n_d)
    base.update(kw)
    return synth.Workload(**base)


class OracleSgd:
    def __init__(self, oracle, master0):
        self.o = oracle
        self.master = np.array(master0, np.float32)
        self.mom = np.zeros_like(self.master)
        self.params = oracle.f32_to_f16(self.master)

    def step(self, contribs, loss_scale):
        g, bad = self.o.grad_reduce(contribs, loss_scale, n=self.master.size)
        if not bad:
            self.o.sgd_apply(g, self.master, self.mom, self.params, lr=LR, momentum=MU, weight_decay=WD)
        return bad


def _compare(run, r, ref, what):
    n = run.n_valid[r]
    master, mom, _, params = run.current(r)
    assert_f32_close(to_np(master[:n]), ref.master, what + " master")
    assert_f32_close(to_np(mom[:n]), ref.mom, what + " momentum")
    assert_f16_close(f16_bits(params[:n]), ref.params, what + " params")


@pytest.mark.parametrize("n", [1, 2049, 65536 + 13])
@pytest.mark.parametrize("n_d", [1, 4, 8, 16, 64, 5])
def test_sgd_step_matches_oracle(zs, oracle, cuda_device, n, n_d):
    w = _workload(n, n_d)
    run = WorkloadRunner(w, cuda_device)
    r = run.shard_ids[0]
    ref = OracleSgd(oracle, to_np(run.state[r][0][0]))
    hp = zs.sgd(LR, MU, WD)
    ls = w.loss_scale
    for step in range(1, 5):
        if step > 1:
            run.refresh_grads(step)
        inject = step == 3 and n > 1
        if inject:
            run.grads[r][0][n - 1] = float("-inf")
        host = [synth.fp16_bits(g[:n]) for g in run.grads[r]]
        before = [t.clone() for t in run.current(r)] if inject else None
        run.step_sgd(hp)
        torch.cuda.synchronize()
        bad = ref.step(host, ls)
        c = run.ctrl_host()
        assert c["last_overflow"] == bad == int(inject)
        if bad:
            ls = max(ls / 2, 1.0)
            for a, b in zip(before, run.current(r)):
                assert torch.equal(a, b)
        assert c["loss_scale"] == ls
        _compare(run, r, ref, f"n={n} n_d={n_d} step {step}")


@pytest.mark.parametrize("n_d", [8, 16, 20])
def test_sgd_multi_shard(zs, oracle, cuda_device, n_d):
    """Every shard of a ragged tensor list in one step: grouped launches (up to
    16 shards each; 20 shards make a group of 16 and one of 4)."""
    numels = tuple(synth.ragged_numels(60, seed=4, max_exp=11))
    w = _workload(0, n_d, numels=numels, rank=None, align=128, grads_fresh_per_step=False, seed=9)
    run = WorkloadRunner(w, cuda_device)
    refs = {r: OracleSgd(oracle, to_np(run.state[r][0][0][: run.n_valid[r]])) for r in run.shard_ids}
    hp = zs.sgd(LR, MU, WD)
    for step in range(1, 4):
        run.step_sgd(hp)
        torch.cuda.synchronize()
        for r in run.shard_ids:
            n = run.n_valid[r]
            assert refs[r].step([synth.fp16_bits(g[:n]) for g in run.grads[r]], w.loss_scale) == 0
            _compare(run, r, refs[r], f"shard {r} step {step}")


def test_sgd_full_size_sampled(zs, oracle, cuda_device):
    w = synth.WORKLOADS["7b5"]
    run = WorkloadRunner(w, cuda_device)
    r = run.shard_ids[0]
    idx = torch.tensor(synth.sample_indices(run.n_valid[r], 50000, seed=5), device=cuda_device)
    ref = OracleSgd(oracle, to_np(run.state[r][0][0][idx]))
    hp = zs.sgd(LR, MU, WD)
    host = [synth.fp16_bits(g[idx]) for g in run.grads[r]]
    for step in range(1, 3):
        run.step_sgd(hp)
        torch.cuda.synchronize()
        assert ref.step(host, w.loss_scale) == 0
        master, mom, _, params = run.current(r)
        assert_f32_close(to_np(master[idx]), ref.master, f"7b5 sgd step {step} master")
        assert_f32_close(to_np(mom[idx]), ref.mom, f"7b5 sgd step {step} momentum")
        assert_f16_close(f16_bits(params[idx]), ref.params, f"7b5 sgd step {step} params")
