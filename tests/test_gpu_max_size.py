"""A shard past the 32-bit index range: n = 2^31 + 777 parameters (N_d = 2,
about 65 GB of contributions, state and parameters on the 288 GB part).
Every index the kernels form is 64-bit; elements on both sides of 2^31, the
ragged tail and random positions are compared with the oracle after two
steps, and an infinity planted above 2^31 must skip the third."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner
from parity_util import OracleShard, f16_bits, oracle_group_step, to_np

pytestmark = pytest.mark.gpu

N = (1 << 31) + 777


def test_shard_beyond_int32(zs, oracle, cuda_device):
    free, _ = torch.cuda.mem_get_info(cuda_device)
    if free < 80 * (1 << 30):
        pytest.skip("needs about 80 GB of free device memory")
    w = synth.Workload(name="max", numels=(2 * N,), n_d=2, rank=1, align=1, steps=3, lr=1e-3, beta1=0.9,
                       beta2=0.999, eps=1e-8, weight_decay=0.01, loss_scale=1024.0, grad_dist="normal",
                       grad_std=1e-2, grad_mult=1024.0, grads_fresh_per_step=False, master_dist="normal",
                       master_param=0.02, seed=31)
    run = WorkloadRunner(w, cuda_device, with_full_params=False)
    r = run.shard_ids[0]
    assert run.n_valid[r] == N
    rng = np.random.Generator(np.random.PCG64(7))
    idx = np.unique(np.concatenate([
        np.arange(0, 300), np.arange((1 << 31) - 300, (1 << 31) + 300), np.arange(N - 300, N),
        rng.integers(0, N, 4000), [(1 << 31) + 12345]]).astype(np.int64))
    idx = idx[idx < N]
    sel = torch.tensor(idx, device=cuda_device)
    ref = OracleShard(oracle, to_np(run.state[r][0][0][sel]))
    host = [[synth.fp16_bits(g[sel]) for g in run.grads[r]]]
    ls, applied = w.loss_scale, 0
    for step in (1, 2):
        run.step()
        torch.cuda.synchronize()
        ovf, ls, applied = oracle_group_step(oracle, [ref], host, w, ls, applied)
        assert ovf == 0 and run.ctrl_host()["step"] == applied
        master, m, v, params = run.current(r)
        ref.compare(to_np(master[sel]), to_np(m[sel]), to_np(v[sel]), f16_bits(params[sel]),
                    what=f"n = 2^31 + 777, step {step}")
    # an overflow planted above 2^31 skips the step and leaves the state as it was
    j = (1 << 31) + 500
    before = [t[sel].clone() for t in run.current(r)]
    run.grads[r][1][j] = float("inf")
    run.step()
    torch.cuda.synchronize()
    c = run.ctrl_host()
    assert c["last_overflow"] == 1 and c["skipped"] == 1 and c["step"] == applied
    for a, b in zip(before, run.current(r)):
        assert torch.equal(a, b[sel])
