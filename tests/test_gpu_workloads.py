"""The five workloads at their full sizes, run exactly as the benchmark runs
them (device layout, one fused kernel per shard, device-side commit), checked
against the oracle on sampled elements (every element for the tiny workload),
with the properties that hold at any size checked on the whole buffers:
the overflow flag, the loss-scale and step bookkeeping, and an overflow step
leaving the committed state and fp16 slice bit-identical."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner
from parity_util import OracleShard, f16_bits, oracle_group_step, to_np

pytestmark = pytest.mark.gpu


def _gather_bits(ts, idx_dev):
    return [synth.fp16_bits(t[idx_dev]) for t in ts]


@pytest.mark.parametrize("math", ["ieee", "fast"])
@pytest.mark.parametrize("name", ["tiny", "gpt2s", "ragged", "xl", "7b5"])
def test_workload_full_size(zs, oracle, cuda_device, name, math):
    """math = fast runs ZS_MATH_FAST, as the benchmark does: the same bar
    (master within tolerance, params within 1 fp16 ulp), and m, v bit-exact
    (they involve no division)."""
    w = synth.WORKLOADS[name]
    run = WorkloadRunner(w, cuda_device, math=zs.ZS_MATH_FAST if math == "fast" else zs.ZS_MATH_IEEE)
    samples, refs = {}, []
    for r in run.shard_ids:
        n = run.n_valid[r]
        if n <= (1 << 21):
            idx = np.arange(n, dtype=np.int64)
        else:
            idx = synth.sample_indices(n, 60000, seed=1000 + r)
            if w.inf_at is not None:
                idx = np.unique(np.append(idx, w.inf_at[2]))
        samples[r] = torch.tensor(idx, device=cuda_device)
        refs.append(OracleShard(oracle, to_np(run.state[r][0][0][samples[r]])))
    ls, applied = w.loss_scale, 0
    for step in range(1, w.steps + 1):
        if w.grads_fresh_per_step and step > 1:
            run.refresh_grads(step)
        inject = w.inf_at is not None and step == w.inf_at[0]
        if inject:
            _, k, j = w.inf_at
            saved_val = run.grads[run.shard_ids[0]][k][j].clone()
            run.grads[run.shard_ids[0]][k][j] = float("inf")
        for r in run.shard_ids:
            finite = all(bool(torch.isfinite(g).all()) for g in run.grads[r])
            assert finite != inject
        host = [_gather_bits(run.grads[r], samples[r]) for r in run.shard_ids]
        if inject:
            before = [[t.clone() for t in run.current(r)] for r in run.shard_ids]
        run.step()
        torch.cuda.synchronize()
        ovf, ls, applied = oracle_group_step(oracle, refs, host, w, ls, applied)
        assert ovf == int(inject)
        c = run.ctrl_host()
        assert c["last_overflow"] == ovf and c["loss_scale"] == ls and c["step"] == applied
        assert c["overflow"] == 0 and c["arrivals"] == 0
        if inject:
            for r, b in zip(run.shard_ids, before):
                for x, y in zip(b, run.current(r)):
                    assert torch.equal(x, y)
            run.grads[run.shard_ids[0]][k][j] = saved_val
        for ref, r in zip(refs, run.shard_ids):
            master, m, v, params = run.current(r)
            i = samples[r]
            ref.compare(to_np(master[i]), to_np(m[i]), to_np(v[i]), f16_bits(params[i]),
                        what=f"{name} {math} shard {r} step {step}")
            assert np.array_equal(to_np(m[i]).view(np.uint32), ref.m.view(np.uint32))
            assert np.array_equal(to_np(v[i]).view(np.uint32), ref.v.view(np.uint32))
    if w.inf_at is not None:
        assert run.ctrl_host()["skipped"] == 1 and ls == w.loss_scale / 2
