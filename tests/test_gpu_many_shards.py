"""The largest step the boundary accepts: ZS_MAX_SHARDS (256) shards updated
together, committed or skipped together ("DeepSpeed ZeRO Stages", sec. 2:
every rank's partition is stepped; here one device plays all of them).  The
shards have ragged sizes, empty ones included, so the commit kernel sized for
256 shards (its table passed in a large kernel-parameter block) walks every
case; an overflow in the last shard must skip and restore all 256.  Both the
asynchronous (device commit) and the synchronous entry points, and the fp16
slices against the oracle element by element."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from parity_util import OracleShard, f16_bits, oracle_group_step, to_np

pytestmark = pytest.mark.gpu


def _workload(n_d):
    return synth.Workload(name="many", numels=(1,), n_d=n_d, rank=0, align=1, steps=3, lr=1e-3, beta1=0.9,
                          beta2=0.999, eps=1e-8, weight_decay=0.01, loss_scale=1024.0, grad_dist="normal",
                          grad_std=1e-2, grad_mult=1024.0, grads_fresh_per_step=False, master_dist="normal",
                          master_param=0.02, seed=5)


def _build(zs, oracle, dev, w, sizes):
    """One fp16 parameter buffer holding every shard's slice back to back
    (each slice 16-element aligned), and per shard its contributions and two
    state sets."""
    offs = np.concatenate([[0], np.cumsum([(n + 15) // 16 * 16 for n in sizes])])
    params_full = torch.zeros(int(offs[-1]) + 16, dtype=torch.float16, device=dev)
    views, host, refs, state = [], [], [], []
    for i, n in enumerate(sizes):
        g = [synth.grad_contribution(w, n, k, 1, shard=i, device=dev) for k in range(w.n_d)]
        master0 = synth.master_init(w, n, shard=i, device=dev)
        st = ((master0, torch.zeros_like(master0)), (torch.zeros_like(master0), torch.zeros_like(master0)),
              (torch.zeros_like(master0), torch.zeros_like(master0)))
        params = params_full[int(offs[i]):int(offs[i]) + n]
        if n:
            zs.zero_params_from_master(master0, params, n)
        views.append(zs.ShardView(g, *st, params, n))
        host.append([synth.fp16_bits(t) for t in g])
        refs.append(OracleShard(oracle, to_np(master0)))
        state.append((st, params))
    return views, host, refs, state


@pytest.mark.parametrize("victim", ["first", "last"])
@pytest.mark.parametrize("path", ["async", "sync"])
def test_max_shards_one_step(zs, oracle, cuda_device, path, victim):
    """victim: the overflow is planted in the first launch of the step (shard 1)
    or in its last (the last shard); either way every shard skips."""
    rng = np.random.Generator(np.random.PCG64(21))
    sizes = [int(x) for x in rng.integers(0, 700, zs.ZS_MAX_SHARDS)]
    sizes[0], sizes[17], sizes[-1] = 0, 1, 513        # empty, single, ragged last shard
    sizes[1] = max(sizes[1], 400)
    w = _workload(3)
    views, host, refs, state = _build(zs, oracle, cuda_device, w, sizes)
    hp = zs.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    ctrl = zs.new_ctrl(cuda_device)
    zs.zero_ctrl_init(ctrl, w.loss_scale)
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    ls, applied, cur = w.loss_scale, 0, 0
    last = len(sizes) - 1 if victim == "last" else 1
    for step in range(1, 4):
        inject = step == 2
        if inject:
            keep = views[last].grads[1][300].clone()
            views[last].grads[1][300] = float("inf")
        host_step = [[synth.fp16_bits(t) for t in v.grads] for v in views] if inject else host
        before = [p.clone() for _, p in state]
        if path == "async":
            zs.zero_shard_step_async(views, w.n_d, hp, ctrl)
            torch.cuda.synchronize()
            c = zs.read_ctrl(ctrl)
            ovf = c["last_overflow"]
            cur = c["cur"]
        else:
            ovf = zs.zero_shard_step(views, w.n_d, hp, ls, applied + 1, cur, flag)
            if not ovf:
                cur ^= 1
        rovf, ls, applied = oracle_group_step(oracle, refs, host_step, w, ls, applied)
        assert ovf == rovf == int(inject)
        if path == "async":
            assert c["step"] == applied and c["loss_scale"] == ls
        if inject:
            for (st, p), b in zip(state, before):
                assert torch.equal(p, b)                     # every slice restored
            views[last].grads[1][300] = keep
        for i, ((st, p), ref) in enumerate(zip(state, refs)):
            if sizes[i] == 0:
                continue
            ref.compare(to_np(st[0][cur]), to_np(st[1][cur]), to_np(st[2][cur]), f16_bits(p),
                        what=f"{path} shard {i} step {step}")
