"""Grouped launches: consecutive shards with one access width (all with or
all without a qwZ copy) are stepped up to 16 at a time by one launch that
walks their concatenated elements (zero_shard_reduce_adam_all_async, and inside zero_shard_step_async
and zero_shard_step).  The result must be bit-identical to one launch per
shard (zero_shard_reduce_adam_async), and equal to the oracle, for groups cut
by a misaligned shard, by a shard with a qwZ copy and by the 16-shard limit,
with empty shards, tails shorter than a vector, both arithmetic modes and an
overflow in one shard of a group."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from parity_util import OracleShard, f16_bits, oracle_group_step, to_np

pytestmark = pytest.mark.gpu


def _workload(n_d, seed):
    return synth.Workload(name="group", numels=(1,), n_d=n_d, rank=0, align=1, steps=3, lr=1e-3, beta1=0.9,
                          beta2=0.999, eps=1e-8, weight_decay=0.01, loss_scale=2.0 ** 12, grad_dist="normal",
                          grad_std=1e-2, grad_mult=2.0 ** 12, grads_fresh_per_step=False, master_dist="normal",
                          master_param=0.02, seed=seed)


def _make(zs, dev, w, sizes, misaligned=(), qwz=()):
    """Views over fresh buffers; shard i misaligned (scalar kernel) if listed,
    with a qwZ copy if listed.  Returns views, state tuples, host contribs."""
    views, state, host = [], [], []
    for i, n in enumerate(sizes):
        off = 1 if i in misaligned else 0
        g = []
        for k in range(w.n_d):
            t = torch.zeros(n + 16, dtype=torch.float16, device=dev)[off:off + n]
            t.copy_(synth.grad_contribution(w, n, k, 1, shard=i, device=dev))
            g.append(t)
        mk = lambda: torch.zeros(n + 16, dtype=torch.float32, device=dev)[off:off + n]
        master = (mk(), mk())
        master[0].copy_(synth.master_init(w, n, shard=i, device=dev))
        m, v = (mk(), mk()), (mk(), mk())
        params = torch.zeros(n + 16, dtype=torch.float16, device=dev)[off:off + n]
        if n:
            zs.zero_params_from_master(master[0], params, n)
        q = {}
        if i in qwz:
            q = dict(qcodes=torch.zeros(n + 16, dtype=torch.int8, device=dev)[:n],
                     qscales=torch.zeros((n + 255) // 256 + 1, dtype=torch.float32, device=dev))
        views.append(zs.ShardView(g, master, m, v, params, n, **q))
        state.append((master, m, v, params))
        host.append([synth.fp16_bits(t) for t in g])
    return views, state, host


CASES = {
    "ragged_like": (16, [19_223_680 // 64] * 15 + [4099], (), ()),
    "over_16": (4, [int(x) for x in np.random.Generator(np.random.PCG64(5)).integers(0, 3000, 37)], (), ()),
    "cut_runs": (8, [2048 * 3 + 5, 4096, 0, 2048 * 2 + 1, 777, 5000, 6, 3000, 2048 * 4], (3,), (6,)),
    "tiny_tails": (64, [1, 3, 15, 17, 33, 0, 250], (), ()),
    "qwz_runs": (16, [5000, 256 * 20, 256 * 7 + 3, 1, 4099, 256 * 40, 3000], (), (0, 1, 2, 3, 4, 5)),
    "qwz_narrow": (4, [256 * 33 + 17, 700, 256 * 8, 9000, 257], (), (0, 1, 2, 3, 4)),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("math", ["ieee", "fast"])
@pytest.mark.parametrize("path", ["split", "async"])
def test_grouped_equals_per_shard_and_oracle(zs, oracle, cuda_device, case, math, path):
    """path = split: the grouped fused launches, then the commit kernel; async:
    zero_shard_step_async, whose last launch commits the step itself (the
    cases with several launches check that an overflow seen by an earlier
    launch reaches the last one's commit)."""
    n_d, sizes, misaligned, qwz = CASES[case]
    w = _workload(n_d, seed=len(sizes) + n_d)
    mode = zs.ZS_MATH_FAST if math == "fast" else zs.ZS_MATH_IEEE
    hp = zs.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, math=mode)
    va, sa, host = _make(zs, cuda_device, w, sizes, misaligned, qwz)
    vb, sb, _ = _make(zs, cuda_device, w, sizes, misaligned, qwz)
    ca, cb = zs.new_ctrl(cuda_device), zs.new_ctrl(cuda_device)
    zs.zero_ctrl_init(ca, w.loss_scale)
    zs.zero_ctrl_init(cb, w.loss_scale)
    refs = [OracleShard(oracle, to_np(st[0][0])) for st in sa]
    ls, applied = w.loss_scale, 0
    victim = max(range(len(sizes)), key=lambda i: sizes[i])
    for step in range(1, 4):
        inject = step == 2
        if inject:
            j = sizes[victim] // 2
            keep = (va[victim].grads[0][j].clone(), vb[victim].grads[0][j].clone())
            va[victim].grads[0][j] = float("inf")
            vb[victim].grads[0][j] = float("inf")
            host_step = [[synth.fp16_bits(t) for t in v.grads] for v in va]
        else:
            host_step = host
        if path == "split":
            zs.zero_shard_reduce_adam_all_async(va, n_d, hp, ca)   # grouped
            zs.zero_step_commit_async(va, hp, ca)
        else:
            zs.zero_shard_step_async(va, n_d, hp, ca)              # grouped, commit in the last launch
        for v in vb:                                                 # one launch per shard
            zs.zero_shard_reduce_adam_async(v, n_d, hp, cb)
        zs.zero_step_commit_async(vb, hp, cb)
        torch.cuda.synchronize()
        ovf, ls, applied = oracle_group_step(oracle, refs, host_step, w, ls, applied)
        c_a, c_b = zs.read_ctrl(ca), zs.read_ctrl(cb)
        assert c_a == c_b and c_a["last_overflow"] == ovf == int(inject) and c_a["step"] == applied
        if inject:
            va[victim].grads[0][j], vb[victim].grads[0][j] = keep
        cur = c_a["cur"]
        for i, ((ma, mma, vva, pa), (mb, mmb, vvb, pb), ref) in enumerate(zip(sa, sb, refs)):
            for x, y in ((ma[cur], mb[cur]), (mma[cur], mmb[cur]), (vva[cur], vvb[cur])):
                assert torch.equal(x.view(torch.int32), y.view(torch.int32)), f"{case} shard {i} step {step}"
            assert torch.equal(pa.view(torch.int16), pb.view(torch.int16)), f"{case} shard {i} step {step}"
            if sizes[i]:
                ref.compare(to_np(ma[cur]), to_np(mma[cur]), to_np(vva[cur]), f16_bits(pa),
                            what=f"{case} {math} shard {i} step {step}")
        for i in qwz:
            codes, scales = oracle.qwz_quantize(f16_bits(sa[i][3]))
            assert np.array_equal(to_np(va[i].qcodes[:sizes[i]]), codes)
            assert np.array_equal(to_np(va[i].qscales[:scales.size]).view(np.uint32), scales.view(np.uint32))
            assert torch.equal(va[i].qcodes, vb[i].qcodes)


def test_sync_step_uses_groups(zs, oracle, cuda_device):
    """zero_shard_step (host round trip) over 20 shards equals the oracle."""
    n_d = 4
    sizes = [1000 + 37 * i for i in range(20)]
    w = _workload(n_d, seed=99)
    views, state, host = _make(zs, cuda_device, w, sizes)
    refs = [OracleShard(oracle, to_np(st[0][0])) for st in state]
    flag = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    hp = zs.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    launches = zs.zero_kernel_launches()
    assert zs.zero_shard_step(views, n_d, hp, w.loss_scale, 1, 0, flag) == 0
    assert zs.zero_kernel_launches() - launches == 2          # 16 shards + 4 shards: two grouped launches
    oracle_group_step(oracle, refs, host, w, w.loss_scale, 0)
    for (master, m, v, params), ref in zip(state, refs):
        ref.compare(to_np(master[1]), to_np(m[1]), to_np(v[1]), f16_bits(params))


@pytest.mark.parametrize("keep_g", [False, True])
@pytest.mark.parametrize("case", ["ragged_like", "cut_runs", "over_16"])
def test_grouped_clip_passes_equal_per_shard(zs, cuda_device, case, keep_g):
    """Both clipping passes over a shard list (grouped launches) give the same
    flags, squared norm (to the rounding of the double additions) and bits as
    one launch per shard."""
    n_d, sizes, misaligned, qwz = CASES[case]
    w = _workload(n_d, seed=3 * len(sizes) + n_d)
    hp = zs.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, math=zs.ZS_MATH_FAST)
    va, sa, _ = _make(zs, cuda_device, w, sizes, misaligned, qwz)
    vb, sb, _ = _make(zs, cuda_device, w, sizes, misaligned, qwz)
    ga = [torch.zeros(n + 16, dtype=torch.float32, device=cuda_device)[(1 if i in misaligned else 0):][:n]
          for i, n in enumerate(sizes)] if keep_g else None
    gb = [t.clone() for t in ga] if keep_g else None
    ca, cb = zs.new_ctrl(cuda_device), zs.new_ctrl(cuda_device)
    zs.zero_ctrl_init(ca, w.loss_scale)
    zs.zero_ctrl_init(cb, w.loss_scale)
    sqa = torch.zeros(1, dtype=torch.float64, device=cuda_device)
    sqb = torch.zeros(1, dtype=torch.float64, device=cuda_device)
    for step in range(1, 3):
        sqa.zero_(); sqb.zero_()
        zs.zero_shard_grad_sqnorm_all_async(va, n_d, sqa, ca, g_dev=ga)
        for i, v in enumerate(vb):
            zs.zero_shard_grad_sqnorm_async(v, n_d, sqb, cb, g_dev=gb[i] if gb else None)
        torch.cuda.synchronize()
        a, b = float(sqa.item()), float(sqb.item())
        assert abs(a - b) <= 1e-12 * max(b, 1e-300), (a, b)
        sqa.copy_(sqb)                          # the same clip factor on both sides
        max_norm = 0.5 * np.sqrt(b)
        zs.zero_shard_clipped_adam_all_async(va, n_d, hp, max_norm, sqa, ca, g_dev=ga)
        for i, v in enumerate(vb):
            zs.zero_shard_clipped_adam_async(v, n_d, hp, max_norm, sqb, cb, g_dev=gb[i] if gb else None)
        zs.zero_step_commit_async(va, hp, ca)
        zs.zero_step_commit_async(vb, hp, cb)
        torch.cuda.synchronize()
        assert zs.read_ctrl(ca) == zs.read_ctrl(cb)
        cur = zs.read_ctrl(ca)["cur"]
        for i, ((ma, mma, vva, pa), (mb, mmb, vvb, pb)) in enumerate(zip(sa, sb)):
            for x, y in ((ma[cur], mb[cur]), (mma[cur], mmb[cur]), (vva[cur], vvb[cur])):
                assert torch.equal(x.view(torch.int32), y.view(torch.int32)), f"{case} shard {i} step {step}"
            assert torch.equal(pa.view(torch.int16), pb.view(torch.int16)), f"{case} shard {i} step {step}"
        for i in qwz:
            assert torch.equal(va[i].qcodes, vb[i].qcodes)
