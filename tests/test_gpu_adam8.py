"""Parity of the 8-bit Adam shard step with the oracle.

Codes and block scales are integers and fp32 values decided by fp32
arithmetic on both sides: they must match bit for bit, in both arithmetic
modes (ZS_MATH_FAST changes only u, which m' and v' do not depend on).  Master
and params: bit-exact in the IEEE mode, within the stated tolerance in the
fast one.  Cases: the 8- and 16-element layouts and the element-wise one
(misaligned buffers), run-time and compile-time N_d, ragged blocks and
tails, an overflow step (everything unchanged, loss scale halved), several
shards in one call, grouped launches, subnormal block scales, and the
full-size 1.5B, 7.5B and ragged workloads on whole sampled blocks (blocks
are independent, so the oracle steps each sampled block on its own)."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner
from parity_util import assert_f16_close, assert_f32_close, f16_bits, to_np

pytestmark = pytest.mark.gpu

B = 2048


def _workload(n, n_d, **kw):
    base = dict(name="adam8", numels=(n * n_d,), n_d=n_d, rank=0, align=1, steps=4, lr=1e-3, beta1=0.9,
                beta2=0.999, eps=1e-8, weight_decay=0.01, loss_scale=1024.0, grad_dist="normal", grad_std=1e-2,
                grad_mult=1024.0, grads_fresh_per_step=True, master_dist="normal", master_param=0.02,
                seed=3 * n + n_d)
    base.update(kw)
    return synth.Workload(**base)


class OracleAdam8:
    def __init__(self, oracle, master0, w):
        self.o, self.w = oracle, w
        self.master = np.array(master0, np.float32)
        n = self.master.size
        self.mc = np.zeros(n, np.uint8)
        self.vc = np.zeros(n, np.uint8)
        self.ms = np.zeros((n + B - 1) // B, np.float32)
        self.vs = np.zeros((n + B - 1) // B, np.float32)
        self.params = oracle.f32_to_f16(self.master)

    def reduce(self, contribs, loss_scale):
        return self.o.grad_reduce(contribs, loss_scale, n=self.master.size)

    def apply(self, g, t):
        w = self.w
        self.o.adam8_apply(g, self.master, self.mc, self.vc, self.ms, self.vs, self.params, lr=w.lr,
                           beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, step=t)

    def compare(self, master, mc, vc, ms, vs, params_bits, exact, what):
        assert np.array_equal(mc, self.mc), f"{what}: m codes differ at {np.flatnonzero(mc != self.mc)[:5]}"
        assert np.array_equal(vc, self.vc), f"{what}: v codes differ at {np.flatnonzero(vc != self.vc)[:5]}"
        assert np.array_equal(ms.view(np.uint32), self.ms.view(np.uint32)), f"{what}: m scales"
        assert np.array_equal(vs.view(np.uint32), self.vs.view(np.uint32)), f"{what}: v scales"
        if exact:
            assert np.array_equal(master.view(np.uint32), self.master.view(np.uint32)), f"{what}: master"
            assert np.array_equal(params_bits, self.params), f"{what}: params"
        else:
            assert_f32_close(master, self.master, f"{what} master")
            assert_f16_close(params_bits, self.params, f"{what} params")


def _state(run, r, n):
    master, mc, vc, ms, vs, params = run.current_adam8(r)
    nb = (n + B - 1) // B
    return to_np(master[:n]), to_np(mc[:n]), to_np(vc[:n]), to_np(ms[:nb]), to_np(vs[:nb]), f16_bits(params[:n])


@pytest.mark.parametrize("math", ["ieee", "fast"])
@pytest.mark.parametrize("n", [1, 7, B, B + 1, 3 * B + 777, 65536 + 13])
@pytest.mark.parametrize("n_d", [1, 4, 5, 8, 16, 64])
def test_adam8_step_matches_oracle(zs, oracle, cuda_device, n, n_d, math):
    mode = zs.ZS_MATH_FAST if math == "fast" else zs.ZS_MATH_IEEE
    w = _workload(n, n_d)
    run = WorkloadRunner(w, cuda_device, math=mode)
    run.enable_adam8()
    r = run.shard_ids[0]
    ref = OracleAdam8(oracle, to_np(run.state[r][0][0][:n]), w)
    ls, applied = w.loss_scale, 0
    for step in range(1, 5):
        if step > 1:
            run.refresh_grads(step)
        inject = step == 3 and n > 1
        if inject:
            run.grads[r][n_d - 1][n - 1] = float("inf")
        host = [synth.fp16_bits(g[:n]) for g in run.grads[r]]
        before = [t.clone() for t in run.current_adam8(r)] if inject else None
        run.step_adam8()
        torch.cuda.synchronize()
        g, bad = ref.reduce(host, ls)
        if not bad:
            ref.apply(g, applied + 1)
        ls, applied = oracle.commit(bad, ls, applied)
        c = run.ctrl_host()
        assert c["last_overflow"] == bad == int(inject) and c["step"] == applied and c["loss_scale"] == ls
        if bad:
            for a, b in zip(before, run.current_adam8(r)):
                assert torch.equal(a, b)
        ref.compare(*_state(run, r, n), exact=math == "ieee", what=f"n={n} n_d={n_d} {math} step {step}")


@pytest.mark.parametrize("n_d", [4, 16])
def test_adam8_misaligned_elementwise(zs, oracle, cuda_device, n_d):
    """Buffers one element off their natural vector alignment: the element-wise
    kernel, same results."""
    n = 2 * B + 333
    w = _workload(n, n_d, grads_fresh_per_step=False)
    dev = cuda_device
    grads = []
    for k in range(n_d):
        t = torch.zeros(n + 16, dtype=torch.float16, device=dev)[1:1 + n]
        t.copy_(synth.grad_contribution(w, n, k, 1, shard=0, device=dev))
        grads.append(t)
    f32 = lambda: torch.zeros(n + 16, dtype=torch.float32, device=dev)[1:1 + n]
    u8 = lambda: torch.zeros(n + 16, dtype=torch.uint8, device=dev)[1:1 + n]
    sc = lambda: torch.zeros(8, dtype=torch.float32, device=dev)[1:]
    master = (f32(), f32())
    master[0].copy_(synth.master_init(w, n, shard=0, device=dev))
    params = torch.zeros(n + 16, dtype=torch.float16, device=dev)[1:1 + n]
    zs.zero_params_from_master(master[0], params, n)
    mc, vc, ms, vs = (u8(), u8()), (u8(), u8()), (sc(), sc()), (sc(), sc())
    view = zs.Adam8View(grads, master, mc, vc, ms, vs, params, n)
    ctrl = zs.new_ctrl(dev)
    zs.zero_ctrl_init(ctrl, w.loss_scale)
    hp = zs.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    ref = OracleAdam8(oracle, to_np(master[0]), w)
    host = [synth.fp16_bits(g) for g in grads]
    for step in range(1, 4):
        zs.zero_shard_step_adam8_async([view], n_d, hp, ctrl)
        torch.cuda.synchronize()
        g, bad = ref.reduce(host, w.loss_scale)
        assert not bad
        ref.apply(g, step)
        cur = zs.read_ctrl(ctrl)["cur"]
        ref.compare(to_np(master[cur]), to_np(mc[cur]), to_np(vc[cur]), to_np(ms[cur][:3]), to_np(vs[cur][:3]),
                    f16_bits(params), exact=True, what=f"misaligned n_d={n_d} step {step}")


def test_adam8_multi_shard(zs, oracle, cuda_device):
    """Every shard of a ragged tensor list in one call: one kernel per shard,
    one commit; an overflow in one shard skips all of them."""
    numels = tuple(synth.ragged_numels(80, seed=6, max_exp=13))
    w = _workload(0, 8, numels=numels, rank=None, align=128, grads_fresh_per_step=False, seed=12)
    run = WorkloadRunner(w, cuda_device)
    run.enable_adam8()
    refs = {r: OracleAdam8(oracle, to_np(run.state[r][0][0][: run.n_valid[r]]), w) for r in run.shard_ids}
    ls, applied = w.loss_scale, 0
    victim = run.shard_ids[3]
    for step in range(1, 5):
        inject = step == 2
        if inject:
            run.grads[victim][2][5] = float("nan")
        run.step_adam8()
        torch.cuda.synchronize()
        reduced, ovf = {}, 0
        for r in run.shard_ids:
            n = run.n_valid[r]
            reduced[r], bad = refs[r].reduce([synth.fp16_bits(g[:n]) for g in run.grads[r]], ls)
            ovf |= bad
        if not ovf:
            for r in run.shard_ids:
                refs[r].apply(reduced[r], applied + 1)
        ls, applied = oracle.commit(ovf, ls, applied)
        assert ovf == int(inject) and run.ctrl_host()["step"] == applied
        if inject:
            run.grads[victim][2][5] = 0.0
        for r in run.shard_ids:
            refs[r].compare(*_state(run, r, run.n_valid[r]), exact=True, what=f"shard {r} step {step}")


@pytest.mark.parametrize("name", ["xl", "7b5", "ragged"])
def test_adam8_full_size_sampled_blocks(zs, oracle, cuda_device, name):
    """The full-size workloads in the benchmark's launch configuration and
    arithmetic mode, two steps, checked on whole blocks: the first, the last
    (partial) and 30 random ones of each checked shard (xl: 375,000,064
    elements, N_d = 4, one-slot staged kernel; 7b5: 117,187,584, N_d = 64,
    16-element kernel; ragged: all 16 shards in one grouped launch, shards 0,
    7 and 15 checked).  Each block's step depends only on its own elements,
    so the oracle steps them one by one."""
    w = synth.WORKLOADS[name]
    run = WorkloadRunner(w, cuda_device, with_full_params=False, math=zs.ZS_MATH_FAST)
    run.enable_adam8()
    ids = run.shard_ids if len(run.shard_ids) == 1 else [run.shard_ids[i] for i in (0, 7, 15)]
    rng = np.random.Generator(np.random.PCG64(77))
    checks = []
    for r in ids:
        n = run.n_valid[r]
        nb = (n + B - 1) // B
        blocks = sorted(set([0, nb - 1] + [int(b) for b in rng.integers(1, nb - 1, 30)]))
        for b in blocks:
            lo, hi = b * B, min(n, (b + 1) * B)
            ref = OracleAdam8(oracle, to_np(run.state[r][0][0][lo:hi]), w)
            host = [synth.fp16_bits(g[lo:hi]) for g in run.grads[r]]
            checks.append((r, b, lo, hi, ref, host))
    for step in (1, 2):
        run.step_adam8()
        torch.cuda.synchronize()
        state = {r: run.current_adam8(r) for r in ids}
        for r, b, lo, hi, ref, host in checks:
            master, mc, vc, ms, vs, params = state[r]
            g, bad = ref.reduce(host, w.loss_scale)
            assert not bad
            ref.apply(g, step)
            ref.compare(to_np(master[lo:hi]), to_np(mc[lo:hi]), to_np(vc[lo:hi]), to_np(ms[b:b + 1]),
                        to_np(vs[b:b + 1]), f16_bits(params[lo:hi]), exact=False,
                        what=f"{name} shard {r} block {b} step {step}")


@pytest.mark.parametrize("n_d", [4, 16])
def test_adam8_tiny_scales(zs, oracle, cuda_device, n_d):
    """Blocks whose moments decayed below 2^-126 (zero gradients, subnormal
    scales): the new scale has no finite reciprocal, x is clamped, the codes
    and scales still equal the oracle's, and every table index stays inside."""
    n = 3 * B + 100
    w = _workload(n, n_d, grads_fresh_per_step=False)
    run = WorkloadRunner(w, cuda_device)
    run.enable_adam8()
    r = run.shard_ids[0]
    for g in run.grads[r]:
        g[: 2 * B].zero_()                                   # blocks 0-1: no gradient; 2-3: ordinary
    rng = np.random.Generator(np.random.PCG64(13))
    mc, vc, ms, vs = run.adam8[r]
    codes_m = rng.integers(0, 256, n).astype(np.uint8)
    codes_v = rng.integers(0, 256, n).astype(np.uint8)
    sc_m = np.array([1e-39, 2e-45, 1e-3, 5e-4], np.float32)
    sc_v = np.array([1e-39, 1e-40, 1e-6, 2e-6], np.float32)
    mc[0][:n].copy_(torch.from_numpy(codes_m))
    vc[0][:n].copy_(torch.from_numpy(codes_v))
    ms[0][:4].copy_(torch.from_numpy(sc_m))
    vs[0][:4].copy_(torch.from_numpy(sc_v))
    ref = OracleAdam8(oracle, to_np(run.state[r][0][0][:n]), w)
    ref.mc[:], ref.vc[:], ref.ms[:], ref.vs[:] = codes_m, codes_v, sc_m, sc_v
    host = [synth.fp16_bits(g[:n]) for g in run.grads[r]]
    for step in (1, 2, 3):
        run.step_adam8()
        torch.cuda.synchronize()
        g, bad = ref.reduce(host, w.loss_scale)
        assert not bad
        ref.apply(g, step)
        ref.compare(*_state(run, r, n), exact=True, what=f"tiny scales n_d={n_d} step {step}")
    assert ref.ms[0] < 2.0 ** -126 and ref.ms[1] == 0.0 or ref.ms[1] < 2.0 ** -126


def _adam8_views(zs, dev, w, sizes, misaligned):
    """Fresh buffers per shard; shard i one element off its alignment (the
    element-wise kernel) when listed.  Returns the views and host contribs."""
    views, host = [], []
    for i, n in enumerate(sizes):
        off = 1 if i in misaligned else 0
        nb = (n + B - 1) // B
        grads = []
        for k in range(w.n_d):
            t = torch.zeros(n + 16, dtype=torch.float16, device=dev)[off:off + n]
            t.copy_(synth.grad_contribution(w, n, k, 1, shard=i, device=dev))
            grads.append(t)
        f32 = lambda: torch.zeros(n + 16, dtype=torch.float32, device=dev)[off:off + n]
        u8 = lambda: torch.zeros(n + 32, dtype=torch.uint8, device=dev)[off:off + n]
        sc = lambda: torch.zeros(nb + 4, dtype=torch.float32, device=dev)[off:off + nb]
        master = (f32(), f32())
        master[0].copy_(synth.master_init(w, n, shard=i, device=dev))
        params = torch.zeros(n + 16, dtype=torch.float16, device=dev)[off:off + n]
        if n:
            zs.zero_params_from_master(master[0], params, n)
        views.append(zs.Adam8View(grads, master, (u8(), u8()), (u8(), u8()), (sc(), sc()), (sc(), sc()), params, n))
        host.append([synth.fp16_bits(g) for g in grads])
    return views, host


@pytest.mark.parametrize("n_d,sizes,misaligned", [
    (4, [int(x) for x in np.random.Generator(np.random.PCG64(21)).integers(0, 9000, 37)], ()),   # groups of 16
    (8, [3 * B + 5, 0, B, 2 * B + 1, 777, 5000, 6, 3000, 4 * B], (3,)),                          # cut by a misaligned shard
    (16, [B + 3, 17, 0, 250, 4099, 2 * B], ()),
    (64, [B - 1, 300, 2 * B + 9], (1,)),
])
def test_adam8_grouped_launches(zs, oracle, cuda_device, n_d, sizes, misaligned):
    """Consecutive shards of one access width share a launch (up to 16) that
    walks their blocks back to back; empty shards join any group; the result
    equals the oracle bit for bit, with an overflow in one shard on step 2."""
    w = _workload(1, n_d, grads_fresh_per_step=False, seed=len(sizes) + n_d)
    views, host = _adam8_views(zs, cuda_device, w, sizes, misaligned)
    refs = [OracleAdam8(oracle, to_np(v.master[0]), w) for v in views]
    ctrl = zs.new_ctrl(cuda_device)
    zs.zero_ctrl_init(ctrl, w.loss_scale)
    hp = zs.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    victim = max(range(len(sizes)), key=lambda i: sizes[i])
    ls, applied = w.loss_scale, 0
    for step in range(1, 4):
        inject = step == 2
        j = sizes[victim] // 2
        if inject:
            keep = views[victim].grads[0][j].clone()
            views[victim].grads[0][j] = float("inf")
        launches = zs.zero_kernel_launches()
        zs.zero_shard_step_adam8_async(views, n_d, hp, ctrl)
        torch.cuda.synchronize()
        reduced, ovf = [], 0
        for ref, v in zip(refs, views):
            g, bad = ref.reduce([synth.fp16_bits(t) for t in v.grads], ls)
            reduced.append(g)
            ovf |= bad
        if not ovf:
            for ref, g in zip(refs, reduced):
                ref.apply(g, applied + 1)
        ls, applied = oracle.commit(ovf, ls, applied)
        c = zs.read_ctrl(ctrl)
        assert ovf == int(inject) and c["last_overflow"] == ovf and c["step"] == applied
        if inject:
            views[victim].grads[0][j] = keep
        cur = c["cur"]
        for i, (ref, v) in enumerate(zip(refs, views)):
            if not sizes[i]:
                continue
            nb = (sizes[i] + B - 1) // B
            ref.compare(to_np(v.master[cur]), to_np(v.m_codes[cur]), to_np(v.v_codes[cur]), to_np(v.m_scale[cur][:nb]),
                        to_np(v.v_scale[cur][:nb]), f16_bits(v.params), exact=True,
                        what=f"n_d={n_d} shard {i} step {step}")
    # one launch per group: runs of one width, at most 16 shards each, plus the restore pass
    live = [i for i, n in enumerate(sizes) if n]
    groups, i = 0, 0
    widths = [0 if k in misaligned else 1 for k in range(len(sizes))]
    while i < len(sizes):
        if not sizes[i]:
            i += 1
            continue
        k = i + 1
        while k < len(sizes) and k - i < 16 and (not sizes[k] or widths[k] == widths[i]):
            k += 1
        groups += 1
        i = k
    assert live and zs.zero_kernel_launches() - launches == groups + 1
