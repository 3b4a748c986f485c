"""How the SGD and 8-bit Adam steps end ("ZeRO Stage 1 Math", "The per-step
mechanics": a step that overflowed is dropped, one that did not is
committed), now that their last fused launch finishes the step in the
control block and a restore pass follows, every launch with programmatic
serialization:

  - five steps enqueued back to back with no host synchronisation in
    between, over 20 shards (two grouped launches, 16 + 4), with an overflow
    in a shard of the FIRST launch on step 3 (the whole step is dropped: the
    state of every shard unchanged, each fp16 slice re-cast, the loss scale
    halved, t not advanced), compared with the oracle bit for bit at the end;
  - a call whose shards are all empty: nothing to launch, so the commit
    kernel ends the step (t advances), and the next call steps normally.
"""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from parity_util import f16_bits, to_np

pytestmark = pytest.mark.gpu

B = 2048
MU, LR, WD = 0.9, 0.01, 1e-3


def _workload(n_d, seed):
    return synth.Workload(name="step-end", numels=(n_d,), n_d=n_d, rank=0, align=1, steps=5, lr=1e-3, beta1=0.9,
                          beta2=0.999, eps=1e-8, weight_decay=0.01, loss_scale=1024.0, grad_dist="normal",
                          grad_std=1e-2, grad_mult=1024.0, grads_fresh_per_step=False, master_dist="normal",
                          master_param=0.02, seed=seed)


def _sizes(count, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return [int(x) for x in g.integers(1, 3 * B + 700, count)]


def _buffers(dev, w, sizes, i, n):
    grads = []
    for k in range(w.n_d):
        t = torch.zeros(n + 16, dtype=torch.float16, device=dev)[:n]
        t.copy_(synth.grad_contribution(w, n, k, 1, shard=i, device=dev))
        grads.append(t)
    master = (torch.zeros(n + 16, dtype=torch.float32, device=dev)[:n],
              torch.zeros(n + 16, dtype=torch.float32, device=dev)[:n])
    master[0].copy_(synth.master_init(w, n, shard=i, device=dev))
    params = torch.zeros(n + 16, dtype=torch.float16, device=dev)[:n]
    return grads, master, params


def _sgd_views(zs, dev, w, sizes):
    views = []
    for i, n in enumerate(sizes):
        grads, master, params = _buffers(dev, w, sizes, i, n)
        mom = (torch.zeros(n + 16, dtype=torch.float32, device=dev)[:n],
               torch.zeros(n + 16, dtype=torch.float32, device=dev)[:n])
        if n:
            zs.zero_params_from_master(master[0], params, n)
        views.append(zs.ShardView(grads, master, mom, mom, params, n))
    return views


def _adam8_views(zs, dev, w, sizes):
    views = []
    for i, n in enumerate(sizes):
        grads, master, params = _buffers(dev, w, sizes, i, n)
        nb = (n + B - 1) // B
        u8 = lambda: torch.zeros(n + 32, dtype=torch.uint8, device=dev)[:n]
        sc = lambda: torch.zeros(nb + 4, dtype=torch.float32, device=dev)[:nb]
        if n:
            zs.zero_params_from_master(master[0], params, n)
        views.append(zs.Adam8View(grads, master, (u8(), u8()), (u8(), u8()), (sc(), sc()), (sc(), sc()), params, n))
    return views


def _run_back_to_back(zs, oracle, dev, kind):
    """Five steps with no host synchronisation between them; an overflow in
    shard 0 (the first grouped launch) on step 3."""
    n_d = 20   # 20 shards of one access width: launches of 16 and 4 shards
    w = _workload(n_d, seed=41 if kind == "sgd" else 43)
    sizes = _sizes(n_d, seed=5)
    views = _sgd_views(zs, dev, w, sizes) if kind == "sgd" else _adam8_views(zs, dev, w, sizes)
    host = [[synth.fp16_bits(g) for g in v.grads] for v in views]
    masters = [np.array(to_np(v.master[0]), np.float32) for v in views]   # before any step writes a set
    ctrl = zs.new_ctrl(dev)
    zs.zero_ctrl_init(ctrl, w.loss_scale)
    adam_hp = zs.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    sgd_hp = zs.sgd(LR, MU, WD)
    victim, j = 0, sizes[0] // 2
    keep = views[victim].grads[1][j].clone()
    stream = torch.cuda.current_stream()
    for step in range(1, 6):
        # the injection and its undoing are stream-ordered with the steps
        if step == 3:
            views[victim].grads[1][j] = float("inf")
        if kind == "sgd":
            zs.zero_shard_step_sgd_async(views, n_d, sgd_hp, ctrl, stream=stream)
        else:
            zs.zero_shard_step_adam8_async(views, n_d, adam_hp, ctrl, stream=stream)
        if step == 3:
            views[victim].grads[1][j] = keep
    torch.cuda.synchronize()

    # the oracle: the same five steps, step 3 dropped
    ls, applied = w.loss_scale, 0
    state = []
    for i, n in enumerate(sizes):
        m0 = masters[i]
        if kind == "sgd":
            state.append({"master": m0.copy(), "mom": np.zeros_like(m0), "params": oracle.f32_to_f16(m0)})
        else:
            nb = (n + B - 1) // B
            state.append({"master": m0.copy(), "mc": np.zeros(n, np.uint8), "vc": np.zeros(n, np.uint8),
                          "ms": np.zeros(nb, np.float32), "vs": np.zeros(nb, np.float32),
                          "params": oracle.f32_to_f16(m0)})
    for step in range(1, 6):
        reduced, ovf = [], 0
        for i, n in enumerate(sizes):
            contribs = [h.copy() for h in host[i]]
            if step == 3 and i == victim:
                contribs[1][j] = 0x7c00   # +inf in fp16
            g, bad = oracle.grad_reduce(contribs, ls, n=n)
            reduced.append(g)
            ovf |= bad
        assert ovf == int(step == 3)
        if not ovf:
            for i, g in enumerate(reduced):
                s = state[i]
                if kind == "sgd":
                    oracle.sgd_apply(g, s["master"], s["mom"], s["params"], lr=LR, momentum=MU, weight_decay=WD)
                else:
                    oracle.adam8_apply(g, s["master"], s["mc"], s["vc"], s["ms"], s["vs"], s["params"], lr=w.lr,
                                       beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                                       step=applied + 1)
        ls, applied = oracle.commit(ovf, ls, applied)

    c = zs.read_ctrl(ctrl)
    assert c["step"] == applied == 4 and c["skipped"] == 1 and c["loss_scale"] == ls
    assert c["last_overflow"] == 0 and c["overflow"] == 0 and c["arrivals"] == 0
    cur = c["cur"]
    for i, (v, s) in enumerate(zip(views, state)):
        what = f"{kind} shard {i}"
        assert np.array_equal(to_np(v.master[cur]).view(np.uint32), s["master"].view(np.uint32)), what + " master"
        assert np.array_equal(f16_bits(v.params), s["params"]), what + " params"
        if kind == "sgd":
            assert np.array_equal(to_np(v.m[cur]).view(np.uint32), s["mom"].view(np.uint32)), what + " momentum"
        else:
            nb = (sizes[i] + B - 1) // B
            assert np.array_equal(to_np(v.m_codes[cur]), s["mc"]), what + " m codes"
            assert np.array_equal(to_np(v.v_codes[cur]), s["vc"]), what + " v codes"
            assert np.array_equal(to_np(v.m_scale[cur][:nb]).view(np.uint32), s["ms"].view(np.uint32)), what
            assert np.array_equal(to_np(v.v_scale[cur][:nb]).view(np.uint32), s["vs"].view(np.uint32)), what


@pytest.mark.parametrize("kind", ["sgd", "adam8"])
def test_back_to_back_steps_with_a_dropped_one(zs, oracle, cuda_device, kind):
    _run_back_to_back(zs, oracle, cuda_device, kind)


@pytest.mark.parametrize("kind", ["sgd", "adam8"])
def test_all_empty_shards_end_in_the_commit_kernel(zs, oracle, cuda_device, kind):
    n_d = 4
    w = _workload(n_d, seed=47)
    sizes = [0, 0, 0]
    make = _sgd_views if kind == "sgd" else _adam8_views
    empty = make(zs, cuda_device, w, sizes)
    live = make(zs, cuda_device, w, [3 * B + 5])
    ctrl = zs.new_ctrl(cuda_device)
    zs.zero_ctrl_init(ctrl, w.loss_scale)

    def step(views):
        launches = zs.zero_kernel_launches()
        if kind == "sgd":
            zs.zero_shard_step_sgd_async(views, n_d, zs.sgd(LR, MU, WD), ctrl)
        else:
            zs.zero_shard_step_adam8_async(views, n_d, zs.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay), ctrl)
        torch.cuda.synchronize()
        return zs.zero_kernel_launches() - launches

    assert step(empty) == 1   # the commit kernel alone
    c = zs.read_ctrl(ctrl)
    assert c["step"] == 1 and c["cur"] == 1 and c["skipped"] == 0 and c["arrivals"] == 0
    assert step(live) == 2    # the fused launch, then the restore pass
    c = zs.read_ctrl(ctrl)
    assert c["step"] == 2 and c["cur"] == 0 and c["arrivals"] == 0 and c["last_overflow"] == 0


@pytest.mark.parametrize("keep_g", [False, True])
def test_clipped_back_to_back_equals_the_split_calls(zs, oracle, cuda_device, keep_g):
    """The clipped step's one call (pass 2's last launch ends the step, then
    the restore pass; every launch with programmatic serialization), five
    steps enqueued without host synchronisation over 20 shards (two launches
    per pass) with an overflow on step 3, against the same steps through the
    separate pass calls and the commit kernel, synchronised after each step:
    equal bit for bit, control block included; and the oracle agrees within
    the stated tolerance."""
    from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner
    from parity_util import OracleShard

    n_d = 20
    numels = tuple(synth.ragged_numels(70, seed=13, max_exp=12))
    w = synth.Workload(name="clip-b2b", numels=numels, n_d=n_d, rank=None, align=128, steps=5, lr=1e-3, beta1=0.9,
                       beta2=0.999, eps=1e-8, weight_decay=0.05, loss_scale=1024.0, grad_dist="normal",
                       grad_std=1e-2, grad_mult=1024.0, grads_fresh_per_step=False, master_dist="normal",
                       master_param=0.02, seed=17)
    a, b = WorkloadRunner(w, cuda_device), WorkloadRunner(w, cuda_device)
    a.enable_clipping(keep_g)
    b.enable_clipping(keep_g)
    victim = a.shard_ids[0]
    host0 = {r: [synth.fp16_bits(g[: a.n_valid[r]]) for g in a.grads[r]] for r in a.shard_ids}
    refs = {r: OracleShard(oracle, to_np(a.state[r][0][0][: a.n_valid[r]])) for r in a.shard_ids}
    sq0 = 0.0
    for r in a.shard_ids:
        g, _ = refs[r].reduce(host0[r], w.loss_scale)
        sq0 = oracle.grad_sqnorm(g, sq0)
    max_norm = 0.5 * float(np.sqrt(sq0))

    keep = a.grads[victim][2][3].clone()
    for step in range(1, 6):          # a: no host synchronisation
        if step == 3:
            a.grads[victim][2][3] = float("inf")
        a.step_clipped(max_norm)
        if step == 3:
            a.grads[victim][2][3] = keep
    for step in range(1, 6):          # b: pass by pass, synchronised
        if step == 3:
            b.grads[victim][2][3] = float("inf")
        b.sqnorm.zero_()
        zs.zero_shard_grad_sqnorm_all_async(b.views, n_d, b.sqnorm, b.ctrl, g_dev=b.gbuf if b.gbuf else None)
        zs.zero_shard_clipped_adam_all_async(b.views, n_d, b.hp, max_norm, b.sqnorm, b.ctrl,
                                             g_dev=b.gbuf if b.gbuf else None)
        zs.zero_step_commit_async(b.views, b.hp, b.ctrl)
        torch.cuda.synchronize()
        if step == 3:
            b.grads[victim][2][3] = keep
    torch.cuda.synchronize()
    ca, cb = a.ctrl_host(), b.ctrl_host()
    assert ca == cb and ca["step"] == 4 and ca["skipped"] == 1 and ca["arrivals"] == 0
    for r in a.shard_ids:
        for x, y in zip(a.current(r), b.current(r)):
            assert torch.equal(x, y), f"shard {r}"

    # the oracle, within the stated tolerance (its norm sums in another order)
    ls, applied = w.loss_scale, 0
    for step in range(1, 6):
        reduced, ovf, sq = [], 0, 0.0
        for r in a.shard_ids:
            contribs = [h.copy() for h in host0[r]]
            if step == 3 and r == victim:
                contribs[2][3] = 0x7c00
            g, bad = refs[r].reduce(contribs, ls)
            reduced.append(g)
            ovf |= bad
            sq = oracle.grad_sqnorm(g, sq)
        c = oracle.clip_factor(sq, max_norm)
        if not ovf:
            for r, g in zip(a.shard_ids, reduced):
                oracle.scale(g, c)
                refs[r].apply(g, w, applied + 1)
        ls, applied = oracle.commit(ovf, ls, applied)
    assert applied == 4 and ca["loss_scale"] == ls
    for r in a.shard_ids:
        n = a.n_valid[r]
        master, m, v, params = a.current(r)
        refs[r].compare(to_np(master[:n]), to_np(m[:n]), to_np(v[:n]), f16_bits(params[:n]), what=f"shard {r}")


@pytest.mark.parametrize("kind", ["sgd", "adam8", "clip"])
def test_graph_captured_steps_of_each_kind(zs, cuda_device, kind):
    """Two steps of each kind captured in one CUDA graph (their launches carry
    programmatic serialization, so the graph holds programmatic edges) and
    replayed three times equal six steps run eagerly on a twin, bit for bit,
    control block included; 20 shards, so each step is two grouped launches
    and the restore pass."""
    from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner

    numels = tuple(synth.ragged_numels(70, seed=19, max_exp=12))
    w = synth.Workload(name="graph", numels=numels, n_d=20, rank=None, align=128, steps=6, lr=1e-3, beta1=0.9,
                       beta2=0.999, eps=1e-8, weight_decay=0.05, loss_scale=1024.0, grad_dist="normal",
                       grad_std=1e-2, grad_mult=1024.0, grads_fresh_per_step=False, master_dist="normal",
                       master_param=0.02, seed=23)
    a, b = WorkloadRunner(w, cuda_device), WorkloadRunner(w, cuda_device)
    hp = zs.sgd(LR, MU, WD)
    for run in (a, b):
        if kind == "adam8":
            run.enable_adam8()
        if kind == "clip":
            run.enable_clipping(True)
    max_norm = 0.05

    def step(run):
        if kind == "sgd":
            run.step_sgd(hp)
        elif kind == "adam8":
            run.step_adam8()
        else:
            run.step_clipped(max_norm)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(a)                                    # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(a)
        step(a)
    for _ in range(3):
        g.replay()
    for _ in range(7):
        step(b)
    torch.cuda.synchronize()
    ca, cb = a.ctrl_host(), b.ctrl_host()
    assert ca == cb and ca["step"] == 7 and ca["skipped"] == 0 and ca["arrivals"] == 0
    for r in a.shard_ids:
        sa = a.current_adam8(r) if kind == "adam8" else a.current(r)
        sb = b.current_adam8(r) if kind == "adam8" else b.current(r)
        for x, y in zip(sa, sb):
            assert torch.equal(x, y), f"{kind} shard {r}"
