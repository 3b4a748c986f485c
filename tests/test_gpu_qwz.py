"""qwZ: the int8 block-quantized copy of the fp16 shard for the parameter
all-gather ("ZeRO Optimization: Stages 1, 2, and 3 Explained", ZeRO++
quantized weights).  Codes and scales must equal the oracle's quantization of
the oracle's fp16 shard bit for bit after every step -- fused into the step
kernel for full blocks (narrow, wide and compile-time-N_d layouts), from the
commit for the partial tail block, rebuilt with the restore after an
overflow, on the synchronous, scalar, clipped and host-memory paths -- and the
standalone quantize / dequantize kernels equal the oracle's."""
import numpy as np
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner
from parity_util import OracleShard, f16_bits, oracle_group_step, to_np

pytestmark = pytest.mark.gpu


def _workload(n, n_d, **kw):
    base = dict(name="qwz", numels=(n * n_d,), n_d=n_d, rank=0, align=1, steps=3, lr=1e-3, beta1=0.9,
                beta2=0.999, eps=1e-8, weight_decay=0.0, loss_scale=1024.0, grad_dist="normal", grad_std=1e-2,
                grad_mult=1024.0, grads_fresh_per_step=True, master_dist="normal", master_param=0.02,
                seed=3 * n + n_d)
    base.update(kw)
    return synth.Workload(**base)


def _check_codes(oracle, run, r, ref_params_bits, what):
    n = run.n_valid[r]
    codes, scales = run.qwz[r]
    want_c, want_s = oracle.qwz_quantize(ref_params_bits)
    got_c = to_np(codes[:n])
    got_s = to_np(scales[: want_s.size])
    assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32)), f"{what}: scales"
    assert np.array_equal(got_c, want_c), f"{what}: codes ({int((got_c != want_c).sum())} differ)"


@pytest.mark.parametrize("n", [256 * 40, 256 * 40 + 77, 200, 4096 * 3 + 8])
@pytest.mark.parametrize("n_d", [4, 8, 64])
@pytest.mark.parametrize("math", ["ieee", "fast"])
def test_fused_qwz_matches_oracle(zs, oracle, cuda_device, n, n_d, math):
    """math = fast (ZS_MATH_FAST): params within the stated tolerance of the
    oracle's, and the codes equal to the oracle's quantization of the kernel's
    own fp16 shard (the same fp32 decision on the same inputs)."""
    w = _workload(n, n_d)
    run = WorkloadRunner(w, cuda_device, math=zs.ZS_MATH_FAST if math == "fast" else zs.ZS_MATH_IEEE)
    run.enable_qwz()
    r = run.shard_ids[0]
    ref = OracleShard(oracle, to_np(run.state[r][0][0]))
    _check_codes(oracle, run, r, ref.params, "initial")
    ls, applied = w.loss_scale, 0
    for step in range(1, 5):
        if step > 1:
            run.refresh_grads(step)
        if step == 3:
            run.grads[r][n_d - 1][n // 2] = float("nan")       # dropped step: restore + re-quantize
        host = [[synth.fp16_bits(g[:n]) for g in run.grads[r]]]
        run.step()
        torch.cuda.synchronize()
        ovf, ls, applied = oracle_group_step(oracle, [ref], host, w, ls, applied)
        assert ovf == int(step == 3) == run.ctrl_host()["last_overflow"]
        master, m, v, params = run.current(r)
        ref.compare(to_np(master), to_np(m), to_np(v), f16_bits(params), what=f"step {step}")
        own = f16_bits(params[:n])
        if math == "ieee":
            assert np.array_equal(own, ref.params[:n])
        _check_codes(oracle, run, r, own, f"{math} n={n} n_d={n_d} step {step}")


@pytest.mark.parametrize("offset", [0, 1])
def test_sync_and_scalar_paths_keep_qwz(zs, oracle, cuda_device, offset):
    """Synchronous entry point; offset 1 makes the buffers misaligned, so the
    scalar kernel steps and the qwZ copy comes from its own pass."""
    n, n_d = 256 * 9 + 31, 4
    w = _workload(n, n_d)
    dev = cuda_device
    pad = lambda dt: torch.zeros(n + 64, dtype=dt, device=dev)[offset:offset + n]
    grads = [pad(torch.float16) for _ in range(n_d)]
    master = (pad(torch.float32), pad(torch.float32))
    m = (pad(torch.float32), pad(torch.float32))
    v = (pad(torch.float32), pad(torch.float32))
    params = pad(torch.float16)
    master[0].copy_(synth.master_init(w, n).to(dev))
    zs.zero_params_from_master(master[0], params, n)
    codes = torch.zeros(n + 64, dtype=torch.int8, device=dev)[offset:offset + n]
    scales = torch.zeros((n + 255) // 256, dtype=torch.float32, device=dev)
    view = zs.ShardView(grads, master, m, v, params, n, qcodes=codes, qscales=scales)
    ref = OracleShard(oracle, to_np(master[0]))
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    cur, ls, applied = 0, w.loss_scale, 0
    for step in range(1, 4):
        contribs = [synth.grad_contribution(w, n, k, step) for k in range(n_d)]
        if step == 2:
            contribs[0][7] = float("inf")
        for g, c in zip(grads, contribs):
            g.copy_(c.to(dev))
        ovf = zs.zero_shard_step([view], n_d, zs.adam(w.lr), ls, applied + 1, cur, flag)
        rovf, ls, applied = oracle_group_step(oracle, [ref], [[synth.fp16_bits(c) for c in contribs]], w, ls,
                                              applied)
        assert ovf == rovf == int(step == 2)
        if not ovf:
            cur ^= 1
        ref.compare(to_np(master[cur]), to_np(m[cur]), to_np(v[cur]), f16_bits(params), what=f"step {step}")
        want_c, want_s = oracle.qwz_quantize(ref.params)
        assert np.array_equal(to_np(codes), want_c) and np.array_equal(to_np(scales), want_s)


@pytest.mark.parametrize("n", [1, 255, 256, 257, 256 * 1000 + 3])
@pytest.mark.parametrize("offset", [0, 1])
def test_quantize_dequantize_kernels(zs, oracle, cuda_device, n, offset):
    rng = np.random.Generator(np.random.PCG64(n + offset))
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-4, 3, n)).astype(np.float16)
    x[::97] = 0.0
    dev = cuda_device
    params = torch.zeros(n + 64, dtype=torch.float16, device=dev)[offset:offset + n]
    params.copy_(torch.from_numpy(x).to(dev))
    codes = torch.zeros(n + 64, dtype=torch.int8, device=dev)[offset:offset + n]
    scales = torch.zeros((n + 255) // 256, dtype=torch.float32, device=dev)
    zs.zero_qwz_quantize(params, n, codes, scales)
    want_c, want_s = oracle.qwz_quantize(x.view(np.uint16))
    assert np.array_equal(to_np(codes), want_c) and np.array_equal(to_np(scales), want_s)
    back = torch.zeros(n + 64, dtype=torch.float16, device=dev)[offset:offset + n]
    zs.zero_qwz_dequantize(codes, scales, n, back)
    assert np.array_equal(f16_bits(back), oracle.qwz_dequantize(want_c, want_s))


def test_clipped_step_keeps_qwz(zs, oracle, cuda_device):
    n, n_d = 256 * 30 + 5, 8
    w = _workload(n, n_d, grads_fresh_per_step=False)
    run = WorkloadRunner(w, cuda_device)
    run.enable_qwz()
    run.enable_clipping(True)
    r = run.shard_ids[0]
    ref = OracleShard(oracle, to_np(run.state[r][0][0]))
    host = [synth.fp16_bits(g[:n]) for g in run.grads[r]]
    for step in range(1, 3):
        g, _ = oracle.grad_reduce(host, w.loss_scale)
        c = oracle.clip_factor(oracle.grad_sqnorm(g), 0.01)
        oracle.scale(g, c)
        ref.apply(g, w, step)
        run.step_clipped(0.01)
        torch.cuda.synchronize()
        master, m, v, params = run.current(r)
        ref.compare(to_np(master), to_np(m), to_np(v), f16_bits(params), what=f"clipped step {step}")
        _check_codes(oracle, run, r, ref.params, f"clipped step {step}")


def test_host_path_keeps_qwz(zs, oracle, cuda_device):
    n, n_d = 256 * 12 + 100, 4
    w = _workload(n, n_d, grads_fresh_per_step=False)
    run = WorkloadRunner(w, cuda_device)
    r = run.shard_ids[0]
    master, m, v, _ = run.state[r]
    host_grads = [g[:n].cpu().pin_memory() for g in run.grads[r]]
    host_params = torch.zeros(n, dtype=torch.float16).pin_memory()
    codes = torch.zeros(n, dtype=torch.int8).pin_memory()
    scales = torch.zeros((n + 255) // 256, dtype=torch.float32).pin_memory()
    view = zs.HostShardView(host_grads, master, m, v, host_params, n, qcodes=codes, qscales=scales)
    ref = OracleShard(oracle, to_np(master[0]))
    for step in range(1, 3):
        assert zs.zero_shard_step_host(view, n_d, run.hp, run.ctrl) == 0
        oracle_group_step(oracle, [ref], [[synth.fp16_bits(g) for g in host_grads]], w, w.loss_scale, step - 1)
        assert np.array_equal(host_params.view(torch.int16).numpy().view(np.uint16), ref.params)
        want_c, want_s = oracle.qwz_quantize(ref.params)
        assert np.array_equal(codes.numpy(), want_c) and np.array_equal(scales.numpy(), want_s)


def test_full_size_qwz_sampled_blocks(zs, oracle, cuda_device):
    w = synth.WORKLOADS["xl"]
    run = WorkloadRunner(w, cuda_device)
    run.enable_qwz()
    r = run.shard_ids[0]
    n = run.n_valid[r]
    nblocks = (n + 255) // 256
    rng = np.random.Generator(np.random.PCG64(8))
    blocks = np.unique(np.concatenate([[0, 1, nblocks - 2, nblocks - 1], rng.integers(0, nblocks, 300)]))
    idx_np = np.concatenate([np.arange(256 * b, min(n, 256 * b + 256)) for b in blocks])
    idx = torch.tensor(idx_np, device=cuda_device)
    ref = OracleShard(oracle, to_np(run.state[r][0][0][idx]))
    for step in range(1, 3):
        host = [[synth.fp16_bits(g[idx]) for g in run.grads[r]]]
        run.step()
        torch.cuda.synchronize()
        oracle_group_step(oracle, [ref], host, w, w.loss_scale, step - 1)
        codes, scales = run.qwz[r]
        got_c = to_np(codes[idx])
        got_s = to_np(scales[torch.tensor(blocks, device=cuda_device)])
        off = 0
        for k, b in enumerate(blocks):
            ln = min(n, 256 * b + 256) - 256 * b
            wc, ws = oracle.qwz_quantize(ref.params[off:off + ln])
            assert got_s[k] == ws[0] and np.array_equal(got_c[off:off + ln], wc), (step, b)
            off += ln
