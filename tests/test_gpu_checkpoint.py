"""Checkpoint / resume of a shard step: 3 steps, save (control block bytes
and the committed state), load into a fresh runner, 2 more steps must equal 5
straight steps bit for bit -- including a skipped overflow step before the
save, so the loss scale, t and beta^t carried in the control block matter."""
import pytest
import torch

from zero_partitioned_mixed_partition_gb300 import synth
from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("qwz", [False, True])
@pytest.mark.parametrize("n_d", [4, 16])
def test_save_load_resume_is_exact(zs, cuda_device, n_d, qwz):
    """qwz: every runner keeps the int8 qwZ copy of its fp16 slice; after
    load() the copy must describe the loaded slice (the resumed runner's copy
    was made from other weights), and after 2 more steps it must equal the
    straight run's bit for bit."""
    n = 2048 * 9 + 5
    w = synth.Workload(name="ckpt", numels=(n * n_d,), n_d=n_d, rank=0, align=1, steps=5, lr=1e-3, beta1=0.9,
                       beta2=0.999, eps=1e-8, weight_decay=0.01, loss_scale=1024.0, grad_dist="normal",
                       grad_std=1e-2, grad_mult=1024.0, grads_fresh_per_step=True, master_dist="normal",
                       master_param=0.02, seed=31 + n_d)

    def run_steps(run, steps):
        for s in steps:
            run.refresh_grads(s)
            if s == 2:
                run.grads[0][1][5] = float("inf")       # step 2 overflows and is skipped
            run.step()
        torch.cuda.synchronize()

    def runner():
        run = WorkloadRunner(w, cuda_device)
        if qwz:
            run.enable_qwz()
        return run

    straight = runner()
    run_steps(straight, [1, 2, 3, 4, 5])
    first = runner()
    run_steps(first, [1, 2, 3])
    ckpt = first.save()
    del first
    resumed = runner()
    for pair in resumed.state[0][:3]:           # scribble over the fresh state: load must replace it
        for t in pair:
            t.fill_(7.0)
    resumed.state[0][3].fill_(-1.0)
    resumed.step()                              # and advance its control block
    torch.cuda.synchronize()
    resumed.load(ckpt)
    if qwz:                                     # the copy now describes the loaded slice
        codes, scales = resumed.qwz[0]
        ref_codes = torch.zeros_like(codes)
        ref_scales = torch.zeros_like(scales)
        zs.zero_qwz_quantize(resumed.state[0][3], resumed.n_valid[0], ref_codes, ref_scales)
        torch.cuda.synchronize()
        assert torch.equal(codes, ref_codes) and torch.equal(scales, ref_scales)
    run_steps(resumed, [4, 5])
    a, b = straight.ctrl_host(), resumed.ctrl_host()
    assert a == b and a["step"] == 4 and a["skipped"] == 1 and a["loss_scale"] == 512.0
    for x, y in zip(straight.current(0), resumed.current(0)):
        assert torch.equal(x, y)
    if qwz:
        for x, y in zip(straight.qwz[0], resumed.qwz[0]):
            assert torch.equal(x, y)


@pytest.mark.parametrize("n_d", [4, 16, 32])
def test_adam8_save_load_resume_is_exact(zs, cuda_device, n_d):
    """The same with 8-bit Adam state: the committed codes and block scales
    travel with the checkpoint, and 3 + 2 steps equal 5 straight steps bit for
    bit (codes, scales, master, params, control block).  n_d = 4 runs the
    staged 8-element kernel, 16 the direct one, 32 the 16-element one."""
    n = 2048 * 9 + 5
    w = synth.Workload(name="ckpt8", numels=(n * n_d,), n_d=n_d, rank=0, align=1, steps=5, lr=1e-3, beta1=0.9,
                       beta2=0.999, eps=1e-8, weight_decay=0.01, loss_scale=1024.0, grad_dist="normal",
                       grad_std=1e-2, grad_mult=1024.0, grads_fresh_per_step=True, master_dist="normal",
                       master_param=0.02, seed=41 + n_d)

    def runner():
        run = WorkloadRunner(w, cuda_device)
        run.enable_adam8()
        return run

    def run_steps(run, steps):
        for s in steps:
            run.refresh_grads(s)
            if s == 2:
                run.grads[0][0][7] = float("nan")        # step 2 overflows and is skipped
            run.step_adam8()
        torch.cuda.synchronize()

    straight = runner()
    run_steps(straight, [1, 2, 3, 4, 5])
    first = runner()
    run_steps(first, [1, 2, 3])
    ckpt = first.save()
    del first
    resumed = runner()
    for pair in resumed.adam8[0]:                # scribble over the fresh 8-bit state: load must replace it
        for t in pair:
            t.fill_(3)
    resumed.step_adam8()
    torch.cuda.synchronize()
    resumed.load(ckpt)
    run_steps(resumed, [4, 5])
    a, b = straight.ctrl_host(), resumed.ctrl_host()
    assert a == b and a["step"] == 4 and a["skipped"] == 1
    for x, y in zip(straight.current_adam8(0), resumed.current_adam8(0)):
        assert torch.equal(x, y)
