"""Pins of the oracle's global gradient-norm clipping ("DeepSpeed ZeRO
Stages", sec. 2.1, Fact 1: clipping couples the coordinates through ||g||_2
over all of P).  The pages name the operation without a formula; the reading
is the common c = min(1, max_norm / (||g|| + 1e-6)), and it is pinned to
torch.nn.utils.clip_grad_norm_ (float64) followed by textbook Adam, to closed
forms and to the sharded == unsharded invariant.  CPU only."""
import numpy as np
import pytest
import torch


def _clipped_oracle_step(oracle, contribs, loss_scale, master, m, v, params, max_norm, step, **hp):
    g, bad = oracle.grad_reduce(contribs, loss_scale, n=master.size)
    assert bad == 0
    sq = oracle.grad_sqnorm(g)
    c = oracle.clip_factor(sq, max_norm)
    oracle.scale(g, c)
    oracle.adam_apply(g, master, m, v, params, step=step, **hp)
    return sq, c


@pytest.mark.parametrize("max_norm", [0.5, 5.0, 1e4])
@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_clip_matches_torch(oracle, max_norm, wd):
    n, steps = 3000, 3
    rng = np.random.Generator(np.random.PCG64(17))
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    grads = [(sign * rng.uniform(0.02, 0.2, n)).astype(np.float16) for _ in range(steps)]
    theta0 = rng.uniform(-1, 1, n).astype(np.float32)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=wd)
    p = torch.nn.Parameter(torch.tensor(theta0.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=hp["lr"], betas=(0.9, 0.999), eps=1e-8, weight_decay=wd, foreach=False)
    master, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    params = np.zeros(n, np.uint16)
    for t in range(1, steps + 1):
        p.grad = torch.tensor(grads[t - 1].astype(np.float64))
        tn = float(torch.nn.utils.clip_grad_norm_([p], max_norm))
        opt.step()
        sq, c = _clipped_oracle_step(oracle, [grads[t - 1].view(np.uint16)], 1.0, master, m, v, params,
                                     max_norm, t, **hp)
        assert abs(np.sqrt(sq) - tn) <= 1e-12 * tn
        st = opt.state[p]
        for got, ref in ((master, p.detach().numpy()), (m, st["exp_avg"].numpy()), (v, st["exp_avg_sq"].numpy())):
            np.testing.assert_allclose(got.astype(np.float64), ref, rtol=2e-6, atol=1e-9)


def test_clip_inactive_is_identity(oracle):
    """||g|| below max_norm: factor exactly 1 and the step is the unclipped one."""
    n = 777
    rng = np.random.Generator(np.random.PCG64(3))
    h = (rng.standard_normal(n) * 0.01).astype(np.float16)
    g, _ = oracle.grad_reduce([h.view(np.uint16)], 1.0)
    sq = oracle.grad_sqnorm(g)
    assert oracle.clip_factor(sq, 10.0 * np.sqrt(sq)) == 1.0
    assert oracle.clip_factor(sq, 0.0) == 1.0            # disabled
    assert oracle.clip_factor(sq, -1.0) == 1.0


def test_clip_closed_form_norm(oracle):
    """After clipping, ||c g|| = max_norm ||g|| / (||g|| + 1e-6)."""
    rng = np.random.Generator(np.random.PCG64(4))
    g = (rng.standard_normal(4096) * 3.0).astype(np.float32)
    sq = oracle.grad_sqnorm(g)
    norm = np.sqrt(np.sum(g.astype(np.float64) ** 2))
    assert abs(np.sqrt(sq) - norm) <= 1e-12 * norm
    c = oracle.clip_factor(sq, 1.0)
    gc = g.copy()
    oracle.scale(gc, c)
    assert np.array_equal(gc, g * np.float32(c))
    want = 1.0 * norm / (norm + 1e-6)
    got = np.sqrt(np.sum(gc.astype(np.float64) ** 2))
    assert abs(got - want) <= 2e-7 * want
    # a one-hot gradient: ||g|| is its magnitude
    e = np.zeros(10, np.float32)
    e[3] = -8.0
    assert oracle.grad_sqnorm(e) == 64.0
    assert oracle.clip_factor(64.0, 2.0) == np.float32(2.0 / (8.0 + 1e-6))


def test_clip_norm_sums_over_shards(oracle):
    """Each rank adds its shard's sum of squares; the total is the norm over P."""
    rng = np.random.Generator(np.random.PCG64(5))
    g = (rng.standard_normal(10000)).astype(np.float32)
    whole = oracle.grad_sqnorm(g)
    parts = 0.0
    for lo in range(0, 10000, 2500):
        parts = oracle.grad_sqnorm(g[lo:lo + 2500], parts)
    assert parts == whole                     # same order of additions
    # partial sums added in another order agree to rounding
    ranks = [oracle.grad_sqnorm(g[lo:lo + 2500]) for lo in range(0, 10000, 2500)]
    assert abs(sum(ranks[::-1]) - whole) <= 1e-12 * whole
