"""Pins of the oracle's mixed-precision SGD with momentum (the optimizer the
state multiplier K names beside Adam, "DeepSpeed ZeRO Stages" sec. 1.2):
torch.optim.SGD in float64 (textbook, a library routine), closed forms, and a
hand-traced dyadic case.  CPU only."""
import numpy as np
import pytest
import torch


@pytest.mark.parametrize("mu,wd", [(0.9, 0.0), (0.9, 0.01), (0.0, 0.0)])
def test_sgd_matches_torch(oracle, mu, wd):
    n, steps, lr = 3000, 4, 0.05
    rng = np.random.Generator(np.random.PCG64(21))
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    grads = [(sign * rng.uniform(0.05, 2.0, n)).astype(np.float16) for _ in range(steps)]
    theta0 = rng.uniform(2.0, 3.0, n).astype(np.float32) * sign.astype(np.float32)  # stays away from 0
    p = torch.nn.Parameter(torch.tensor(theta0.astype(np.float64)))
    opt = torch.optim.SGD([p], lr=lr, momentum=mu, weight_decay=wd, foreach=False)
    master, mom = theta0.copy(), np.zeros(n, np.float32)
    params = np.zeros(n, np.uint16)
    for t in range(steps):
        p.grad = torch.tensor(grads[t].astype(np.float64))
        opt.step()
        g, _ = oracle.grad_reduce([grads[t].view(np.uint16)], 1.0)
        oracle.sgd_apply(g, master, mom, params, lr=lr, momentum=mu, weight_decay=wd)
        np.testing.assert_allclose(master.astype(np.float64), p.detach().numpy(), rtol=2e-6, atol=1e-9)
        if mu:
            np.testing.assert_allclose(mom.astype(np.float64), opt.state[p]["momentum_buffer"].numpy(),
                                       rtol=2e-6, atol=1e-9)
    assert np.array_equal(params, master.astype(np.float16).view(np.uint16))


def test_sgd_constant_gradient_closed_form(oracle):
    """wd = 0, constant g: b_t = g (1 - mu^t) / (1 - mu) and
    theta_t = theta_0 - lr g sum_{s<=t} (1 - mu^s) / (1 - mu)."""
    n, mu, lr = 512, 0.5, 0.25
    g = np.linspace(-2, 2, n).astype(np.float32)
    master, mom = np.full(n, 10.0, np.float32), np.zeros(n, np.float32)   # no cancellation near 0
    acc = 0.0
    for t in range(1, 6):
        oracle.sgd_apply(g.copy(), master, mom, None, lr=lr, momentum=mu, weight_decay=0.0)
        b = g.astype(np.float64) * (1 - mu ** t) / (1 - mu)
        acc += (1 - mu ** t) / (1 - mu)
        np.testing.assert_allclose(mom, b, rtol=1e-6, atol=1e-9)
        np.testing.assert_allclose(master, 10.0 - lr * g.astype(np.float64) * acc, rtol=1e-6, atol=1e-9)


def test_sgd_hand_traced_dyadic(oracle):
    # mu = 0.5, lr = 0.5, wd = 0.25, theta0 = 2, g = 1, 1, 1:
    #   d1 = 1 + 0.5 = 1.5,  b1 = 1.5,   th1 = 2 - 0.75 = 1.25
    #   d2 = 1 + 0.3125 = 1.3125, b2 = 0.75 + 1.3125 = 2.0625, th2 = 1.25 - 1.03125 = 0.21875
    #   d3 = 1 + 0.0546875 = 1.0546875, b3 = 1.03125 + 1.0546875 = 2.0859375,
    #   th3 = 0.21875 - 1.04296875 = -0.82421875
    master, mom = np.array([2.0], np.float32), np.zeros(1, np.float32)
    want = [(1.5, 1.25), (2.0625, 0.21875), (2.0859375, -0.82421875)]
    for b, th in want:
        oracle.sgd_apply(np.ones(1, np.float32), master, mom, None, lr=0.5, momentum=0.5, weight_decay=0.25)
        assert mom[0] == b and master[0] == th
