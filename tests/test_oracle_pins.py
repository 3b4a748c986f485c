"""Pins of the oracle to facts that do not come from the oracle itself.

Each test names what fixes the expected value: a number printed on the pages
(tests/golden/, with its citation), a closed form of the update rule, an
exhaustive comparison with numpy's binary16 conversion, the textbook Adam of
torch.optim in float64, or brute force on tiny inputs.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- state bytes

def _read_golden_state_bytes():
    rows = []
    with open(os.path.join(GOLDEN, "state_bytes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            vals, cite = line.split("|", 1)
            psi, n_d, stage, k, gb, tol = vals.split()
            rows.append((float(psi), int(n_d), int(stage), float(k), float(gb), float(tol), cite.strip()))
    return rows


@pytest.mark.parametrize("row", _read_golden_state_bytes(), ids=lambda r: f"{r[0]:g}-N{r[1]}-s{r[2]}")
def test_state_bytes_printed_values(oracle, row):
    psi, n_d, stage, k, gb, tol, cite = row
    got = oracle.state_bytes(psi, n_d, stage, k) / 1e9
    assert abs(got - gb) <= tol, (got, gb, cite)


def test_state_bytes_limits(oracle):
    # "At N = 1 ... the formula returns 16 Psi" (ZeRO Stage 1 Math, The memory math):
    # with one rank every stage stores everything.
    for stage in range(4):
        assert oracle.state_bytes(1e9, 1, stage, 12) == 16e9
    # plain DP does not depend on N_d
    assert oracle.state_bytes(1e9, 7, 0, 12) == oracle.state_bytes(1e9, 1024, 0, 12) == 16e9
    # large N_d: the floors 4 Psi (stage 1), 2 Psi (stage 2) and 0 (stage 3)
    big = 1 << 30
    assert abs(oracle.state_bytes(1e9, big, 1, 12) - 4e9) < 100.0
    assert abs(oracle.state_bytes(1e9, big, 2, 12) - 2e9) < 100.0
    assert oracle.state_bytes(1e9, big, 3, 12) < 100.0
    # optimizer-state share of a 7B model drops from 84 GB to about 1.31 GB at
    # N_d = 64 (ZeRO Optimization: Stages 1, 2, and 3 Explained, Stage 1)
    drop = oracle.state_bytes(7e9, 1, 1, 12) - oracle.state_bytes(7e9, 64, 1, 12)
    assert abs(drop / 1e9 - (84.0 - 1.3125)) < 1e-9
    # K is a free multiplier: SGD with momentum (K = 4) at stage 0 is 8 Psi
    assert oracle.state_bytes(1e9, 8, 0, 4) == 8e9


def test_state_bytes_bad_stage_is_nan(oracle):
    # the pages' Python raises for a stage outside 0..3; the oracle answers NaN
    assert math.isnan(oracle.state_bytes(1e9, 4, 4, 12))
    assert math.isnan(oracle.state_bytes(1e9, 4, -1, 12))
    assert math.isnan(oracle.state_bytes(1e9, 0, 1, 12))


def test_state_bytes_page_conflict_7b_stage2(oracle):
    # ZeRO Optimization: Stages 1, 2, and 3 Explained prints "roughly 14.9 GB"
    # for stage 2 of a 7B model on 64 GPUs, but its own formula
    # 2 Psi + (2 Psi + 12 Psi) / N_d gives 14 + 1.53125 GB.  The formula wins.
    got = oracle.state_bytes(7e9, 64, 2, 12) / 1e9
    assert abs(got - 15.53125) < 1e-9
    assert abs(got - 14.9) > 0.5


# ------------------------------------------------------------------- fp16

def test_f16_decode_exhaustive(oracle):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = oracle.f16_to_f32(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _f16_probe_values():
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    h = h[np.isfinite(h)].astype(np.float64)
    h = np.unique(h)
    mids = (h[:-1] + h[1:]) / 2.0          # exact ties (binary16 neighbours)
    vals = [h, mids]
    for d in (-1, 1):                      # one float32 ulp either side of each tie
        vals.append(np.nextafter(mids.astype(np.float32), np.float32(d * np.inf)).astype(np.float64))
    vals.append(np.array([65504.0, 65519.99, 65520.0, 65536.0, 1e30, 2.0 ** -25, 2.0 ** -26,
                          3 * 2.0 ** -26, 2.0 ** -24 * 1.5, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -11)]))
    rng = np.random.Generator(np.random.PCG64(11))
    vals.append(rng.standard_normal(1 << 18) * 10.0 ** rng.uniform(-9, 5, 1 << 18))
    v = np.concatenate(vals).astype(np.float32)
    return np.concatenate([v, -v])


def test_f16_encode_matches_numpy(oracle):
    x = _f16_probe_values()
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = oracle.f32_to_f16(x)
    assert np.array_equal(got, ref)


def test_f16_encode_specials(oracle):
    x = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0], np.float32)
    got = oracle.f32_to_f16(x)
    assert got[0] == 0x7C00 and got[1] == 0xFC00
    assert (got[2] & 0x7C00) == 0x7C00 and (got[2] & 0x03FF) != 0
    assert got[3] == 0x0000 and got[4] == 0x8000


# ------------------------------------------------ hand-traced Adam / AdamW

def _read_dyadic():
    rows = []
    with open(os.path.join(GOLDEN, "adam_dyadic.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, wd0, wd5, mv = line.split("|")
            j, h0, h1, h2, g, u, th0 = head.split()
            rows.append(dict(h=(float(h0), float(h1), float(h2)), g=float(g), u=float(u),
                             th0=float(th0), wd0=[float(x) for x in wd0.split()],
                             wd5=[float(x) for x in wd5.split()],
                             m3=float(mv.split()[0]), v3=float(mv.split()[1])))
    return rows


@pytest.mark.parametrize("wd,key", [(0.0, "wd0"), (0.5, "wd5")])
def test_adam_hand_traced_dyadic(oracle, wd, key):
    rows = _read_dyadic()
    contribs = [np.array([r["h"][k] for r in rows], np.float16).view(np.uint16) for k in range(3)]
    master = np.array([r["th0"] for r in rows], np.float32)
    m = np.zeros(8, np.float32)
    v = np.zeros(8, np.float32)
    params = np.zeros(8, np.uint16)
    g, bad = oracle.grad_reduce(contribs, 1.0)
    assert bad == 0
    assert np.array_equal(g, np.array([r["g"] for r in rows], np.float32))
    for t in (1, 2, 3):
        ovf = oracle.shard_step(contribs, master, m, v, params, lr=0.5, beta1=0.5, beta2=0.75,
                                eps=2.0, weight_decay=wd, loss_scale=1.0, step=t)
        assert ovf == 0
        want = np.array([r[key][t - 1] for r in rows], np.float32)
        assert np.array_equal(master, want), (t, master, want)
        assert np.array_equal(params, want.astype(np.float16).view(np.uint16))
    assert np.array_equal(m, np.array([r["m3"] for r in rows], np.float32))
    assert np.array_equal(v, np.array([r["v3"] for r in rows], np.float32))


# --------------------------------------- textbook Adam (torch.optim, float64)

@pytest.mark.parametrize("wd", [0.0, 0.1])
def test_adam_matches_torch_textbook(oracle, wd):
    """N_d = 1, loss scale 1: the step is textbook Adam (AdamW when wd > 0).
    Gradients keep one sign per coordinate so m never cancels to ~0 and the
    fp32 oracle stays within the 2e-6 relative bar of the float64 reference."""
    n, steps = 4096, 3
    rng = np.random.Generator(np.random.PCG64(5))
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    grads = [(sign * rng.uniform(0.05, 4.0, n)).astype(np.float16) for _ in range(steps)]
    theta0 = rng.uniform(-1, 1, n).astype(np.float32)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)

    p = torch.nn.Parameter(torch.tensor(theta0.astype(np.float64)))
    if wd:
        opt = torch.optim.AdamW([p], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                                weight_decay=wd, foreach=False)
    else:
        opt = torch.optim.Adam([p], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                               weight_decay=0.0, foreach=False)
    master, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    params = np.zeros(n, np.uint16)
    for t in range(1, steps + 1):
        p.grad = torch.tensor(grads[t - 1].astype(np.float64))
        opt.step()
        ovf = oracle.shard_step([grads[t - 1].view(np.uint16)], master, m, v, params, weight_decay=wd,
                                loss_scale=1.0, step=t, **hp)
        assert ovf == 0
        st = opt.state[p]
        for got, ref in ((master, p.detach().numpy()), (m, st["exp_avg"].numpy()),
                         (v, st["exp_avg_sq"].numpy())):
            # the stated bar: |a - b| <= 1e-9 + 2e-6 |b|
            np.testing.assert_allclose(got.astype(np.float64), ref, rtol=2e-6, atol=1e-9)


# ------------------------------------------------------------ closed forms

def test_adam_constant_gradient_closed_form(oracle):
    """Constant g: m_t = g (1 - b1^t), v_t = g^2 (1 - b2^t), so m_hat = g,
    v_hat = g^2 and theta_t = theta_0 - t lr g / (|g| + eps)."""
    n, steps, lr, b1, b2, eps = 1024, 6, 1e-3, 0.9, 0.999, 1e-8
    rng = np.random.Generator(np.random.PCG64(9))
    h = (rng.standard_normal(n) * 3).astype(np.float16)
    h[0] = 0.0
    g = h.astype(np.float64)
    theta0 = rng.uniform(-2, 2, n).astype(np.float32)
    master, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    params = np.zeros(n, np.uint16)
    for t in range(1, steps + 1):
        oracle.shard_step([h.view(np.uint16)], master, m, v, params, lr=lr, beta1=b1, beta2=b2, eps=eps,
                          weight_decay=0.0, loss_scale=1.0, step=t)
        np.testing.assert_allclose(m, g * (1 - b1 ** t), rtol=2e-6, atol=0)
        np.testing.assert_allclose(v, g * g * (1 - b2 ** t), rtol=2e-6, atol=0)
        want = theta0.astype(np.float64) - t * lr * g / (np.abs(g) + eps)
        np.testing.assert_allclose(master, want, rtol=2e-6, atol=1e-9)
    assert master[0] == theta0[0]  # g = 0 leaves theta alone


def test_adamw_zero_gradient_is_pure_decay(oracle):
    """g = 0: m = v = 0, u = 0, so AdamW gives theta_t = theta_0 (1 - lr wd)^t."""
    n, lr, wd = 512, 0.01, 0.1
    theta0 = np.linspace(-1, 1, n).astype(np.float32)
    zero = np.zeros(n, np.float16).view(np.uint16)
    master, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, 5):
        oracle.shard_step([zero, zero], master, m, v, None, lr=lr, beta1=0.9, beta2=0.999, eps=1e-8,
                          weight_decay=wd, loss_scale=1024.0, step=t)
        np.testing.assert_allclose(master, theta0 * (1 - lr * wd) ** t, rtol=2e-6, atol=0)
        assert not m.any() and not v.any()


def test_update_direction_opposes_gradient(oracle):
    n = 256
    rng = np.random.Generator(np.random.PCG64(3))
    h = rng.uniform(0.5, 2, n).astype(np.float16) * np.where(np.arange(n) % 2, 1, -1).astype(np.float16)
    master = np.zeros(n, np.float32)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    oracle.shard_step([h.view(np.uint16)], master, m, v, None, lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8,
                      weight_decay=0.0, loss_scale=1.0, step=1)
    assert np.all(np.sign(master) == -np.sign(h.astype(np.float32)))


# ------------------------------------------- reduction, averaging, unscale

def test_average_of_identical_contributions(oracle):
    """N_d identical contributions h with N_d and L powers of two average to
    exactly h / L: the result equals N_d = 1, L = 1 fed with h / L."""
    n = 2048
    rng = np.random.Generator(np.random.PCG64(4))
    h = (rng.standard_normal(n) * 64).astype(np.float16)
    for n_d, L in ((2, 1.0), (4, 65536.0), (8, 1024.0), (64, 32768.0)):
        g, bad = oracle.grad_reduce([h.view(np.uint16)] * n_d, L)
        assert bad == 0
        assert np.array_equal(g, (h.astype(np.float64) / L).astype(np.float32))


def test_loss_scale_invariance(oracle):
    """Contributions scaled by a power-of-two L and unscaled by L give the
    same step, bit for bit, as unscaled contributions with L = 1."""
    n = 1024
    rng = np.random.Generator(np.random.PCG64(8))
    base = [(rng.standard_normal(n) * 0.5).astype(np.float16) for _ in range(3)]
    scaled = [(b.astype(np.float32) * 256).astype(np.float16) for b in base]
    theta0 = rng.uniform(-1, 1, n).astype(np.float32)
    out = []
    for contribs, L in ((base, 1.0), (scaled, 256.0)):
        master, m, v = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
        oracle.shard_step([c.view(np.uint16) for c in contribs], master, m, v, None, lr=1e-3, beta1=0.9,
                          beta2=0.999, eps=1e-8, weight_decay=0.0, loss_scale=L, step=1)
        out.append((master, m, v))
    for a, b in zip(*out):
        assert np.array_equal(a, b)


def test_sum_in_rank_order(oracle):
    """Contributions are accumulated in fp32 in rank order 0..N_d-1:
    (65504, 2^-24, -65504, 0) sums to exactly 0 (the tiny term is absorbed),
    (65504, -65504, 2^-24, 0) to 2^-24, which averages to 2^-26 over N_d = 4."""
    tiny = np.float16(2.0 ** -24)
    big, neg, zero = (np.array([x], np.float16) for x in (65504.0, -65504.0, 0.0))
    t = np.array([tiny], np.float16)
    g, _ = oracle.grad_reduce([x.view(np.uint16) for x in (big, t, neg, zero)], 1.0)
    assert g[0] == 0.0
    g, _ = oracle.grad_reduce([x.view(np.uint16) for x in (big, neg, t, zero)], 1.0)
    assert g[0] == np.float32(2.0 ** -26)


def test_fp32_accumulate_does_not_overflow(oracle):
    """64 contributions of 65504 overflow fp16 but not the fp32 accumulator."""
    h = np.full(4, 65504.0, np.float16).view(np.uint16)
    g, bad = oracle.grad_reduce([h] * 64, 1.0)
    assert bad == 0
    assert np.all(g == np.float32(65504.0))


# -------------------------------------------------------- overflow / skip

@pytest.mark.parametrize("where", [0, 5, 8, 12])
@pytest.mark.parametrize("kind", ["inf", "-inf", "nan", "inf-inf"])
def test_overflow_detection_and_skip(oracle, where, kind):
    n = 13
    rng = np.random.Generator(np.random.PCG64(where))
    contribs = [(rng.standard_normal(n)).astype(np.float16) for _ in range(3)]
    if kind == "inf":
        contribs[1][where] = np.inf
    elif kind == "-inf":
        contribs[2][where] = -np.inf
    elif kind == "nan":
        contribs[0][where] = np.nan
    else:
        contribs[0][where] = np.inf
        contribs[2][where] = -np.inf
    master = rng.standard_normal(n).astype(np.float32)
    m = rng.standard_normal(n).astype(np.float32)
    v = rng.uniform(0, 1, n).astype(np.float32)
    params = master.astype(np.float16).view(np.uint16)
    before = [a.copy() for a in (master, m, v, params)]
    ovf = oracle.shard_step([c.view(np.uint16) for c in contribs], master, m, v, params, lr=1e-3,
                            beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, loss_scale=4.0, step=3)
    assert ovf == 1
    for a, b in zip((master, m, v, params), before):
        assert np.array_equal(a, b)
    # a finite tail element beyond n is never looked at
    g, bad = oracle.grad_reduce([c.view(np.uint16) for c in contribs], 4.0, n=where)
    assert bad == 0


def test_commit_bookkeeping(oracle):
    ls, t = 65536.0, 3
    ls, t = oracle.commit(1, ls, t)
    assert (ls, t) == (32768.0, 3)
    ls, t = oracle.commit(0, ls, t)
    assert (ls, t) == (32768.0, 4)
    ls, t = oracle.commit(1, 1.5, t)
    assert (ls, t) == (1.0, 4)        # never below 1
    ls, t = oracle.commit(1, 1.0, t)
    assert (ls, t) == (1.0, 4)
