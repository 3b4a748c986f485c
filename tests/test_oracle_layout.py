"""Pins of the oracle's partition of the flat buffer.

The partition definition ("DeepSpeed ZeRO Stages" sec. 2): disjoint shards
P_1..P_Nd whose union is the index set, each of about Psi / N_d elements.
Padding reading: Psi is padded to the least multiple of N_d * align and cut
into equal contiguous shards.  Checked here by brute force (element-by-element
owner maps built by walking the buffer) and by properties that fix the answer
uniquely.  CPU only.
"""
import numpy as np
import pytest

from zero_partitioned_mixed_partition_gb300 import synth


def _brute_force(numels, n_d, align):
    """Walk the padded buffer one element at a time, cutting a new shard every
    time the current one reaches the common size; returns per-element
    (tensor, index-in-tensor, shard, index-in-shard) rows for real elements."""
    psi = sum(numels)
    unit = n_d * align
    psi_pad = psi
    while psi_pad % unit:
        psi_pad += 1
    size = psi_pad // n_d
    rows = []
    shard, pos = 0, 0
    for t, n in enumerate(numels):
        for i in range(n):
            if pos == size:
                shard, pos = shard + 1, 0
            rows.append((t, i, shard, pos))
            pos += 1
    return psi, psi_pad, size, rows


def _expand(fr):
    rows = []
    for f in fr:
        for k in range(int(f["length"])):
            rows.append((int(f["tensor"]), int(f["tensor_offset"]) + k, int(f["shard"]),
                         int(f["shard_offset"]) + k))
    return rows


TINY_CASES = []
_rng = np.random.Generator(np.random.PCG64(21))
for _ in range(40):
    t = int(_rng.integers(0, 9))
    numels = [int(x) for x in _rng.integers(0, 700, size=t)]
    if t and _rng.random() < 0.3:
        numels[int(_rng.integers(0, t))] = 0
    n_d = int(_rng.choice([1, 2, 3, 4, 7, 16]))
    align = int(_rng.choice([1, 2, 128]))
    TINY_CASES.append((numels, n_d, align))
TINY_CASES += [([], 4, 1), ([0, 0], 3, 2), ([1], 16, 128), ([4096], 4, 1), ([5, 5, 5], 3, 1)]


@pytest.mark.parametrize("numels,n_d,align", TINY_CASES)
def test_layout_brute_force(oracle, numels, n_d, align):
    psi, psi_pad, size, rows = _brute_force(numels, n_d, align)
    lay = oracle.layout(numels, n_d, align)
    assert lay["psi"] == psi and lay["psi_pad"] == psi_pad and lay["shard_numel"] == size
    assert list(lay["shard_offsets"]) == [i * size for i in range(n_d + 1)]
    assert list(lay["tensor_offsets"]) == [int(x) for x in np.cumsum([0] + numels[:-1])][: len(numels)]
    assert _expand(lay["fragments"]) == rows


@pytest.mark.parametrize("name", ["tiny", "gpt2s", "ragged", "xl", "7b5"])
def test_layout_invariants_on_workloads(oracle, name):
    w = synth.WORKLOADS[name]
    numels = np.asarray(w.numels, np.int64)
    lay = oracle.layout(w.numels, w.n_d, w.align)
    psi, psi_pad, s = lay["psi"], lay["psi_pad"], lay["shard_numel"]
    unit = w.n_d * w.align
    # least multiple of N_d * align that holds Psi
    assert psi == int(numels.sum()) and psi_pad % unit == 0 and psi <= psi_pad < psi + unit
    assert s * w.n_d == psi_pad and s % w.align == 0
    fr = lay["fragments"]
    # disjoint and covering: per tensor the fragments tile [0, numel) in order,
    # and flat positions are strictly increasing and contiguous
    flat = fr["shard"].astype(np.int64) * s + fr["shard_offset"]
    assert np.all(flat[1:] == flat[:-1] + fr["length"][:-1])
    assert flat[0] == 0 and flat[-1] + fr["length"][-1] == psi
    assert np.all(fr["length"] > 0) and np.all(fr["shard_offset"] + fr["length"] <= s)
    tstart = lay["tensor_offsets"][fr["tensor"]] + fr["tensor_offset"]
    assert np.array_equal(tstart, flat)
    # near-equal: real elements per shard differ by less than N_d * align
    valid = np.bincount(fr["shard"], weights=fr["length"], minlength=w.n_d)
    assert valid.sum() == psi and valid.max() - valid.min() < unit


def test_layout_workload_shard_sizes(oracle):
    # shard sizes the workload statements give
    assert oracle.layout(synth.WORKLOADS["tiny"].numels, 4, 128)["shard_numel"] == 262_144
    assert oracle.layout(synth.WORKLOADS["xl"].numels, 4, 128)["shard_numel"] == 375_000_064
    lay = oracle.layout(synth.WORKLOADS["7b5"].numels, 64, 128)
    assert lay["shard_numel"] == 117_187_584
    assert lay["shard_offsets"][17] == 1_992_188_928
    g2 = oracle.layout(synth.WORKLOADS["gpt2s"].numels, 8, 128)
    assert g2["psi"] == 124_419_840 and abs(g2["psi"] - 124e6) < 1e6


def test_layout_rejects_bad_arguments(oracle):
    for args in (([1, 2], 0, 1), ([1, 2], 2, 3), ([1, 2], 2, 0), ([1, -2], 2, 1)):
        with pytest.raises(ValueError):
            oracle.layout(*args)


def test_sharded_step_equals_unsharded(oracle):
    """Fact 1 ("DeepSpeed ZeRO Stages" sec. 2.1): stepping every shard on its
    own equals one update of the whole buffer, bit for bit."""
    numels = [3000, 17, 0, 5100, 1, 999]
    n_d, align = 4, 8
    lay = oracle.layout(numels, n_d, align)
    psi, s = lay["psi"], lay["shard_numel"]
    rng = np.random.Generator(np.random.PCG64(1))
    full_contrib = [(rng.standard_normal(lay["psi_pad"]) * 100).astype(np.float16).view(np.uint16)
                    for _ in range(n_d)]
    theta0 = rng.standard_normal(lay["psi_pad"]).astype(np.float32)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, loss_scale=128.0)

    whole = [theta0[:psi].copy(), np.zeros(psi, np.float32), np.zeros(psi, np.float32)]
    whole_p = np.zeros(psi, np.uint16)
    pieces = [theta0.copy(), np.zeros_like(theta0), np.zeros_like(theta0)]
    pieces_p = np.zeros(lay["psi_pad"], np.uint16)
    for t in (1, 2):
        oracle.shard_step([c[:psi] for c in full_contrib], *whole, whole_p, step=t, **hp)
        for r in range(n_d):
            lo = r * s
            valid = max(0, min(psi - lo, s))
            views = [a[lo:lo + s] for a in pieces]
            pv = pieces_p[lo:lo + s]
            sl = [c[lo:lo + s].copy() for c in full_contrib]
            state = [v.copy() for v in views]
            pp = pv.copy()
            oracle.shard_step(sl, *state, pp, step=t, n=valid, **hp)
            for dst, src in zip(views, state):
                dst[:] = src
            pv[:] = pp
    for a, b in zip(whole, pieces):
        assert np.array_equal(a, b[:psi])
    assert np.array_equal(whole_p, pieces_p[:psi])
    assert not pieces[0][psi:].any() or np.array_equal(pieces[0][psi:], theta0[psi:])
