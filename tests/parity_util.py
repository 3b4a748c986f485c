"""Comparison helpers for the CUDA-vs-oracle parity tests.

Tolerances (the stated bar): shard offsets and overflow flags bit-exact; fp16
parameters within 1 ulp; fp32 master, m and v within |a - b| <= 1e-9 + 2e-6 |b|.
The kernel performs the oracle's operations in the oracle's order with one
IEEE rounding each, so the tests also record the largest ulp distance seen
(expected 0) in ``MAX_ULP``.
"""
import numpy as np
import torch

RTOL, ATOL = 2e-6, 1e-9
MAX_ULP = {"f32": 0, "f16": 0}


def _ordered(bits: np.ndarray, width: int) -> np.ndarray:
    """Map IEEE bit patterns to integers whose difference is the ulp distance."""
    b = bits.astype(np.int64)
    sign = 1 << (width - 1)
    return np.where(b & sign, -(b & (sign - 1)), b)


def ulp_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(_ordered(a.view(np.uint32), 32) - _ordered(b.view(np.uint32), 32))


def ulp_f16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(_ordered(a_bits.astype(np.uint16), 16) - _ordered(b_bits.astype(np.uint16), 16))


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def f16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_f32_close(got: np.ndarray, ref: np.ndarray, what: str):
    got = np.asarray(got, np.float32)
    ref = np.asarray(ref, np.float32)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    bad = ~(np.abs(got.astype(np.float64) - ref.astype(np.float64)) <= ATOL + RTOL * np.abs(ref.astype(np.float64)))
    both_nan = np.isnan(got) & np.isnan(ref)
    bad &= ~both_nan
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside tolerance; first at {i}: "
                             f"got {got[i]!r} want {ref[i]!r}")
    finite = np.isfinite(got) & np.isfinite(ref)
    if finite.any():
        MAX_ULP["f32"] = max(MAX_ULP["f32"], int(ulp_f32(got[finite], ref[finite]).max()))


def assert_f16_close(got_bits: np.ndarray, ref_bits: np.ndarray, what: str):
    d = ulp_f16(got_bits, ref_bits)
    if (d > 1).any():
        i = int(np.flatnonzero(d > 1)[0])
        raise AssertionError(f"{what}: {int((d > 1).sum())} fp16 values more than 1 ulp apart; first at {i}: "
                             f"got {got_bits[i]:#06x} want {ref_bits[i]:#06x}")
    if d.size:
        MAX_ULP["f16"] = max(MAX_ULP["f16"], int(d.max()))


class OracleShard:
    """Host copy of one shard's state, stepped by the oracle."""

    def __init__(self, oracle, master0: np.ndarray):
        self.oracle = oracle
        self.master = np.array(master0, np.float32, copy=True)
        self.m = np.zeros_like(self.master)
        self.v = np.zeros_like(self.master)
        self.params = oracle.f32_to_f16(self.master)

    def reduce(self, contribs, loss_scale):
        return self.oracle.grad_reduce(contribs, loss_scale, n=self.master.size)

    def apply(self, g, w, step):
        self.oracle.adam_apply(g, self.master, self.m, self.v, self.params, lr=w.lr, beta1=w.beta1,
                               beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, step=step)

    def compare(self, master, m, v, params_bits, what=""):
        assert_f32_close(master, self.master, f"{what} master")
        assert_f32_close(m, self.m, f"{what} m")
        assert_f32_close(v, self.v, f"{what} v")
        assert_f16_close(params_bits, self.params, f"{what} params")


def oracle_group_step(oracle, shards, contribs_per_shard, w, loss_scale, applied):
    """One oracle step over several shards that commit or skip together.
    Returns (overflow, new loss scale, new applied-step count)."""
    reduced, ovf = [], 0
    for sh, contribs in zip(shards, contribs_per_shard):
        g, bad = sh.reduce(contribs, loss_scale)
        reduced.append(g)
        ovf |= bad
    if not ovf:
        for sh, g in zip(shards, reduced):
            sh.apply(g, w, applied + 1)
    loss_scale, applied = oracle.commit(ovf, loss_scale, applied)
    return ovf, loss_scale, applied
