"""Seeded synthetic inputs and the workload table.

This module is shared by the tests, the benchmark and the oracle-side checks.
It holds NO arithmetic of the method: it only describes the workloads (tensor
lists, data-parallel degree, hyper-parameters) and draws seeded random inputs
of the stated distributions.  It imports neither the CUDA binding nor the
oracle.

Workloads (all inputs synthetic; no dataset or checkpoint is involved):

  tiny     one flat buffer of 1,048,576 params, N_d = 4, device plays rank 1;
           grads fp16 ~ N(0, 1e-3) * 65536, fresh per (step, rank);
           master ~ N(0, 0.02); Adam 0.9 / 0.999 / lr 1e-3 / eps 1e-8; 3 steps
  gpt2s    GPT-2-small-shaped list of 110 tensors (124,419,840 params),
           N_d = 8, rank 3; grads ~ N(0, 1e-3) * 2^16 fresh per step;
           AdamW lr 6e-4, wd 0.1; 10 steps
  ragged   4096 tensors with log-uniform numels in [1, 2^20] (seed 7),
           N_d = 16, every shard stepped each step; grads ~ Laplace(0, 5e-4)
           * 2^14 drawn once; master ~ U(-0.05, 0.05); 5 steps
  xl       one flat buffer of 1.5e9 params (GPT-2-XL scale), N_d = 4, rank 0;
           grads ~ N(0, 1e-3) * 2^16 drawn once; a +inf is placed in rank 2's
           slice at step 4 and removed at step 5; lr 1e-4; 8 steps
  7b5      LLaMA-7B-shaped list (32 layers, d 4096, ffn 11008, vocab 32000)
           padded by one extra tensor to 7.5e9 params, N_d = 64, rank 17;
           grads ~ N(0, 5e-4) * 2^15 drawn once; AdamW lr 3e-4, beta2 0.95,
           wd 0.1; 5 steps
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    numels: tuple            # tensor sizes in list order
    n_d: int                 # simulated data-parallel ranks
    rank: Optional[int]      # the rank the device plays; None = every shard in turn
    align: int               # shard alignment in elements
    steps: int
    lr: float
    beta1: float
    beta2: float
    eps: float
    weight_decay: float
    loss_scale: float
    grad_dist: str           # "normal" | "laplace"
    grad_std: float          # std (normal) or scale b (laplace) before the loss scale
    grad_mult: float         # loss-scale factor the synthetic gradients carry
    grads_fresh_per_step: bool
    master_dist: str         # "normal" | "uniform"
    master_param: float      # std (normal) or half-width (uniform)
    seed: int
    inf_at: Optional[tuple] = None   # (step, rank, element of the shard) where a +inf is placed

    @property
    def psi(self) -> int:
        return int(sum(self.numels))


def _gpt2_small_numels() -> List[int]:
    d, vocab, ctx, ffn = 768, 50257, 1024, 3072
    out = [vocab * d, ctx * d]
    for _ in range(12):
        out += [2 * d,              # ln (one 2 x 768 tensor per block)
                d * 3 * d, 3 * d,   # qkv weight, bias
                d * d, d,           # attention projection weight, bias
                d * ffn, ffn,       # fc weight, bias
                ffn * d, d]         # out weight, bias
    return out


def ragged_numels(n: int = 4096, seed: int = 7, max_exp: int = 20) -> List[int]:
    """Log-uniform integer sizes in [1, 2^max_exp] (floor of exp(U ln 2^max_exp))."""
    u = np.random.Generator(np.random.PCG64(seed)).random(n)
    vals = np.floor(np.exp(u * (max_exp * math.log(2.0)))).astype(np.int64)
    return [int(x) for x in np.clip(vals, 1, 2 ** max_exp)]


def _llama7b_padded_numels(total: int = 7_500_000_000) -> List[int]:
    d, ffn, vocab = 4096, 11008, 32000
    out = [vocab * d]
    for _ in range(32):
        out += [d * d, d * d, d * d, d * d,   # q, k, v, o
                ffn * d, ffn * d, d * ffn,    # gate, up, down
                d, d]                         # two norms
    out += [d, vocab * d]                     # final norm, lm head
    out.append(total - sum(out))              # one pad tensor up to the stated size
    return out


WORKLOADS = {
    "tiny": Workload("tiny", (1_048_576,), 4, 1, 128, 3, 1e-3, 0.9, 0.999, 1e-8, 0.0, 65536.0,
                     "normal", 1e-3, 65536.0, True, "normal", 0.02, 0),
    "gpt2s": Workload("gpt2s", tuple(_gpt2_small_numels()), 8, 3, 128, 10, 6e-4, 0.9, 0.999, 1e-8,
                      0.1, 65536.0, "normal", 1e-3, 65536.0, True, "normal", 0.02, 2),
    "ragged": Workload("ragged", tuple(ragged_numels()), 16, None, 128, 5, 1e-3, 0.9, 0.999, 1e-8,
                       0.0, 16384.0, "laplace", 5e-4, 16384.0, False, "uniform", 0.05, 7),
    "xl": Workload("xl", (1_500_000_000,), 4, 0, 128, 8, 1e-4, 0.9, 0.999, 1e-8, 0.0, 65536.0,
                   "normal", 1e-3, 65536.0, False, "normal", 0.02, 4,
                   inf_at=(4, 2, 187_500_000)),
    "7b5": Workload("7b5", tuple(_llama7b_padded_numels()), 64, 17, 128, 5, 3e-4, 0.9, 0.95, 1e-8,
                    0.1, 32768.0, "normal", 5e-4, 32768.0, False, "normal", 0.02, 5),
}


def subseed(*ids: int) -> int:
    """Mix integers into one 63-bit seed (splitmix64 finaliser over the list)."""
    x = 0x9E3779B97F4A7C15
    mask = (1 << 64) - 1
    for i in ids:
        x = (x + (int(i) & mask) + 0x9E3779B97F4A7C15) & mask
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
        x = z ^ (z >> 31)
    return x & ((1 << 63) - 1)


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def grad_contribution(w: Workload, n: int, rank: int, step: int, *, shard: int = 0,
                      device="cpu", n_alloc: Optional[int] = None) -> torch.Tensor:
    """fp16 gradient contribution of simulated rank ``rank`` for one shard.

    Values beyond ``n`` (up to ``n_alloc``) are zero padding.  ``step`` is
    ignored when the workload draws its gradients once."""
    n_alloc = n if n_alloc is None else n_alloc
    s = step if w.grads_fresh_per_step else 0
    gen = _generator(subseed(w.seed, 1, shard, rank, s), device)
    out = torch.zeros(n_alloc, dtype=torch.float16, device=device)
    if n == 0:
        return out
    if w.grad_dist == "normal":
        x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        x.mul_(w.grad_std * w.grad_mult)
    elif w.grad_dist == "laplace":
        u = torch.rand(n, generator=gen, device=device, dtype=torch.float32).sub_(0.5)
        # inverse CDF of Laplace(0, b): -b sign(u) log(1 - 2|u|)
        x = u.sign().mul_(torch.log1p(u.abs().mul_(-2.0).clamp_(min=-1.0 + 2.0 ** -24)))
        x.mul_(-w.grad_std * w.grad_mult)
    else:
        raise ValueError(w.grad_dist)
    out[:n] = x.to(torch.float16)
    return out


def master_init(w: Workload, n: int, *, shard: int = 0, device="cpu",
                n_alloc: Optional[int] = None) -> torch.Tensor:
    """fp32 master weights of one shard (zero padding beyond ``n``)."""
    n_alloc = n if n_alloc is None else n_alloc
    gen = _generator(subseed(w.seed, 2, shard), device)
    out = torch.zeros(n_alloc, dtype=torch.float32, device=device)
    if n == 0:
        return out
    if w.master_dist == "normal":
        out[:n] = torch.randn(n, generator=gen, device=device, dtype=torch.float32).mul_(w.master_param)
    elif w.master_dist == "uniform":
        out[:n] = torch.rand(n, generator=gen, device=device, dtype=torch.float32).mul_(
            2.0 * w.master_param).sub_(w.master_param)
    else:
        raise ValueError(w.master_dist)
    return out


def random_fp16(n: int, seed: int, scale: float = 1.0, device="cpu") -> torch.Tensor:
    """Generic seeded N(0, scale) fp16 vector for edge-case tests."""
    gen = _generator(subseed(seed, 3), device)
    return torch.randn(n, generator=gen, device=device, dtype=torch.float32).mul_(scale).to(torch.float16)


def random_f32(n: int, seed: int, scale: float = 1.0, device="cpu") -> torch.Tensor:
    gen = _generator(subseed(seed, 4), device)
    return torch.randn(n, generator=gen, device=device, dtype=torch.float32).mul_(scale)


def sample_indices(n: int, count: int, seed: int, tile: int = 2048) -> np.ndarray:
    """Sorted unique sample of [0, n): the ends, tile edges near both ends and
    a seeded uniform draw."""
    if n <= 0:
        return np.zeros(0, np.int64)
    rng = np.random.Generator(np.random.PCG64(seed))
    fixed = [0, 1, 7, 8, 9, n - 9, n - 8, n - 7, n - 2, n - 1]
    for k in range(1, 5):
        fixed += [k * tile - 1, k * tile, n - k * tile, n - k * tile - 1]
    body = rng.integers(0, n, size=count)
    idx = np.concatenate([np.asarray(fixed, np.int64), body])
    idx = idx[(idx >= 0) & (idx < n)]
    return np.unique(idx)


def fp16_bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 view of an fp16 tensor (bit patterns, for the oracle)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def stack_bits(ts: Sequence[torch.Tensor]) -> List[np.ndarray]:
    return [fp16_bits(t) for t in ts]
