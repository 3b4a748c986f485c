"""Device buffers for one workload and its steps through the C ABI.

Plumbing only: torch allocates the memory and draws the seeded inputs
(``synth``); the partition, the fused step and the commit run in the library's
kernels through :mod:`binding`.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

from . import binding, synth


class _Arena:
    """One device allocation carved into buffers of the given (numel, dtype),
    handed out in order by take(); every buffer starts on a 2 MiB boundary."""

    ALIGN = 2 << 20

    def __init__(self, device, specs):
        self.specs = list(specs)
        sizes = [(n * torch.tensor([], dtype=dt).element_size() + self.ALIGN - 1) // self.ALIGN * self.ALIGN
                 for n, dt in self.specs]
        self.offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
        self.storage = torch.empty(int(self.offsets[-1]), dtype=torch.uint8, device=device)
        self.next = 0

    def take(self, dtype) -> torch.Tensor:
        n, dt = self.specs[self.next]
        if dt != dtype:
            raise RuntimeError(f"arena buffer {self.next} is {dt}, {dtype} was asked for")
        off = int(self.offsets[self.next])
        self.next += 1
        nbytes = n * torch.tensor([], dtype=dt).element_size()
        return self.storage[off:off + nbytes].view(dt)


class WorkloadRunner:
    """Simulates one or more ranks of a workload on one GPU.

    For every stepped shard r it holds the N_d fp16 gradient contributions
    (one per simulated rank, S elements each, zero past the shard's real
    parameters), two sets of fp32 master/m/v and the shard's slice of the full
    fp16 parameter buffer, plus one device control block shared by the shards
    (they form one step, committed or skipped together)."""

    def __init__(self, w: synth.Workload, device, shards: Optional[Sequence[int]] = None,
                 with_full_params: bool = True,
                 stream: Optional[torch.cuda.Stream] = None, math: int = binding.ZS_MATH_IEEE):
        self.w = w
        self.device = torch.device(device)
        self.stream = stream
        self.layout = binding.zero_partition_layout(w.numels, w.n_d, w.align)
        lay = self.layout
        self.S = int(lay["shard_numel"])
        if shards is None:
            shards = [w.rank] if w.rank is not None else list(range(w.n_d))
        self.shard_ids = list(shards)
        fr = lay["fragments"]
        valid = np.bincount(fr["shard"], weights=fr["length"], minlength=w.n_d).astype(np.int64)
        self.n_valid = {r: int(valid[r]) for r in self.shard_ids}
        self.hp = binding.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay, math=math)

        nshards_full = w.n_d if with_full_params else len(self.shard_ids)
        self.params_full = torch.zeros(nshards_full * self.S, dtype=torch.float16, device=self.device)
        self.grads = {}
        self.state = {}
        self.views: List[binding.ShardView] = []
        # One arena for every stepped shard's N_d contributions and both state
        # sets, each buffer starting on a 2 MiB boundary: one allocation and a
        # layout that does not depend on the allocator's history.  On the
        # 375M-parameter N_d = 4 shard the fused kernel ran at 6.76-6.80 TB/s
        # from the arena in fresh processes, against 6.70-6.75 TB/s with one
        # allocation per buffer; offsetting the buffers against each other
        # (4 KiB to 32 MiB) changed nothing.
        per_shard = [(self.S, torch.float16)] * w.n_d + [(self.S, torch.float32)] * 6
        arena = _Arena(self.device, per_shard * len(self.shard_ids))
        self._arena = arena
        for i, r in enumerate(self.shard_ids):
            n = self.n_valid[r]
            g = []
            for k in range(w.n_d):
                buf = arena.take(torch.float16)
                buf.copy_(synth.grad_contribution(w, n, k, 1, shard=r, device=self.device, n_alloc=self.S))
                g.append(buf)
            master0 = arena.take(torch.float32)
            master0.copy_(synth.master_init(w, n, shard=r, device=self.device, n_alloc=self.S))
            f32 = lambda: arena.take(torch.float32).zero_()
            master = (master0, f32())
            m = (f32(), f32())
            v = (f32(), f32())
            slot = r if with_full_params else i
            params = self.params_full[slot * self.S:(slot + 1) * self.S]
            self.grads[r] = g
            self.state[r] = (master, m, v, params)
            self.views.append(binding.ShardView(g, master, m, v, params, n))
            binding.zero_params_from_master(master0, params, n, stream=self.stream)
        self.ctrl = binding.new_ctrl(self.device)
        binding.zero_ctrl_init(self.ctrl, w.loss_scale, stream=self.stream)

    def enable_qwz(self):
        """Give every stepped shard an int8 qwZ copy of its fp16 slice (codes
        and per-256 scales) that each step keeps in sync, and quantize the
        initial slice."""
        self.qwz = {}
        views = []
        for view, r in zip(self.views, self.shard_ids):
            n = self.n_valid[r]
            codes = torch.zeros(self.S, dtype=torch.int8, device=self.device)
            scales = torch.zeros((self.S + binding.ZS_QWZ_BLOCK - 1) // binding.ZS_QWZ_BLOCK, dtype=torch.float32,
                                 device=self.device)
            master, m, v, params = self.state[r]
            views.append(binding.ShardView(self.grads[r], master, m, v, params, n, qcodes=codes, qscales=scales))
            binding.zero_qwz_quantize(params, n, codes, scales, stream=self.stream)
            self.qwz[r] = (codes, scales)
        self.views = views

    def enable_adam8(self):
        """Give every stepped shard 8-bit Adam state -- uint8 codes of m and v
        and fp32 scales per 2048-element block, two sets each, all zero (m = v
        = 0) -- beside the shard's fp32 master and fp16 slice, which it shares."""
        self.adam8 = {}
        self.adam8_views = []
        nb = (self.S + binding.ZS_ADAM8_BLOCK - 1) // binding.ZS_ADAM8_BLOCK
        for r in self.shard_ids:
            codes = lambda: torch.zeros(self.S, dtype=torch.uint8, device=self.device)
            scales = lambda: torch.zeros(nb, dtype=torch.float32, device=self.device)
            mc, vc, ms, vs = (codes(), codes()), (codes(), codes()), (scales(), scales()), (scales(), scales())
            master, _, _, params = self.state[r]
            self.adam8[r] = (mc, vc, ms, vs)
            self.adam8_views.append(binding.Adam8View(self.grads[r], master, mc, vc, ms, vs, params,
                                                      self.n_valid[r]))

    # ---------------------------------------------------------------- steps --
    def step(self):
        """One whole step over every stepped shard, stream-ordered."""
        binding.zero_shard_step_async(self.views, self.w.n_d, self.hp, self.ctrl, stream=self.stream)

    def step_sgd(self, hp):
        """One step with SGD with momentum (momentum kept in the m buffers)."""
        binding.zero_shard_step_sgd_async(self.views, self.w.n_d, hp, self.ctrl, stream=self.stream)

    def step_adam8(self):
        """One step with 8-bit Adam states (enable_adam8 first)."""
        binding.zero_shard_step_adam8_async(self.adam8_views, self.w.n_d, self.hp, self.ctrl, stream=self.stream)

    def reduce_adam(self, i: int = 0):
        binding.zero_shard_reduce_adam_async(self.views[i], self.w.n_d, self.hp, self.ctrl, stream=self.stream)

    def reduce_adam_all(self):
        """The fused kernels of every stepped shard (grouped launches), no commit."""
        binding.zero_shard_reduce_adam_all_async(self.views, self.w.n_d, self.hp, self.ctrl, stream=self.stream)

    def commit(self):
        binding.zero_step_commit_async(self.views, self.hp, self.ctrl, stream=self.stream)

    def enable_clipping(self, keep_g: bool):
        """Allocate the squared-norm accumulator (and, with keep_g, one fp32
        buffer per shard for the reduced gradient kept between the passes)."""
        self.sqnorm = binding.new_sqnorm(self.device)
        self.gbuf = None
        if keep_g:
            self.gbuf = [torch.zeros(self.S, dtype=torch.float32, device=self.device) for _ in self.shard_ids]

    def step_clipped(self, max_norm: float):
        """One clipped step over every stepped shard, stream-ordered."""
        binding.zero_shard_step_clipped_async(self.views, self.w.n_d, self.hp, max_norm, self.sqnorm, self.ctrl,
                                              g_dev=self.gbuf, stream=self.stream)

    def clipped_bytes_per_step(self) -> int:
        """Algorithmic HBM bytes of one clipped step: 4 N_d + 26 per element
        when pass 2 re-reduces, 2 N_d + 34 when it reads the kept g."""
        per = (2 * self.w.n_d + 34) if self.gbuf is not None else (4 * self.w.n_d + 26)
        return sum(per * self.n_valid[r] for r in self.shard_ids)

    def refresh_grads(self, step: int):
        """Draw the contributions of ``step`` (workloads with fresh gradients)."""
        for r in self.shard_ids:
            n = self.n_valid[r]
            for k in range(self.w.n_d):
                self.grads[r][k].copy_(synth.grad_contribution(self.w, n, k, step, shard=r, device=self.device,
                                                               n_alloc=self.S))

    def ctrl_host(self) -> dict:
        return binding.read_ctrl(self.ctrl)

    def current(self, r: int):
        """(master, m, v, params) tensors holding the committed state of shard r."""
        cur = self.ctrl_host()["cur"]
        master, m, v, params = self.state[r]
        return master[cur], m[cur], v[cur], params

    def current_adam8(self, r: int):
        """(master, m_codes, v_codes, m_scale, v_scale, params) holding the
        committed 8-bit Adam state of shard r."""
        cur = self.ctrl_host()["cur"]
        master, _, _, params = self.state[r]
        mc, vc, ms, vs = self.adam8[r]
        return master[cur], mc[cur], vc[cur], ms[cur], vs[cur], params

    # ------------------------------------------------------- checkpointing --
    def save(self) -> dict:
        """Host copy of everything a resumed run needs: the control block's
        bytes (loss scale, t, beta^t, ping-pong set, counters) and, per shard,
        the committed master/m/v and the fp16 slice -- plus, with 8-bit Adam
        state (enable_adam8), its committed codes and block scales.  Call with
        the stream idle."""
        torch.cuda.synchronize(self.device)
        cur = self.ctrl_host()["cur"]
        out = {"ctrl": self.ctrl.detach().cpu().clone(), "shards": {}}
        for r in self.shard_ids:
            master, m, v, params = self.state[r]
            out["shards"][r] = tuple(t.detach().cpu().clone() for t in (master[cur], m[cur], v[cur], params))
        if getattr(self, "adam8", None):
            out["adam8"] = {r: tuple(pair[cur].detach().cpu().clone() for pair in self.adam8[r]) for r in self.shard_ids}
        return out

    def load(self, ckpt: dict):
        """Restore a save() of a runner of the same workload: the state goes
        into the set the saved control block names, the control block is
        copied back as bytes; with a qwZ copy (enable_qwz), the copy is
        re-quantized from the loaded fp16 slices."""
        ctrl = ckpt["ctrl"]
        self.ctrl.copy_(ctrl.to(self.device))
        cur = binding.read_ctrl(self.ctrl)["cur"]
        for r, (master, m, v, params) in ckpt["shards"].items():
            dm, dmm, dv, dp = self.state[r]
            dm[cur].copy_(master.to(self.device))
            dmm[cur].copy_(m.to(self.device))
            dv[cur].copy_(v.to(self.device))
            dp.copy_(params.to(self.device))
        if "adam8" in ckpt:
            if not getattr(self, "adam8", None):
                raise RuntimeError("the checkpoint holds 8-bit Adam state: call enable_adam8() first")
            for r, saved in ckpt["adam8"].items():
                for pair, t in zip(self.adam8[r], saved):
                    pair[cur].copy_(t.to(self.device))
        if getattr(self, "qwz", None):
            # the int8 copy is a function of the fp16 slice: rebuild it from
            # the loaded slice so no reader sees the old weights' codes
            torch.cuda.synchronize(self.device)
            for r in ckpt["shards"]:
                codes, scales = self.qwz[r]
                binding.zero_qwz_quantize(self.state[r][3], self.n_valid[r], codes, scales, stream=self.stream)
        torch.cuda.synchronize(self.device)

    # ------------------------------------------------------------ accounting --
    def bytes_per_step(self) -> int:
        """Algorithmic HBM bytes of one step: (26 + 2 N_d) per stepped element."""
        return sum((26 + 2 * self.w.n_d) * self.n_valid[r] for r in self.shard_ids)

    def adam8_bytes_per_step(self) -> int:
        """Algorithmic HBM bytes of one 8-bit Adam step: 2 N_d + 14 per stepped
        element and 16 per 2048-element block (the scales read and written)."""
        blk = binding.ZS_ADAM8_BLOCK
        return sum((2 * self.w.n_d + 14) * self.n_valid[r] + 16 * ((self.n_valid[r] + blk - 1) // blk)
                   for r in self.shard_ids)

    def elements_per_step(self) -> int:
        return sum(self.n_valid[r] for r in self.shard_ids)
