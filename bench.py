"""Benchmark of the ZeRO shard Adam step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload xl] [--impl gb300|reference]

One step = one pass of the whole hot path over one batch of synthetic inputs
already resident in HBM: the fused reduce + overflow test + Adam + fp16 cast
kernel over the rank's shard, whose last block commits the step on the device,
and the restore check that rewrites the fp16 slice only after an overflow.
The partition / indexing kernel runs once per job before the steps and is
timed on its own.  After the main workload the other target configurations
(7.5B / N_d = 64 and GPT-2-small by default) are timed the same way and
reported under "configs".  Prints ONE JSON line on rank 0.

N > 1 (launched by torch.distributed.run): every GPU runs an independent
replica on its own shard (weak scaling, no collective on the data path); the
timed region is bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Gparams/s and achieved HBM GB/s (% of GB300 peak) of the ZeRO shard Adam step"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20
ROOFLINE_DURATION = ("the timed region's time per step (the step's launches back to back, gaps included); "
                     "kernel_ms_*: an event pair around each step in a second pass of as many steps")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="xl", help="tiny | gpt2s | ragged | xl | 7b5")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--rank", type=int, default=None,
                    help="simulated rank whose shard is stepped (default: the workload's; the ragged "
                         "workload steps all shards unless a rank is given)")
    ap.add_argument("--shard-params", type=int, default=0,
                    help="shrink the workload to this many params per shard (profiling runs)")
    ap.add_argument("--prewarm-s", type=float, default=3.0,
                    help="seconds of untimed steps before the warm-up steps (HBM power ramp)")
    ap.add_argument("--clip", type=float, default=0.0,
                    help="global gradient-norm clipping at this max norm (two-pass step); 0 = off")
    ap.add_argument("--clip-keep-g", action="store_true",
                    help="with --clip: pass 1 keeps the fp32 reduced gradient for pass 2")
    ap.add_argument("--optimizer", default="adam", choices=["adam", "sgd", "adam8"],
                    help="adam (the pages' mixed-precision Adam), sgd (SGD with momentum 0.9) or adam8 "
                         "(8-bit Adam: m, v as 8-bit codes with a scale per 2048 elements)")
    ap.add_argument("--qwz", action="store_true",
                    help="keep the int8 qwZ copy of the fp16 shard in each step (1 + 4/256 bytes per element)")
    ap.add_argument("--api", default="async", choices=["async", "sync", "noalloc"],
                    help="entry point of the fp32 Adam step: zero_shard_step_async (device commit, no host "
                         "sync), zero_shard_step (flag buffer, host sync and commit per step) or "
                         "zero_shard_step_noalloc (as zero_shard_step, flag words inside the library)")
    ap.add_argument("--math", default="fast", choices=["fast", "ieee"],
                    help="rounding of the Adam update's last division: fast (ZS_MATH_FAST, corrected hardware "
                         "reciprocal, within 1 ulp) or ieee (every operation IEEE, bit-exact)")
    ap.add_argument("--log-steps", default="",
                    help="write one JSON record per timed step (kernel ms, rank, workload) to this file")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-mode", default="mapped", choices=["mapped", "staged"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-offload", action="store_true",
                    help="skip the ZeRO-Offload step (device -> host -> device) measurement")
    ap.add_argument("--offload-params", type=int, default=96_000_000,
                    help="parameters of the rank's shard the ZeRO-Offload measurement steps")
    ap.add_argument("--extra-configs", default="7b5,gpt2s,ragged",
                    help="other workloads timed in the same run after the main one (fp32 Adam step only), "
                         "reported under 'configs'; '' for none")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers --

def workload(args):
    from zero_partitioned_mixed_partition_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.shard_params:
        w = dataclasses.replace(w, name=f"{w.name}-small", numels=(args.shard_params * w.n_d,), align=128)
    if args.rank is not None:
        if not 0 <= args.rank < w.n_d:
            raise SystemExit(f"--rank must be in [0, {w.n_d})")
        w = dataclasses.replace(w, rank=args.rank)
    return w


def step_api_name(args) -> str:
    """The C-ABI entry point one timed step calls."""
    opt = getattr(args, "optimizer", "adam")
    if opt != "adam":
        return f"zero_shard_step_{opt}_async"
    if getattr(args, "clip", 0.0) > 0:
        return "zero_shard_step_clipped_async"
    return {"async": "zero_shard_step_async", "sync": "zero_shard_step",
            "noalloc": "zero_shard_step_noalloc"}[getattr(args, "api", "async")]


def arm_config(args, w, elems: int, bytes_step: int, world: int) -> dict:
    """The workload description both arms print (the reference arm times a
    bounded sample of this same workload and says so in its cpu_baseline)."""
    return {"workload": workload_label(w, elems, getattr(args, "optimizer", "adam")), "n_d": w.n_d, "shard_params": elems,
            "bytes_per_param": round(bytes_step / max(elems, 1), 4), "bytes_per_step": bytes_step,
            "storage": {"sgd": "fp16 grads and params, fp32 master/momentum (ping-pong)",
                        "adam8": "fp16 grads and params, fp32 master, 8-bit m/v codes + fp32 scale per 2048 "
                                 "(ping-pong)"}.get(getattr(args, "optimizer", "adam"),
                                                   "fp16 grads and params, fp32 master/m/v (ping-pong)"),
            "api": step_api_name(args),
            "math": ("ZS_MATH_FAST: u by corrected hardware reciprocal (within 1 ulp), all else IEEE; "
                     "m/v bit-exact" if args.math == "fast" else "ZS_MATH_IEEE: every fp32 operation IEEE, "
                     "bit-exact"),
            "l2": f"inputs larger than L2 ({bytes_step / 1e9:.2f} GB per step vs 129 MB); no flush"
            if bytes_step > L2_BYTES else "inputs fit in L2: not an HBM number",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def shard_elements(w) -> int:
    """Parameters one step updates (the rank's shard, or every shard), from
    the oracle's partition (host arithmetic, as the library's)."""
    import oracle
    oracle.build()
    lay = oracle.layout(list(w.numels), w.n_d, w.align)
    s = int(lay["shard_numel"])
    psi = int(lay["psi"])
    valid = [max(0, min(s, psi - r * s)) for r in range(w.n_d)]
    return valid[w.rank] if w.rank is not None else sum(valid)


def workload_label(w, n_valid, optimizer: str = "adam"):
    state = {"sgd": "fp32 master/momentum", "adam8": "fp32 master + 8-bit m/v"}.get(optimizer, "fp32 master/m/v")
    return (f"{w.name}: Psi={w.psi:,} ({len(w.numels)} tensors), N_d={w.n_d}, "
            f"rank {w.rank} shard of {n_valid:,} params, fp16 grads x{w.n_d} + {state}")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Per step kind: the committed DRAM-traffic record of its dominant kernel and
# the sources that kernel is compiled from (the record holds their digest).
TRAFFIC_RECORDS = {
    "adam": ("shard_step_kernel_traffic.txt", ("shard_step.cu", "step_common.cuh", "step_end.cuh")),
    "adam8": ("adam8_step_kernel_traffic.txt", ("adam8.cu", "adam8_math.cuh", "step_common.cuh", "step_end.cuh")),
}


def kernel_source_digest(kind: str = "adam") -> str:
    """sha256 prefix over the sources the step kind's kernel is compiled from."""
    h = hashlib.sha256()
    for f in TRAFFIC_RECORDS[kind][1]:
        h.update(open(os.path.join(ROOT, "zero_partitioned_mixed_partition_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kind: str = "adam"):
    """DRAM bytes per stepped parameter from the committed ncu summary, valid
    only while the kernel sources are unchanged (else None)."""
    path = os.path.join(ROOT, "profiles", TRAFFIC_RECORDS[kind][0])
    try:
        digest = kernel_source_digest(kind)
        vals = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        if vals.get("kernel_source_sha256_16") != digest:
            return None
        return {int(k.split("_")[-1]): float(v.split()[0]) for k, v in vals.items() if k.startswith("bytes_per_param_nd_")}
    except Exception:
        return None


def recorded_instructions(kind: str):
    """Thread instructions per stepped parameter from the same record (keyed
    by N_d), valid only while the kernel sources are unchanged (else None)."""
    path = os.path.join(ROOT, "profiles", TRAFFIC_RECORDS[kind][0])
    try:
        vals = dict(line.split(":", 1) for line in open(path) if ":" in line and not line.startswith("#"))
        vals = {k.strip(): v.strip() for k, v in vals.items()}
        if vals.get("kernel_source_sha256_16") != kernel_source_digest(kind):
            return None
        return {int(k.split("_")[-1]): float(v) for k, v in vals.items()
                if k.startswith("thread_instructions_per_param_nd_")}
    except Exception:
        return None


# Peak instruction issue of the GPU: 152 SMs x 4 schedulers x 32 lanes at the
# 2070 MHz maximum SM clock (the clock the timed runs hold), thread
# instructions per second.
ISSUE_PEAK_TINSTR_S = 152 * 4 * 32 * 2.07e9


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for nm, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(nm)
        if sm:
            out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                   "samples": len(sm)}
        return out


# --------------------------------------------------------------- cpu side ---

class OracleSample:
    """The oracle, as it stands, on a bounded sample of the workload: n_sample
    params of the rank's shard with their contributions, generated once, split
    into contiguous chunks over ``threads`` host threads (ctypes releases the
    GIL; 8-bit Adam chunks start on its 2048-element blocks).  ``optimizer``
    picks the oracle's update: adam, sgd (momentum 0.9) or adam8."""

    def __init__(self, w, n_sample: int, threads: int, optimizer: str = "adam"):
        import numpy as np
        import oracle
        from zero_partitioned_mixed_partition_gb300 import synth

        oracle.build()
        self.oracle, self.w, self.n, self.threads, self.optimizer = oracle, w, n_sample, threads, optimizer
        self.contribs = [synth.fp16_bits(synth.grad_contribution(w, n_sample, k, 1, shard=w.rank or 0))
                         for k in range(w.n_d)]
        self.master = synth.master_init(w, n_sample, shard=w.rank or 0).numpy()
        self.m = np.zeros_like(self.master)
        self.v = np.zeros_like(self.master)
        self.params = np.zeros(n_sample, np.uint16)
        blk = self.blk = oracle.ADAM8_BLOCK
        self.mc, self.vc = np.zeros(n_sample, np.uint8), np.zeros(n_sample, np.uint8)
        self.ms = np.zeros((n_sample + blk - 1) // blk, np.float32)
        self.vs = np.zeros((n_sample + blk - 1) // blk, np.float32)
        bounds = np.linspace(0, n_sample, threads + 1).astype(np.int64)
        if optimizer == "adam8":
            bounds = np.minimum((bounds + blk - 1) // blk * blk, n_sample)
        self.bounds = [int(b) for b in bounds]
        self.steps = 0

    def _chunk(self, lo, hi, step):
        if hi <= lo:
            return
        o, w, blk = self.oracle, self.w, self.blk
        if self.optimizer == "adam":
            o.shard_step([c[lo:hi] for c in self.contribs], self.master[lo:hi], self.m[lo:hi], self.v[lo:hi],
                         self.params[lo:hi], lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps,
                         weight_decay=w.weight_decay, loss_scale=w.loss_scale, step=step)
            return
        g, bad = o.grad_reduce([c[lo:hi] for c in self.contribs], w.loss_scale)
        if bad:
            return
        if self.optimizer == "sgd":
            o.sgd_apply(g, self.master[lo:hi], self.m[lo:hi], self.params[lo:hi], lr=w.lr, momentum=0.9,
                        weight_decay=w.weight_decay)
        else:
            o.adam8_apply(g, self.master[lo:hi], self.mc[lo:hi], self.vc[lo:hi], self.ms[lo // blk:(hi + blk - 1) // blk],
                          self.vs[lo // blk:(hi + blk - 1) // blk], self.params[lo:hi], lr=w.lr, beta1=w.beta1,
                          beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay, step=step)

    def run(self, seconds: float):
        """Oracle steps over the sample, repeated until ``seconds`` have
        passed (at least one).  Returns (Gparams/s, steps, seconds)."""
        steps, t0 = 0, time.perf_counter()
        while True:
            steps += 1
            self.steps += 1
            ts = [threading.Thread(target=self._chunk, args=(self.bounds[i], self.bounds[i + 1], self.steps))
                  for i in range(self.threads)]
            for t in ts:
                t.start()
            for t in ts:
                t.join()
            el = time.perf_counter() - t0
            if el >= seconds:
                break
        return self.n * steps / el / 1e9, steps, el


def oracle_throughput(w, n_sample: int, seconds: float, threads: int, optimizer: str = "adam"):
    """The oracle on a bounded sample (OracleSample), timed for ``seconds``.
    Returns (Gparams/s, steps, seconds, threads)."""
    g, steps, el = OracleSample(w, n_sample, threads, optimizer).run(seconds)
    return g, steps, el, threads


def oracle_sample(optimizer: str, full: int) -> int:
    """Parameters the timed oracle sample holds (the 8-bit Adam oracle's
    nearest-code search is the slowest per element)."""
    return min(1_000_000 if optimizer == "adam8" else 4_000_000, full)


def step_bytes_per_param(optimizer: str, n_d: int) -> float:
    """Algorithmic HBM bytes per stepped parameter of the step kind."""
    if optimizer == "sgd":
        return 2 * n_d + 18
    if optimizer == "adam8":
        return 2 * n_d + 14 + 16 / 2048
    return 2 * n_d + 26


def native_cpu_throughput(w, n_sample: int, seconds: float, threads: int):
    """The library's own CPU step (zero_shard_step_cpu: the ZeRO-Offload
    optimizer on the host cores) on a bounded sample of the workload.
    Returns (Gparams/s, steps, seconds, threads)."""
    import torch
    from zero_partitioned_mixed_partition_gb300 import binding, synth
    grads = [synth.grad_contribution(w, n_sample, k, 1, shard=w.rank or 0) for k in range(w.n_d)]
    master = (synth.master_init(w, n_sample, shard=w.rank or 0), torch.zeros(n_sample))
    m = (torch.zeros(n_sample), torch.zeros(n_sample))
    v = (torch.zeros(n_sample), torch.zeros(n_sample))
    params = torch.zeros(n_sample, dtype=torch.float16)
    view = binding.CpuShardView(grads, master, m, v, params, n_sample)
    hp = binding.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    binding.zero_shard_step_cpu([view], w.n_d, hp, w.loss_scale, 1, 0, n_threads=threads)
    steps, t0 = 0, time.perf_counter()
    while True:
        ovf = binding.zero_shard_step_cpu([view], w.n_d, hp, w.loss_scale, steps + 2, (steps + 1) % 2,
                                          n_threads=threads)
        assert ovf == 0
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return n_sample * steps / el / 1e9, steps, el, threads


def offload_throughput(run, w, n_sample: int, steps: int, threads: int):
    """The ZeRO-Offload step with its transfers (zero_shard_step_offload) on
    the first n_sample parameters of the rank's shard: the contributions come
    from the runner's device buffers, the fp32 state lives in host memory, the
    fp16 parameters go to a device buffer; two CUDA streams for the two link
    directions.  Wall-clock of each synchronous step after one untimed step;
    the rate is taken from the median step (the host threads share the cores
    with the rest of the machine, so single steps vary).  Returns a dict for
    the JSON line."""
    import torch
    from zero_partitioned_mixed_partition_gb300 import binding, synth
    r = run.shard_ids[0]
    n = min(n_sample, run.n_valid[r])
    dev = run.device
    grads_dev = [g[:n] for g in run.grads[r]]
    grads_host = [torch.empty(n, dtype=torch.float16).pin_memory() for _ in range(w.n_d)]
    params_host = torch.empty(n, dtype=torch.float16).pin_memory()
    params_dev = torch.empty(n, dtype=torch.float16, device=dev)
    master = (synth.master_init(w, n, shard=r), torch.zeros(n))
    m = (torch.zeros(n), torch.zeros(n))
    v = (torch.zeros(n), torch.zeros(n))
    view = binding.OffloadShardView(grads_dev, params_dev, grads_host, params_host, master, m, v, n)
    hp = binding.adam(w.lr, w.beta1, w.beta2, w.eps, w.weight_decay)
    d2h, h2d = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    cur, times = 0, []
    for k in range(steps + 1):
        t0 = time.perf_counter()
        ovf = binding.zero_shard_step_offload(view, w.n_d, hp, w.loss_scale, k + 1, cur, n_threads=threads,
                                              d2h_stream=d2h, h2d_stream=h2d)
        if k > 0:
            times.append((time.perf_counter() - t0) * 1e3)
        assert ovf == 0
        cur ^= 1
    ms = statistics.median(times)
    d2h_b, h2d_b = 2 * w.n_d * n, 2 * n
    return {"value": round(n / (ms / 1e3) / 1e9, 4), "unit": "Gparams/s", "ms_per_step": round(ms, 3),
            "ms_min_max": [round(min(times), 3), round(max(times), 3)],
            "shard_params": n, "cores": threads, "steps": steps,
            "link_bytes_per_step": {"d2h": d2h_b, "h2d": h2d_b},
            "link_gbs": {"d2h": round(d2h_b / (ms / 1e3) / 1e9, 1), "h2d": round(h2d_b / (ms / 1e3) / 1e9, 1)},
            "pages_link_bytes_per_step": 4 * n,
            "path": "zero_shard_step_offload: N_d fp16 contributions device -> pinned host, the step on the host "
                    "cores (fp32 state in host memory), fp16 params pinned host -> device; chunked, both link "
                    "directions and the host arithmetic overlapped",
            "note": "the pages' 4 Psi per step is fp16 grads down + fp16 params up for one rank's model "
                    "(N_d = 1); with N_d simulated ranks the N_d contributions cross instead of the reduced "
                    "gradient: 2 N_d + 2 bytes per parameter"}


def host_copy_gbs(threads: int, nbytes: int = 1 << 30) -> float:
    """Host memory bandwidth ceiling: PyTorch's parallel CPU copy of a 1 GiB
    fp32 tensor on `threads` threads, read + write bytes, best of 5."""
    import torch
    prev = torch.get_num_threads()
    torch.set_num_threads(threads)
    try:
        a = torch.ones(nbytes // 4, dtype=torch.float32)
        b = torch.empty_like(a)
        b.copy_(a)
        best = None
        for _ in range(5):
            t0 = time.perf_counter()
            b.copy_(a)
            el = time.perf_counter() - t0
            best = el if best is None else min(best, el)
        return 2 * nbytes / best / 1e9
    finally:
        torch.set_num_threads(prev)


def reference_arm(args, rank: int):
    """The oracle timed on the host cores as the reference arm."""
    if rank != 0:
        return
    w = workload(args)
    elems = shard_elements(w)
    threads = os.cpu_count() or 1
    n_sample = oracle_sample(args.optimizer, max(w.psi // w.n_d, 1))
    # inputs generated once; each step at least one pass over the sample, the
    # whole run about a minute (and never past three)
    sample_run = OracleSample(w, n_sample, threads, args.optimizer)
    per_step_s = max(0.0, min(5.0, 60.0 / max(args.steps + args.warmup, 1)))
    for _ in range(args.warmup):
        sample_run.run(0.0)
    vals = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        g, _, _ = sample_run.run(per_step_s)
        vals.append(g)
        if time.perf_counter() - t_all > 180:
            break
    value = statistics.median(vals)
    sample = (f"{n_sample:,} params of the rank's shard x N_d={w.n_d} contributions, {args.optimizer} oracle, "
              f"{threads} threads over contiguous chunks, >= {per_step_s:.3f} s per step (at least one pass)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "Gparams/s",
            "n_gpus": args.gpus, "steps": len(vals), "warmup": args.warmup,
            "ms_per_step": round(n_sample / (value * 1e9) * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": arm_config(args, w, elems, round(step_bytes_per_param(args.optimizer, w.n_d) * elems), args.gpus),
            "cpu_baseline": {"value": round(value, 4), "unit": "Gparams/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "Gparams/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- gpu side ---

def time_steps(args, run, w, stream, world, steps, warmup, prewarm_s, local):
    """Pre-warm, warm up and time ``steps`` steps of ``run`` on ``stream``.

    One step is the whole hot path over the stepped shards: the fused
    reduce + overflow test + Adam + fp16 cast launches and the end of the step
    (for the fp32 Adam, SGD, 8-bit Adam and clipped steps, the last fused
    launch commits and a restore kernel follows that leaves at once unless the
    step overflowed; a step with a qwZ copy ends with the commit kernel).  The
    per-launch pass of the clipped step calls its two passes one by one, with
    an event between them and the commit kernel after them.  Returns a dict of
    the measurements."""
    import torch
    import torch.distributed as dist
    from zero_partitioned_mixed_partition_gb300 import binding
    from zero_partitioned_mixed_partition_gb300 import dist as zdist

    clip = args.clip > 0
    sgd_hp = binding.sgd(w.lr, 0.9, w.weight_decay)
    api = getattr(args, "api", "async")
    # the synchronous entry points take the loss scale, t and the state set
    # from the caller, who commits or skips after each step (kept here)
    host = run.ctrl_host()
    hstate = {"ls": host["loss_scale"], "t": host["step"] + 1, "cur": host["cur"], "applied": 0}
    flag_dev = torch.zeros(1, dtype=torch.int32, device=run.device) if api == "sync" else None

    def sync_step():
        if api == "sync":
            ovf = binding.zero_shard_step(run.views, w.n_d, run.hp, hstate["ls"], hstate["t"], hstate["cur"],
                                          flag_dev, stream=stream)
        else:
            ovf = binding.zero_shard_step_noalloc(run.views, w.n_d, run.hp, hstate["ls"], hstate["t"],
                                                  hstate["cur"], stream=stream)
        if ovf:
            hstate["ls"] = max(hstate["ls"] / 2, 1.0)
        else:
            hstate["cur"] ^= 1
            hstate["t"] += 1
            hstate["applied"] += 1

    def one_step(ev=None):
        if clip and ev is None:
            # the clipped step's one call: sqnorm cleared, pass 1, pass 2
            # (its last launch ends the step), then the restore check
            run.step_clipped(args.clip)
            return
        if clip:
            # per-pass times: the same passes called one by one, an event
            # between them, and the commit kernel after them
            with torch.cuda.stream(stream):
                run.sqnorm.zero_()
        if ev is not None:
            ev[0].record(stream)
        if args.optimizer == "sgd":
            run.step_sgd(sgd_hp)      # fused kernel(s) ending the step, then the restore check
        elif args.optimizer == "adam8":
            run.step_adam8()          # fused kernel(s) ending the step, then the restore check
        elif not clip and api != "async":
            sync_step()               # fused kernel(s), host sync, commit kept on the host
        elif not clip:
            run.step()                # fused kernel(s) ending the step, then the restore check
        else:
            binding.zero_shard_grad_sqnorm_all_async(run.views, w.n_d, run.sqnorm, run.ctrl,
                                                     g_dev=run.gbuf if run.gbuf else None, stream=stream)
            if ev is not None:
                ev[2].record(stream)
            binding.zero_shard_clipped_adam_all_async(run.views, w.n_d, run.hp, args.clip, run.sqnorm, run.ctrl,
                                                      g_dev=run.gbuf if run.gbuf else None, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        if clip:
            run.commit()

    # untimed pre-warm: the first seconds of sustained HBM traffic after idle
    # run a few percent slower; the timed region should see the steady state
    t0 = time.perf_counter()
    prewarm_steps = 0
    while time.perf_counter() - t0 < prewarm_s:
        for _ in range(10):
            one_step()
        prewarm_steps += 10
        torch.cuda.synchronize()
    for _ in range(warmup):
        one_step()
    torch.cuda.synchronize()

    pairs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = binding.zero_kernel_launches()
    # the timed region: the steps back to back, nothing else on the stream
    t_start.record(stream)
    for _ in range(steps):
        one_step()
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = binding.zero_kernel_launches() - launches0
    if world > 1:
        dist.barrier()
    # then as many steps again with an event pair around each (and around each
    # pass of the clipped step): the per-launch durations.  Events between the
    # launches keep the next step from being scheduled while the current one
    # drains, so this pass is not the timed region.
    for k in range(steps):
        one_step(pairs[k])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms_total = t_start.elapsed_time(t_end)
    out = {"ms_total": ms_total, "kern_ms": [ev[0].elapsed_time(ev[1]) for ev in pairs],
           "launches": launches, "clocks": clocks, "prewarm_steps": prewarm_steps}
    if clip:
        out["norm_ms"] = [ev[0].elapsed_time(ev[2]) for ev in pairs]
        out["upd_ms"] = [ev[2].elapsed_time(ev[1]) for ev in pairs]
    ctrl = run.ctrl_host()
    if api == "async" or clip or args.optimizer != "adam":
        assert ctrl["skipped"] == 0 and ctrl["step"] == prewarm_steps + warmup + 2 * steps, ctrl
    else:
        assert hstate["applied"] == prewarm_steps + warmup + 2 * steps, hstate
    out["ctrl"] = ctrl
    out["ms_max"] = zdist.max_over_ranks(ms_total, device=torch.device("cuda", local))
    return out


def time_partition(w, dev, stream, repeats: int = 5):
    """The partition / indexing kernel (zero_partition_layout_device), which
    runs once per job: its outputs checked against the library's host layout
    and its launch timed with CUDA events (best of a few, after one untimed
    run).  Returns (kernel microseconds, fragments)."""
    import torch
    from zero_partitioned_mixed_partition_gb300 import binding
    with torch.cuda.stream(stream):
        numels_dev = torch.tensor(list(w.numels), dtype=torch.int64, device=dev)
        scalars = torch.zeros(5, dtype=torch.int64, device=dev)
        toff = torch.zeros(len(w.numels), dtype=torch.int64, device=dev)
        soff = torch.zeros(w.n_d + 1, dtype=torch.int64, device=dev)
        cap = len(w.numels) + w.n_d
        frags = torch.zeros(cap * 4, dtype=torch.int64, device=dev)
    best = None
    for i in range(repeats + 1):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.zero_partition_layout_device(numels_dev, w.n_d, w.align, scalars, toff, soff, frags, cap,
                                             stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        if i > 0:
            us = a.elapsed_time(b) * 1e3
            best = us if best is None else min(best, us)
    host = binding.zero_partition_layout(w.numels, w.n_d, w.align)
    got = scalars.cpu().tolist()
    assert got[4] == 0 and got[2] == int(host["shard_numel"]), (got, host["shard_numel"])
    return best, int(got[3])


def workload_summary(args, w, run, res, peak, peak_kind):
    """Rate, bandwidth and roofline of one timed workload."""
    elems = run.elements_per_step()
    world = res.get("world", 1)
    steps = len(res["kern_ms"])
    bytes_step = run.bytes_per_step()
    value = elems * world * steps / (res["ms_max"] / 1e3) / 1e9
    hbm_gbs = bytes_step * world * steps / (res["ms_max"] / 1e3) / 1e9
    # roofline over the timed region: its time per step, every microsecond of
    # it charged to the step's launches
    step_ms = res["ms_max"] / steps
    achieved = bytes_step / (step_ms / 1e3) / 1e9
    mean_kern_ms = statistics.mean(res["kern_ms"])
    traffic = None
    per = recorded_traffic("adam")
    if per and w.n_d in per:
        traffic = round(per[w.n_d] * elems)
    return {"workload": workload_label(w, elems), "n_d": w.n_d, "shard_params": elems,
            "value": round(value, 3), "unit": "Gparams/s", "steps": steps,
            "ms_per_step": round(res["ms_max"] / steps, 5), "bytes_per_step": bytes_step,
            "hbm_gbs": round(hbm_gbs, 1), "pct_of_nominal_8tbs": round(100 * hbm_gbs / NOMINAL_HBM_GBS, 2),
            f"pct_of_{peak_kind}_peak": round(100 * hbm_gbs / peak, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "kernel": ("group_step_kernel" if len(run.views) > 1 else "shard_step_kernel")
                         + " + restore_kernel", "peak_kind": peak_kind,
                         "duration": ROOFLINE_DURATION, "step_ms": round(step_ms, 5),
                         "kernel_ms_mean": round(mean_kern_ms, 5),
                         "kernel_ms_median": round(statistics.median(res["kern_ms"]), 5),
                         "kernel_ms_min": round(min(res["kern_ms"]), 5),
                         "frac_per_launch_events": round(bytes_step / (mean_kern_ms / 1e3) / 1e9 / peak, 4)},
            "clocks": res["clocks"], "gpu_launches": int(res["launches"]),
            "l2": f"inputs larger than L2 ({bytes_step / 1e9:.2f} GB per step vs 129 MB); no flush"
            if bytes_step > L2_BYTES else "inputs fit in L2: not an HBM number"}


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        reference_arm(args, rank)
        return

    import torch
    import torch.distributed as dist

    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from zero_partitioned_mixed_partition_gb300 import binding, build, synth
    from zero_partitioned_mixed_partition_gb300 import dist as zdist
    from zero_partitioned_mixed_partition_gb300.runner import WorkloadRunner

    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    binding.lib()

    def make_runner(w, stream):
        if w.rank is not None and world > 1:
            w = dataclasses.replace(w, rank=zdist.replica_shard(w.rank, rank, w.n_d))
        with torch.cuda.stream(stream):
            run = WorkloadRunner(w, dev, stream=stream,
                                 math=binding.ZS_MATH_FAST if args.math == "fast" else binding.ZS_MATH_IEEE)
        torch.cuda.synchronize()
        return w, run

    w = workload(args)
    stream = torch.cuda.Stream(device=dev)
    w, run = make_runner(w, stream)
    # the partition runs once per job, before the steps: timed on its own
    part_us, part_frags = time_partition(w, dev, stream)

    clip = args.clip > 0
    if args.optimizer != "adam" and (clip or args.qwz):
        raise SystemExit(f"--optimizer {args.optimizer} goes without --clip / --qwz")
    if args.api != "async" and (args.optimizer != "adam" or clip):
        raise SystemExit("--api sync|noalloc times the fp32 Adam step without --clip")
    if args.optimizer == "adam8":
        run.enable_adam8()
    if clip:
        run.enable_clipping(args.clip_keep_g)
    if args.qwz:
        run.enable_qwz()

    res = time_steps(args, run, w, stream, world, args.steps, args.warmup, args.prewarm_s, local)
    ms_max, kern_ms, ctrl = res["ms_max"], res["kern_ms"], res["ctrl"]
    prewarm_steps = res["prewarm_steps"]
    elems = run.elements_per_step()
    total_elems = elems * world
    value = total_elems * args.steps / (ms_max / 1e3) / 1e9
    bytes_step = run.clipped_bytes_per_step() if clip else run.bytes_per_step()
    if args.optimizer == "sgd":  # fp32 master + momentum: 2 N_d + 18 bytes per element
        bytes_step = sum((2 * w.n_d + 18) * run.n_valid[r] for r in run.shard_ids)
    if args.optimizer == "adam8":  # fp32 master + 8-bit m, v: 2 N_d + 14 bytes per element + the scales
        bytes_step = run.adam8_bytes_per_step()
    if args.qwz:  # int8 codes + one fp32 scale per 256 elements, written by the step
        bytes_step += sum(run.n_valid[r] + 4 * ((run.n_valid[r] + 255) // 256) for r in run.shard_ids)
    hbm_gbs = bytes_step * world * args.steps / (ms_max / 1e3) / 1e9
    if args.log_steps:
        # one record per step of the per-launch pass that follows the timed
        # region; no step overflowed (checked above), so t advances by one per
        # step and L is constant
        peak_gbs, _ = measured_peaks()
        t_first = prewarm_steps + args.warmup + args.steps + 1
        path = args.log_steps if world == 1 else f"{args.log_steps}.rank{rank}"
        with open(path, "w") as f:
            for k, ms in enumerate(kern_ms):
                gbs = bytes_step / (ms / 1e3) / 1e9
                f.write(json.dumps({"workload": w.name, "n_d": w.n_d, "process_rank": rank,
                                    "shard": w.rank if w.rank is not None else "all", "t": t_first + k,
                                    "overflow": 0, "loss_scale": ctrl["loss_scale"], "kernel_ms": round(ms, 5),
                                    "gparams_s": round(elems / (ms / 1e3) / 1e9, 3), "kernel_gbs": round(gbs, 1),
                                    "pct_of_peak": round(100 * gbs / peak_gbs, 2)}) + "\n")
    peak, peak_kind = measured_peaks()

    # roofline of the step: algorithmic bytes per step / the timed region's
    # time per step (back-to-back launches; the gaps between them count too)
    step_ms = ms_max / args.steps
    achieved = bytes_step / (step_ms / 1e3) / 1e9
    mean_kern_ms = statistics.mean(kern_ms)
    traffic = None
    if args.optimizer in TRAFFIC_RECORDS and not clip and not args.qwz:
        traffic_per_param = recorded_traffic(args.optimizer)
        if traffic_per_param and w.n_d in traffic_per_param:
            traffic = round(traffic_per_param[w.n_d] * elems)
    clip_info = None
    if clip:
        # per pass: algorithmic bytes / mean launch time (pass 1 reads the
        # contributions, writes g if kept; pass 2 reads g or re-reduces)
        b1 = (2 * w.n_d + (4 if run.gbuf else 0)) * elems
        b2 = ((4 if run.gbuf else 2 * w.n_d) + 26) * elems
        norm_ms, upd_ms = res["norm_ms"], res["upd_ms"]
        clip_info = {"max_norm": args.clip, "keep_g": bool(run.gbuf),
                     "bytes_per_param": (2 * w.n_d + 34) if run.gbuf else (4 * w.n_d + 26),
                     "norm_pass": {"ms_mean": round(statistics.mean(norm_ms), 5),
                                   "gbs": round(b1 / (statistics.mean(norm_ms) / 1e3) / 1e9, 1)},
                     "update_pass": {"ms_mean": round(statistics.mean(upd_ms), 5),
                                     "gbs": round(b2 / (statistics.mean(upd_ms) / 1e3) / 1e9, 1)},
                     "sqnorm_last": float(run.sqnorm.item())}

    # end to end through the C ABI with host buffers: pinned H2D of the step's
    # gradient contributions, the step, D2H of the fp16 shard and the control block
    e2e = None
    if not args.no_e2e and args.optimizer == "adam" and not clip and not args.qwz:
        e2e = end_to_end(args, run, stream, dev, world)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "Gparams/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "prewarm_steps": prewarm_steps,
        "ms_per_step": round(ms_max / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": arm_config(args, w, elems, bytes_step, world),
        "hbm_gbs": round(hbm_gbs, 1),
        "pct_of_nominal_8tbs": round(100 * hbm_gbs / NOMINAL_HBM_GBS, 2),
        f"pct_of_{peak_kind}_peak": round(100 * hbm_gbs / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": ("group_step_kernel" if len(run.views) > 1 else "shard_step_kernel")
                     + (" + restore_kernel" if not args.qwz else " + commit_kernel"),
                     "peak_kind": peak_kind,
                     "duration": ROOFLINE_DURATION, "step_ms": round(step_ms, 5),
                     "kernel_ms_mean": round(mean_kern_ms, 5), "kernel_ms_median": round(statistics.median(kern_ms), 5),
                     "kernel_ms_min": round(min(kern_ms), 5),
                     "frac_per_launch_events": round(bytes_step / (mean_kern_ms / 1e3) / 1e9 / peak, 4)},
        "clocks": res["clocks"],
        "gpu_launches": int(res["launches"]),
        "partition": {"kernel_us": round(part_us, 2), "fragments": part_frags,
                      "when": "once per job, before the timed steps (zero_partition_layout_device)"},
        "e2e": e2e,
    }
    if args.optimizer == "sgd":
        line["optimizer"] = {"kind": "sgd", "momentum": 0.9,
                             "timed": "fused kernel(s), the last ending the step, + restore check"}
        line["roofline"]["kernel"] = ("sgd_group_kernel" if len(run.views) > 1 else "sgd_step_kernel") + " + restore_kernel"
    if args.optimizer == "adam8":
        instr = recorded_instructions("adam8")
        if instr and w.n_d in instr:
            # the N_d <= 4 kernel is bound by instruction issue, not HBM: its
            # issue roofline, from the ncu-counted instructions per parameter
            rate = instr[w.n_d] * elems / (step_ms / 1e3)
            line["roofline_issue"] = {"bound": "alu", "achieved": round(rate / 1e12, 3),
                                      "peak": round(ISSUE_PEAK_TINSTR_S / 1e12, 3), "unit": "T thread-instr/s",
                                      "frac": round(rate / ISSUE_PEAK_TINSTR_S, 4),
                                      "instructions_per_param": instr[w.n_d], "source": "ncu, recorded"}
        line["optimizer"] = {"kind": "adam8", "block": binding.ZS_ADAM8_BLOCK,
                             "state": "fp32 master, uint8 codes of m and v, fp32 scale per block (ping-pong)",
                             "timed": "fused kernel(s), the last ending the step, + restore check"}
        line["roofline"]["kernel"] = "adam8_step_kernel + restore_kernel"
    if args.qwz:
        line["qwz"] = {"block": 256, "extra_bytes_per_param": round(1 + 4 / 256, 4)}
    if clip_info is not None:
        line["clip"] = clip_info
        line["roofline"]["kernel"] = "grad_norm_kernel + clipped_step_kernel + restore_kernel"
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        opt = args.optimizer
        ns = oracle_sample(opt, elems)
        g, steps, el, th = oracle_throughput(w, ns, args.cpu_seconds, os.cpu_count() or 1, opt)
        line["cpu_baseline"] = {"value": round(g, 4), "unit": "Gparams/s", "cores": th, "kind": "oracle",
                                "sample": f"{ns:,} params of the shard x N_d={w.n_d}, {opt} oracle, "
                                          f"{steps} steps in {el:.1f} s over {th} threads"}
        ns1 = min(ns // 4, elems)
        g1, steps1, el1, _ = oracle_throughput(w, ns1, 3.0, 1, opt)
        line["cpu_baseline"]["single_thread"] = {
            "value": round(g1, 4), "unit": "Gparams/s", "cores": 1,
            "sample": f"{ns1:,} params x N_d={w.n_d}, {opt} oracle, {steps1} steps in {el1:.1f} s on one thread"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.optimizer == "adam" and not clip:
        ns = min(32_000_000, elems)
        g, steps, el, th = native_cpu_throughput(w, ns, 3.0, os.cpu_count() or 1)
        ceiling = host_copy_gbs(th)
        line["cpu_native"] = {"value": round(g, 4), "unit": "Gparams/s", "cores": th,
                              "kind": "zero_shard_step_cpu (ZeRO-Offload step on the host cores)",
                              "sample": f"{ns:,} params x N_d={w.n_d}, {steps} steps in {el:.1f} s",
                              "host_gbs": round(g * step_bytes_per_param("adam", w.n_d), 1),
                              "host_copy_gbs": round(ceiling, 1),
                              "frac_of_host_copy": round(g * step_bytes_per_param("adam", w.n_d) / ceiling, 3)}
        if not args.no_offload:
            line["offload"] = offload_throughput(run, w, args.offload_params, 10, th)

    # the other target configurations of the same step, each on its own
    # buffers after the previous ones are freed, timed the same way
    extras = [x for x in args.extra_configs.split(",") if x and x != args.workload]
    if extras and args.optimizer == "adam" and not clip and not args.qwz and not args.shard_params:
        del run
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["configs"] = {}
        for name in extras:
            w2, run2 = make_runner(synth.WORKLOADS[name], stream)
            res2 = time_steps(args, run2, w2, stream, world, args.steps, args.warmup,
                              min(args.prewarm_s, 2.0), local)
            res2["world"] = world
            line["configs"][name] = workload_summary(args, w2, run2, res2, peak, peak_kind)
            del run2
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def end_to_end(args, run, stream, dev, world):
    """The same step through the C ABI with the step's inputs and result in
    page-locked HOST memory.  mapped: zero_shard_step_host, whose fused kernel
    reads the N_d contributions from and writes the fp16 shard to host memory
    over NVLink-C2C, then returns the overflow flag.  staged: cudaMemcpyAsync
    of the contributions to device buffers, zero_shard_step_async, copies of
    the fp16 shard and the control block back.  Wall-clock per step, after the
    stream is idle."""
    import torch
    from zero_partitioned_mixed_partition_gb300 import binding
    from zero_partitioned_mixed_partition_gb300 import dist as zdist

    r = run.shard_ids[0]
    n = run.n_valid[r]
    host_grads = [g[:n].cpu().pin_memory() for g in run.grads[r]]
    host_params = torch.empty(n, dtype=torch.float16).pin_memory()
    master, m, v, _ = run.state[r]
    if args.e2e_mode == "mapped":
        view = binding.HostShardView(host_grads, master, m, v, host_params, n)
        h2d = sum(h.numel() * 2 for h in host_grads)
        d2h = host_params.numel() * 2 + 4

        def step():
            ovf = binding.zero_shard_step_host(view, run.w.n_d, run.hp, run.ctrl, stream=stream)
            assert ovf == 0
    else:
        host_ctrl = torch.empty(run.ctrl.numel(), dtype=torch.int64).pin_memory()
        h2d = sum(h.numel() * 2 for h in host_grads)
        d2h = host_params.numel() * 2 + host_ctrl.numel() * 8

        def step():
            with torch.cuda.stream(stream):
                for h, g in zip(host_grads, run.grads[r]):
                    g[:n].copy_(h, non_blocking=True)
                binding.zero_shard_step_async([run.views[0]], run.w.n_d, run.hp, run.ctrl, stream=stream)
                host_params.copy_(run.state[r][3][:n], non_blocking=True)
                host_ctrl.copy_(run.ctrl, non_blocking=True)
            stream.synchronize()

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        step()
    torch.cuda.synchronize()
    ms = zdist.max_over_ranks((time.perf_counter() - t0) * 1e3, device=dev)
    # the end-to-end step covers one shard (the first stepped one) per rank
    val = n * world * args.e2e_steps / (ms / 1e3) / 1e9
    path = ("zero_shard_step_host: contributions read from and fp16 shard written to pinned host memory "
            "by the fused kernel (NVLink-C2C), device commit, flag returned"
            if args.e2e_mode == "mapped" else
            "pinned host grads -> device (cudaMemcpyAsync), zero_shard_step_async, fp16 shard + control block "
            "-> pinned host")
    return {"value": round(val, 3), "unit": "Gparams/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / args.e2e_steps, 4), "mode": args.e2e_mode, "path": path,
            "shard_params": n}


if __name__ == "__main__":
    main()
