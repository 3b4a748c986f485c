// step_end.cuh -- how a fused step kernel orders itself against the kernels
// around it and ends the step on the device.  Included inside an anonymous
// namespace by the step translation units (shard_step.cu, sgd.cu, adam8.cu),
// after zs_internal.h.
//
// "ZeRO Stage 1 Math", "The per-step mechanics": a step that overflowed is
// dropped (the loss scale halves and t does not advance); one that did not is
// committed (the state set flips and t advances).  The decision needs every
// block's overflow test, so the block that finishes last takes it.
#pragma once

// Programmatic dependent launch (sm_90 and later).  A kernel launched with the
// programmatic stream-serialization attribute may be scheduled while the
// kernel before it in the stream is still running; griddep_wait() returns once
// that kernel has completed and its writes are visible (at once when the
// launch carried no such dependency), so every kernel that can be launched
// this way calls it before touching global memory.
// griddep_launch_dependents() lets the next such kernel of the stream be
// scheduled before this one ends.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// The end of a step in the control block, called by thread 0 of each of the
// `total` blocks that take part, after that block's overflow atomic: the last
// block to arrive commits (flip the state set, t += 1, beta^t updated) or, if
// the step overflowed, skips (L <- max(L / 2, 1), skipped += 1); it records
// the flag in last_overflow and clears the flag and the arrival count for the
// next step.  Nothing waits: the other blocks just leave.
__device__ void arrive_and_finish(zs_ctrl* ctrl, uint32_t total, double beta1, double beta2) {
    __threadfence();
    const unsigned prev = atomicAdd(&ctrl->arrivals, 1u);
    if (prev != total - 1) return;
    __threadfence();  // every block's flag update is visible past this point
    volatile zs_ctrl* c = ctrl;
    const int ovf = c->overflow;
    c->last_overflow = ovf;
    if (ovf) {
        const double half = __dmul_rn(c->loss_scale, 0.5);
        c->loss_scale = half < 1.0 ? 1.0 : half;
        c->skipped = c->skipped + 1;
    } else {
        c->cur = c->cur ^ 1;
        c->step = c->step + 1;
        c->beta1_pow = __dmul_rn(c->beta1_pow, beta1);
        c->beta2_pow = __dmul_rn(c->beta2_pow, beta2);
    }
    c->overflow = 0;
    c->arrivals = 0u;
    __threadfence();
}

// Enqueues kernel<<<blocks, threads, smem, stream>>>(args), with the
// programmatic-serialization attribute when pdl (the kernel then waits for
// its predecessor with griddep_wait before touching global memory).
template <typename Args>
int32_t launch_ex(void (*kernel)(Args), int blocks, int threads, size_t smem, bool pdl, cudaStream_t stream,
                  const Args& args, const char* name) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, args);
    if (err != cudaSuccess) return zs::cuda_fail(err, name);
    return zs::check_launch(name);
}
