// shard_step.cu -- the fused ZeRO shard step for sm_103a and its C ABI.
//
// One rank's optimizer step over its shard ("ZeRO Stage 1 Math", "The
// per-step mechanics", beats 2-3; "DeepSpeed ZeRO Stages", sec. 2.1 Fact 1):
//   reduce   gs_j = sum_k fp32(h_k[j]) over the N_d fp16 contributions, in
//            rank order, g_j = gs_j * (float)(1 / (N_d L))      (averaged,
//            and the loss scale L removed)
//   test     any non-finite gs_j in the valid range -> overflow for the step
//   Adam     m' = b1 m + (1-b1) g,  v' = b2 v + (1-b2) g^2,
//            u = (m'/(1-b1^t)) / (sqrt(v'/(1-b2^t)) + eps),
//            th' = th - lr (u + wd th)                 (wd = 0: plain Adam)
//   cast     params_j = fp16_rn(th')
// all in one pass over memory.  The step is elementwise with O(1) work per
// parameter and touches every byte once, so it is bound by HBM bandwidth: per
// stepped element it reads 2 N_d + 12 bytes and writes 12 + 2 bytes.  The
// kernel therefore streams wide vectors (8 or 16 parameters per thread and
// iteration, see Mem<> below), runs a persistent grid sized from the SM count
// and occupancy, and keeps every fp32 operation a single IEEE
// round-to-nearest step (explicit _rn intrinsics, no fused multiply-add), so
// its results are reproducible bit for bit.
//
// Skip without a second pass: the non-finite test is only known once the whole
// step has run, so the state is double-buffered.  A step reads set `cur` and
// writes set `cur ^ 1`; committing flips `cur`, skipping leaves it and only the
// fp16 slice (already overwritten) is re-cast from the kept master weights.
#include <cuda_fp16.h>
#include <stdint.h>

#include <cuda.h>  // driver types only (CUcontext); the entry point is fetched at run time

#include <map>
#include <mutex>
#include <unordered_map>
#include <utility>

#include "zs_internal.h"

namespace {

constexpr int kThreads = 256;          // threads per block of the fused kernel
constexpr int kCommitThreads = 512;    // threads per block of the commit kernel
constexpr int kCastThreads = 256;

#include "step_common.cuh"

#include "step_end.cuh"

// ------------------------------------------------------------ fused kernel ---

// Kernel parameters (passed by value, so the contribution table needs no
// device memory).  CAP bounds n_d and sizes the pointer table.
template <int CAP>
struct StepArgs {
    const uint16_t* grads[CAP];
    float* master[2];
    float* m[2];
    float* v[2];
    uint16_t* params;
    int64_t n;
    int32_t n_d;
    int32_t cur;          // host-resolved ping-pong set (ctrl == nullptr)
    Coef coef;            // host-resolved coefficients (ctrl == nullptr)
    zs_adam hp;           // hyper-parameters for device-resolved coefficients
    const zs_ctrl* ctrl;  // non-null: loss scale, t and cur come from here
    int32_t* flag;        // overflow accumulator (ORed)
    zs_ctrl* commit;      // non-null: this launch ends the step (arrive_and_finish)
    int8_t* qcodes;       // qwZ copy (QZ kernels only)
    float* qscales;
};

// VEC elements of one shard starting at element e: reduce, test, update,
// cast.  grads / n_d: the shard's contribution table; params, n: its fp16
// slice and length.  The updated master values are left in th.  FAST selects
// ZS_MATH_FAST.
template <int CAP, int VEC, int ND, bool FAST>
__device__ __forceinline__ uint32_t step_elements(const uint16_t* const (&grads)[CAP], int32_t n_d,
                                                  uint16_t* params, int64_t n, const Coef& c, int64_t e,
                                                  const float* th_in, const float* m_in,
                                                  const float* v_in, float* th_out, float* m_out,
                                                  float* v_out, float* th) {
    float m[VEC], v[VEC], acc[VEC];
    if (!ZS_RANGE_OK(kSiteStep, e, VEC, n)) return 0u;
    Mem<VEC>::load_f(th_in + e, th);
    Mem<VEC>::load_f(m_in + e, m);
    Mem<VEC>::load_f(v_in + e, v);
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.0f;
    sum_contributions<CAP, VEC, ND>(grads, n_d, e, acc);
    uint32_t bad = 0;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        bad |= nonfinite(acc[j]) ? 1u : 0u;
        adam_update<FAST>(c, acc[j], th[j], m[j], v[j]);
    }
    Mem<VEC>::store_f(th_out + e, th);
    Mem<VEC>::store_f(m_out + e, m);
    Mem<VEC>::store_f(v_out + e, v);
    Mem<VEC>::store_h(params + e, th);
    return bad;
}

// Minimum resident blocks per SM promised to the compiler (0: none).  The
// 16-element kernels run two blocks per SM (about 100-128 registers each).  With
// the qwZ epilogue and at most 16 compiled contributions the compiler left ~100
// registers unused by default; promising two blocks lets it use the 128 they
// have: +6.8 % on the ragged workload's qwZ step, +24 % at N_d = 8 (measured).
// With 32 or 64 contributions it already uses 128, and the promise measured
// 2.8 % slower there, so it is not made.
//
// The 16-element kernel with a run-time N_d and no qwZ copy also gets the
// promise: without it, the end-of-step code after its element loop led the
// compiler to a 99-register allocation of the loop (127 before that code was
// added), 24 % slower on the N_d = 8 GPT-2-small shard (0.112 -> 0.139 ms per
// step, measured); with it the loop gets 128.
template <int VEC, int ND, bool QZ>
constexpr int step_min_blocks() { return (VEC == 16 && (QZ ? ND <= 16 : ND == 0)) ? 2 : 0; }
// The grouped kernel keeps the first rule (its registers did not move).
template <int VEC, int ND, bool QZ>
constexpr int group_min_blocks() { return (VEC == 16 && QZ && ND <= 16) ? 2 : 0; }

// The element loop of shard_step_kernel over the shard (set cur in, set
// cur ^ 1 out); returns this thread's non-finite bits.
template <int CAP, int VEC, int ND, bool QZ, bool FAST>
__device__ __forceinline__ uint32_t step_range(const StepArgs<CAP>& p, const Coef c, const int cur) {
    const float* th_in = p.master[cur];
    const float* m_in = p.m[cur];
    const float* v_in = p.v[cur];
    float* th_out = p.master[cur ^ 1];
    float* m_out = p.m[cur ^ 1];
    float* v_out = p.v[cur ^ 1];

    uint32_t bad = 0;
    const int64_t nvec = p.n / VEC;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if constexpr (!QZ) {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
            float th[VEC];
            bad |= step_elements<CAP, VEC, ND, FAST>(p.grads, p.n_d, p.params, p.n, c, i * VEC, th_in, m_in, v_in,
                                                     th_out, m_out, v_out, th);
        }
    } else {
        // qwZ: whole warps iterate together so that the G lanes holding one
        // 256-parameter block can reduce its max by shuffles; every full block
        // gets its codes and scale here, the trailing partial one in the commit
        static_assert(VEC == 8 || VEC == 16, "qwZ needs the vector layouts");
        constexpr int G = kQwzBlock / VEC;
        const int lane = threadIdx.x & 31;
        for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); i0 < nvec; i0 += stride) {
            const int64_t i = i0 + lane;
            const bool active = i < nvec;
            float th[VEC], x[VEC];
            if (active)
                bad |= step_elements<CAP, VEC, ND, FAST>(p.grads, p.n_d, p.params, p.n, c, i * VEC, th_in, m_in,
                                                         v_in, th_out, m_out, v_out, th);
#pragma unroll
            for (int j = 0; j < VEC; ++j) x[j] = active ? as_fp16_value(th[j]) : 0.0f;
            int8_t q[VEC];
            const float scale = qwz_group_codes<VEC, G>(x, active ? VEC : 0, q);
            const int64_t block = (i0 + (lane & ~(G - 1))) * VEC / kQwzBlock;
            if ((block + 1) * kQwzBlock <= p.n) {  // full block: every lane of the group is active
                if (ZS_RANGE_OK(kSiteQwzFused, i * VEC, VEC, p.n)) store_codes<VEC>(p.qcodes + i * VEC, q);
                if ((lane & (G - 1)) == 0 && ZS_RANGE_OK(kSiteScale, block, 1, (p.n + kQwzBlock - 1) / kQwzBlock))
                    p.qscales[block] = scale;
            }
        }
    }
    if (VEC > 1) {  // ragged tail: fewer than VEC elements, one per thread of block 0
        const int64_t e = nvec * VEC + threadIdx.x;
        if (blockIdx.x == 0 && e < p.n) {
            float th[1];
            bad |= step_elements<CAP, 1, ND, FAST>(p.grads, p.n_d, p.params, p.n, c, e, th_in, m_in, v_in, th_out,
                                                   m_out, v_out, th);
        }
    }
    return bad;
}

template <int CAP, int VEC, int ND, bool QZ, bool FAST>
__global__ void __launch_bounds__(kThreads, step_min_blocks<VEC, ND, QZ>())
shard_step_kernel(const __grid_constant__ StepArgs<CAP> p) {
    __shared__ Coef s_coef;
    __shared__ int s_cur;
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        if (p.ctrl != nullptr) {
            const zs_ctrl* ctrl = p.ctrl;
            const double p1 = __dmul_rn(ctrl->beta1_pow, p.hp.beta1);  // beta1^(t+1)
            const double p2 = __dmul_rn(ctrl->beta2_pow, p.hp.beta2);
            s_coef = coef_device(p.hp, p1, p2, p.n_d, ctrl->loss_scale);
            s_cur = ctrl->cur;
        } else {
            s_coef = p.coef;
            s_cur = p.cur;
        }
    }
    __syncthreads();
    const Coef c = s_coef;
    const int cur = s_cur;
    const uint32_t bad = step_range<CAP, VEC, ND, QZ, FAST>(p, c, cur);
    // overflow: warp/block OR, one atomic per block that saw a non-finite value
    // (a step with a qwZ copy ends in the commit kernel, so QZ kernels carry no
    // end-of-step code)
    const int any_bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        if (any_bad) atomicOr(p.flag, 1);
        if constexpr (!QZ) {
            if (p.commit != nullptr) arrive_and_finish(p.commit, gridDim.x, p.hp.beta1, p.hp.beta2);
        }
    }
}

// ------------------------------------------------ several shards, one launch ---

// Shards stepped by one launch of the grouped kernel.
constexpr int kGroupMax = 16;

// Parameters of the grouped kernel: up to kGroupMax shards of one step, all
// with the same access width and no qwZ copy.  vstart[s] is the first vector
// of shard s in the launch's index space (vstart[n_shards] = total vectors).
template <int CAP>
struct GroupArgs {
    const uint16_t* grads[kGroupMax][CAP];
    float* master[kGroupMax][2];
    float* m[kGroupMax][2];
    float* v[kGroupMax][2];
    uint16_t* params[kGroupMax];
    int64_t n[kGroupMax];
    int8_t* qcodes[kGroupMax];   // qwZ copies (QZ kernels only)
    float* qscales[kGroupMax];
    int64_t vstart[kGroupMax + 1];
    int32_t n_shards;
    int32_t n_d;
    int32_t cur;          // host-resolved ping-pong set (ctrl == nullptr)
    Coef coef;            // host-resolved coefficients (ctrl == nullptr)
    zs_adam hp;
    const zs_ctrl* ctrl;  // non-null: loss scale, t and cur come from here
    int32_t* flag;
    zs_ctrl* commit;      // non-null: this launch ends the step (arrive_and_finish)
};

// The fused step of several shards in one persistent launch: the grid walks
// the concatenated vector index space of the shards, so one launch's ramp and
// tail replace one per shard (measured on the ragged workload's 16 shards:
// 6.86 TB/s as 16 launches, 7.06 TB/s as one grouped launch).
// Each thread keeps a cursor on its current shard; the index only grows, so
// the cursor only moves forward.  Each shard's ragged tail (fewer than VEC
// elements) is stepped by one block.  Arithmetic and order per element are
// those of shard_step_kernel.  QZ (shards with a qwZ copy): every shard's
// vector range starts on a warp boundary (vstart rounded up to 32), so the
// lanes that hold one 256-parameter block always belong to one shard and
// reduce its scale by shuffles, as in shard_step_kernel.
template <int CAP, int VEC, int ND, bool QZ, bool FAST>
__global__ void __launch_bounds__(kThreads, group_min_blocks<VEC, ND, QZ>())
group_step_kernel(const __grid_constant__ GroupArgs<CAP> a) {
    __shared__ Coef s_coef;
    __shared__ int s_cur;
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        if (a.ctrl != nullptr) {
            const zs_ctrl* ctrl = a.ctrl;
            const double p1 = __dmul_rn(ctrl->beta1_pow, a.hp.beta1);
            const double p2 = __dmul_rn(ctrl->beta2_pow, a.hp.beta2);
            s_coef = coef_device(a.hp, p1, p2, a.n_d, ctrl->loss_scale);
            s_cur = ctrl->cur;
        } else {
            s_coef = a.coef;
            s_cur = a.cur;
        }
    }
    __syncthreads();
    const Coef c = s_coef;
    const int cur = s_cur;
    uint32_t bad = 0;
    const int64_t total = a.vstart[a.n_shards];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int s = 0;
    if constexpr (!QZ) {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
            while (i >= a.vstart[s + 1]) ++s;
            float th[VEC];
            bad |= step_elements<CAP, VEC, ND, FAST>(a.grads[s], a.n_d, a.params[s], a.n[s], c,
                                                     (i - a.vstart[s]) * VEC, a.master[s][cur], a.m[s][cur],
                                                     a.v[s][cur], a.master[s][cur ^ 1], a.m[s][cur ^ 1],
                                                     a.v[s][cur ^ 1], th);
        }
    } else {
        static_assert(VEC == 8 || VEC == 16, "qwZ needs the vector layouts");
        constexpr int G = kQwzBlock / VEC;
        const int lane = threadIdx.x & 31;
        for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); i0 < total; i0 += stride) {
            while (i0 >= a.vstart[s + 1]) ++s;        // the same shard for the whole warp
            const int64_t w0 = i0 - a.vstart[s];      // warp's first vector in the shard, a multiple of 32
            const int64_t li = w0 + lane;
            const bool active = li < a.n[s] / VEC;
            float th[VEC], x[VEC];
            if (active)
                bad |= step_elements<CAP, VEC, ND, FAST>(a.grads[s], a.n_d, a.params[s], a.n[s], c, li * VEC,
                                                         a.master[s][cur], a.m[s][cur], a.v[s][cur],
                                                         a.master[s][cur ^ 1], a.m[s][cur ^ 1], a.v[s][cur ^ 1], th);
#pragma unroll
            for (int j = 0; j < VEC; ++j) x[j] = active ? as_fp16_value(th[j]) : 0.0f;
            int8_t q[VEC];
            const float scale = qwz_group_codes<VEC, G>(x, active ? VEC : 0, q);
            const int64_t block = (w0 + (lane & ~(G - 1))) * VEC / kQwzBlock;
            if ((block + 1) * kQwzBlock <= a.n[s]) {  // full block: every lane of the group is active
                if (ZS_RANGE_OK(kSiteQwzFused, li * VEC, VEC, a.n[s])) store_codes<VEC>(a.qcodes[s] + li * VEC, q);
                if ((lane & (G - 1)) == 0 && ZS_RANGE_OK(kSiteScale, block, 1, (a.n[s] + kQwzBlock - 1) / kQwzBlock))
                    a.qscales[s][block] = scale;
            }
        }
    }
    if (VEC > 1) {
        for (int t = blockIdx.x; t < a.n_shards; t += gridDim.x) {
            const int64_t e = a.n[t] / VEC * VEC + threadIdx.x;
            if (e < a.n[t]) {
                float th[1];
                bad |= step_elements<CAP, 1, ND, FAST>(a.grads[t], a.n_d, a.params[t], a.n[t], c, e,
                                                       a.master[t][cur], a.m[t][cur], a.v[t][cur],
                                                       a.master[t][cur ^ 1], a.m[t][cur ^ 1], a.v[t][cur ^ 1], th);
            }
        }
    }
    const int any_bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        if (any_bad) atomicOr(a.flag, 1);
        if constexpr (!QZ) {
            if (a.commit != nullptr) arrive_and_finish(a.commit, gridDim.x, a.hp.beta1, a.hp.beta2);
        }
    }
}

// ---------------------------------------------------------- commit kernel ---

struct CommitShard {
    uint16_t* params;
    const float* master[2];
    int64_t n;
    int8_t* qcodes;  // qwZ copy or nullptr
    float* qscales;
};

template <int MAXS>
struct CommitArgs {
    CommitShard shards[MAXS];
    int32_t n_shards;
    int32_t early_dependents;  // restore pass: let the next kernel be scheduled before waiting
    double beta1, beta2;
    zs_ctrl* ctrl;
};

// params = fp16_rn(master) over [0, n) by the whole grid.
__device__ __forceinline__ void cast_range(const float* master, uint16_t* params, int64_t n, int64_t tid,
                                           int64_t stride) {
    const bool vec = ((reinterpret_cast<uintptr_t>(master) | reinterpret_cast<uintptr_t>(params)) & 15) == 0;
    int64_t done = 0;
    if (vec) {
        const int64_t nvec = n / 8;
        for (int64_t i = tid; i < nvec; i += stride) {
            float x[8];
            if (!ZS_RANGE_OK(kSiteCast, 8 * i, 8, n)) continue;
            Mem<8>::load_f(master + 8 * i, x);
            Mem<8>::store_h(params + 8 * i, x);
        }
        done = nvec * 8;
    }
    for (int64_t j = done + tid; j < n; j += stride) {
        float x[1];
        if (!ZS_RANGE_OK(kSiteCast, j, 1, n)) continue;
        Mem<1>::load_f(master + j, x);
        Mem<1>::store_h(params + j, x);
    }
}

// qwZ blocks [b0, b1) of one shard, one warp per block (warp gw of nw, in
// grid-stride order).  With master: the fp16 values are re-cast from it and
// written to params first (the restore of a dropped step); without: they are
// read from params.  Then each block's scale and codes are written.  Lane l
// holds the block's values 8l .. 8l+7; the trailing partial block is masked.
__device__ void qwz_blocks(const float* master, uint16_t* params, int64_t n, int8_t* codes, float* scales,
                           int64_t b0, int64_t b1, int64_t gw, int64_t nw) {
    const int lane = threadIdx.x & 31;
    const bool vec = ((reinterpret_cast<uintptr_t>(master) | reinterpret_cast<uintptr_t>(params)) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(codes) & 7) == 0;
    for (int64_t b = b0 + gw; b < b1; b += nw) {
        const int64_t e0 = b * kQwzBlock + 8 * lane;
        const int64_t left = n - e0;
        int valid = left <= 0 ? 0 : (left >= 8 ? 8 : (int)left);
        // b is the same in every lane of the warp, so this skip keeps the warp
        // together for the shuffles below; a failed element check only empties
        // the lane (it still takes part in the block's max)
        if (!ZS_RANGE_OK(kSiteScale, b, 1, (n + kQwzBlock - 1) / kQwzBlock)) continue;
        const bool in_range = valid == 0 || ZS_RANGE_OK(kSiteQwz, e0, valid, n);
        if (!in_range) valid = 0;
        float x[8];
        if (vec && (b + 1) * kQwzBlock <= n && in_range) {
            if (master != nullptr) {
                Mem<8>::load_f(master + e0, x);
                Mem<8>::store_h(params + e0, x);
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = as_fp16_value(x[j]);
            } else {
                Mem<8>::load_h(params + e0, x);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                x[j] = 0.0f;
                if (j < valid) {
                    if (master != nullptr) {
                        const __half h = __float2half_rn(master[e0 + j]);
                        params[e0 + j] = __half_as_ushort(h);
                        x[j] = __half2float(h);
                    } else {
                        x[j] = __half2float(__ushort_as_half(params[e0 + j]));
                    }
                }
            }
        }
        int8_t q[8];
        const float scale = qwz_group_codes<8, 32>(x, valid, q);
        if (vec && valid == 8) {
            store_codes<8>(codes + e0, q);
        } else {
            for (int j = 0; j < valid; ++j) codes[e0 + j] = q[j];
        }
        if (lane == 0) scales[b] = scale;
    }
}

// End of a step on the device: restore the fp16 slices (and their qwZ copies)
// if the step overflowed, else write the qwZ copy of each shard's trailing
// partial block; then the last block to finish commits or skips in the
// control block.
template <int MAXS>
__global__ void __launch_bounds__(kCommitThreads) commit_kernel(const __grid_constant__ CommitArgs<MAXS> p) {
    __shared__ int s_ovf, s_cur;
    zs_ctrl* ctrl = p.ctrl;
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        s_ovf = *reinterpret_cast<volatile int32_t*>(&ctrl->overflow);
        s_cur = *reinterpret_cast<volatile int32_t*>(&ctrl->cur);
    }
    __syncthreads();
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int s = 0; s < p.n_shards; ++s) {
        const CommitShard& sh = p.shards[s];
        const int64_t nblocks = (sh.n + kQwzBlock - 1) / kQwzBlock;
        if (s_ovf) {
            if (sh.qcodes != nullptr)
                qwz_blocks(sh.master[s_cur], sh.params, sh.n, sh.qcodes, sh.qscales, 0, nblocks, tid >> 5,
                           stride >> 5);
            else
                cast_range(sh.master[s_cur], sh.params, sh.n, tid, stride);
        } else if (sh.qcodes != nullptr && sh.n % kQwzBlock != 0) {
            qwz_blocks(nullptr, sh.params, sh.n, sh.qcodes, sh.qscales, nblocks - 1, nblocks, tid >> 5,
                       stride >> 5);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) arrive_and_finish(ctrl, gridDim.x, p.beta1, p.beta2);
}

// After a step whose last fused launch already finished it in the control
// block (arrive_and_finish): if that step overflowed, re-cast each shard's
// fp16 slice from the kept master weights (set cur, unchanged by a skip);
// otherwise every block leaves at once.  Shards with a qwZ copy do not take
// this path.  Launched with programmatic serialization, so its launch overlaps
// the end of the fused kernel; it reads the control block only after that
// kernel has completed.  With early_dependents it lets the next kernel of the
// stream be scheduled before it waits (that kernel's own wait still covers
// this one's completion): the 8-bit Adam kernel then copies its code tables
// while the step ahead drains.
template <int MAXS>
__global__ void __launch_bounds__(kCommitThreads) restore_kernel(const __grid_constant__ CommitArgs<MAXS> p) {
    __shared__ int s_ovf, s_cur;
    if (p.early_dependents) {
        griddep_launch_dependents();
        griddep_wait();
    } else {
        griddep_wait();
        griddep_launch_dependents();
    }
    if (threadIdx.x == 0) {
        s_ovf = *reinterpret_cast<volatile int32_t*>(&p.ctrl->last_overflow);
        s_cur = *reinterpret_cast<volatile int32_t*>(&p.ctrl->cur);
    }
    __syncthreads();
    if (!s_ovf) return;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int s = 0; s < p.n_shards; ++s)
        cast_range(p.shards[s].master[s_cur], p.shards[s].params, p.shards[s].n, tid, stride);
}

// qwZ blocks [b0, b1) on their own (see qwz_blocks).
__global__ void __launch_bounds__(kCastThreads) qwz_kernel(const float* master, uint16_t* params, int64_t n,
                                                           int8_t* codes, float* scales, int64_t b0, int64_t b1) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    qwz_blocks(master, params, n, codes, scales, b0, b1, tid >> 5, ((int64_t)gridDim.x * blockDim.x) >> 5);
}

// The all-gather receiver: params = fp16_rn(code * scale of its block).
__global__ void __launch_bounds__(kCastThreads) dequant_kernel(const int8_t* codes, const float* scales, int64_t n,
                                                               uint16_t* params) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const bool vec = ((reinterpret_cast<uintptr_t>(codes) & 7) | (reinterpret_cast<uintptr_t>(params) & 15)) == 0;
    int64_t done = 0;
    if (vec) {
        const int64_t nvec = n / 8;
        for (int64_t i = tid; i < nvec; i += stride) {
            if (!ZS_RANGE_OK(kSiteDequant, 8 * i, 8, n)) continue;
            const uint2 w = *reinterpret_cast<const uint2*>(codes + 8 * i);
            const float s = scales[(8 * i) / kQwzBlock];
            float x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t word = j < 4 ? w.x : w.y;
                const int8_t q = (int8_t)((word >> (8 * (j & 3))) & 0xffu);
                x[j] = __fmul_rn((float)q, s);
            }
            Mem<8>::store_h(params + 8 * i, x);
        }
        done = nvec * 8;
    }
    for (int64_t j = done + tid; j < n; j += stride) {
        if (!ZS_RANGE_OK(kSiteDequant, j, 1, n)) continue;
        float x[1] = {__fmul_rn((float)codes[j], scales[j / kQwzBlock])};
        Mem<1>::store_h(params + j, x);
    }
}

__global__ void __launch_bounds__(kCastThreads) cast_kernel(const float* master, uint16_t* params, int64_t n) {
    cast_range(master, params, n, (int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
}

__global__ void ctrl_init_kernel(zs_ctrl* ctrl, double loss_scale) {
    zs_ctrl c;
    c.loss_scale = loss_scale;
    c.beta1_pow = 1.0;
    c.beta2_pow = 1.0;
    c.step = 0;
    c.skipped = 0;
    c.cur = 0;
    c.overflow = 0;
    c.last_overflow = 0;
    c.arrivals = 0u;
    *ctrl = c;
}


}  // namespace

namespace zs {

// ------------------------------------------------------------ host helpers ---

// Persistent grid: enough blocks to fill every SM at the kernel's occupancy,
// never more than the work needs.
int persistent_blocks(const void* kernel, int threads, int64_t work_items, int max_per_sm) {
    static std::mutex mu;
    static std::unordered_map<const void*, int> per_sm;
    int bps = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = per_sm.find(kernel);
        if (it != per_sm.end()) bps = it->second;
    }
    if (bps == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kernel, threads, 0) != cudaSuccess || bps < 1)
            bps = 1;
        std::lock_guard<std::mutex> lock(mu);
        per_sm[kernel] = bps;
    }
    if (max_per_sm > 0 && bps > max_per_sm) bps = max_per_sm;
    const int64_t full = (int64_t)bps * zs::device_sm_count();
    const int64_t need = (work_items + threads - 1) / threads;
    int64_t blocks = need < full ? need : full;
    return (int)(blocks < 1 ? 1 : blocks);
}

bool valid_hp(const zs_adam* hp) {
    if (hp == nullptr) return false;
    const double v[] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
    for (double x : v)
        if (!(x == x) || x > 1e300 || x < -1e300) return false;
    if (hp->math != ZS_MATH_IEEE && hp->math != ZS_MATH_FAST) return false;
    if (hp->reserved != 0) return false;
    return hp->beta1 >= 0.0 && hp->beta1 < 1.0 && hp->beta2 >= 0.0 && hp->beta2 < 1.0 && hp->eps >= 0.0;
}

// Access width a shard's buffers allow: 2 = wide (fp32 32-byte, fp16 16-byte
// aligned), 1 = narrow (all 16-byte aligned), 0 = scalar.
int32_t check_shard(const zs_shard& s, int32_t n_d, int* width) {
    if (s.n < 0) return ZS_ERR_ARG;
    *width = 2;
    if (s.n == 0) return ZS_OK;
    if (s.grads == nullptr || s.params == nullptr) return ZS_ERR_ARG;
    for (int i = 0; i < 2; ++i)
        if (!s.master[i] || !s.m[i] || !s.v[i]) return ZS_ERR_ARG;
    auto narrow_to = [width](int w) { if (w < *width) *width = w; };
    for (int k = 0; k < n_d; ++k) {
        if (s.grads[k] == nullptr) return ZS_ERR_ARG;
        if (!zs::aligned_to(s.grads[k], 2)) return ZS_ERR_ALIGN;
        if (!zs::aligned_to(s.grads[k], 16)) narrow_to(0);
    }
    if (!zs::aligned_to(s.params, 2)) return ZS_ERR_ALIGN;
    if (!zs::aligned_to(s.params, 16)) narrow_to(0);
    for (int i = 0; i < 2; ++i) {
        const void* st[] = {s.master[i], s.m[i], s.v[i]};
        for (const void* q : st) {
            if (!zs::aligned_to(q, 4)) return ZS_ERR_ALIGN;
            if (!zs::aligned_to(q, 16)) narrow_to(0);
            else if (!zs::aligned_to(q, 32)) narrow_to(1);
        }
    }
    if ((s.qcodes == nullptr) != (s.qscales == nullptr)) return ZS_ERR_ARG;
    if (s.qcodes != nullptr) {
        if (!zs::aligned_to(s.qscales, 4)) return ZS_ERR_ALIGN;
        if (!zs::aligned_to(s.qcodes, 8)) narrow_to(0);
        else if (!zs::aligned_to(s.qcodes, 16)) narrow_to(1);
    }
    return ZS_OK;
}

int32_t launch_cast(const float* master, uint16_t* params, int64_t n, cudaStream_t stream) {
    if (n == 0) return ZS_OK;
    const int blocks = persistent_blocks((const void*)cast_kernel, kCastThreads, (n + 7) / 8);
    cast_kernel<<<blocks, kCastThreads, 0, stream>>>(master, params, n);
    return zs::check_launch("cast_kernel");
}

// qwZ blocks [b0, b1) of one shard (see qwz_blocks); master != nullptr
// re-casts the fp16 values from it first.
int32_t launch_qwz(const float* master, uint16_t* params, int64_t n, int8_t* codes, float* scales, int64_t b0,
                   int64_t b1, cudaStream_t stream) {
    if (b1 <= b0) return ZS_OK;
    const int blocks = persistent_blocks((const void*)qwz_kernel, kCastThreads, (b1 - b0) * 32);
    qwz_kernel<<<blocks, kCastThreads, 0, stream>>>(master, params, n, codes, scales, b0, b1);
    return zs::check_launch("qwz_kernel");
}

// After a synchronous step: the qwZ copy of every listed shard made to match
// its fp16 slice -- on overflow the restore re-casts the slice from master[cur]
// and re-quantizes it all (the fp16-only shards get the plain cast); else only
// the trailing partial blocks the fused kernel left (all blocks for shards the
// scalar kernel stepped).
int32_t finish_sync_step(const zs_shard* shards, int32_t n_shards, const int* width, int32_t cur, bool overflow,
                         cudaStream_t stream) {
    for (int32_t i = 0; i < n_shards; ++i) {
        const zs_shard& s = shards[i];
        const int64_t nblocks = (s.n + kQwzBlock - 1) / kQwzBlock;
        int32_t rc = ZS_OK;
        if (overflow) {
            if (s.qcodes != nullptr)
                rc = launch_qwz(s.master[cur], s.params, s.n, s.qcodes, s.qscales, 0, nblocks, stream);
            else
                rc = launch_cast(s.master[cur], s.params, s.n, stream);
        } else if (s.qcodes != nullptr && width[i] >= 1 && s.n % kQwzBlock != 0) {
            rc = launch_qwz(nullptr, s.params, s.n, s.qcodes, s.qscales, nblocks - 1, nblocks, stream);
        }
        if (rc != ZS_OK) return rc;
    }
    return ZS_OK;
}

template <int MAXS>
int32_t launch_commit_cap(const zs_shard* shards, int32_t n_shards, const zs_adam& hp, zs_ctrl* ctrl,
                          cudaStream_t stream) {
    CommitArgs<MAXS> a;
    for (int i = 0; i < MAXS; ++i) {
        if (i < n_shards) {
            a.shards[i].params = shards[i].params;
            a.shards[i].master[0] = shards[i].master[0];
            a.shards[i].master[1] = shards[i].master[1];
            a.shards[i].n = shards[i].n;
            a.shards[i].qcodes = shards[i].qcodes;
            a.shards[i].qscales = shards[i].qscales;
        } else {
            a.shards[i] = CommitShard{nullptr, {nullptr, nullptr}, 0, nullptr, nullptr};
        }
    }
    a.n_shards = n_shards;
    a.early_dependents = 0;
    a.beta1 = hp.beta1;
    a.beta2 = hp.beta2;
    a.ctrl = ctrl;
    // one block per SM: enough to restore the slices at full bandwidth on an
    // overflow step, few enough that a normal step costs only the arrivals;
    // programmatic serialization, as the fused launches
    const int blocks = zs::device_sm_count();
    return launch_ex(commit_kernel<MAXS>, blocks, kCommitThreads, 0, true, stream, a, "commit_kernel");
}

int32_t launch_commit(const zs_shard* shards, int32_t n_shards, const zs_adam& hp, zs_ctrl* ctrl,
                      cudaStream_t stream) {
    if (n_shards <= 1) return launch_commit_cap<1>(shards, n_shards, hp, ctrl, stream);
    if (n_shards <= 16) return launch_commit_cap<16>(shards, n_shards, hp, ctrl, stream);
    return launch_commit_cap<ZS_MAX_SHARDS>(shards, n_shards, hp, ctrl, stream);
}

int32_t check_shard_list(const zs_shard* shards, int32_t n_shards, int32_t n_d, int* width) {
    if (shards == nullptr || n_shards < 1 || n_shards > ZS_MAX_SHARDS) return ZS_ERR_ARG;
    for (int32_t i = 0; i < n_shards; ++i) {
        int32_t rc = check_shard(shards[i], n_d, &width[i]);
        if (rc != ZS_OK) return rc;
    }
    return ZS_OK;
}

}  // namespace zs

using zs::check_shard;
using zs::check_shard_list;
using zs::finish_sync_step;
using zs::launch_cast;
using zs::launch_qwz;
using zs::launch_commit;
using zs::persistent_blocks;
using zs::valid_hp;

namespace {

// How the fused launches of one step are enqueued.
struct LaunchOpts {
    zs_ctrl* commit = nullptr;  // non-null: the step's last launch finishes it in the control block
    bool pdl = false;           // launch with programmatic stream serialization
};

// Enqueues kernel<<<blocks, threads, 0, stream>>>(args) (launch_ex).
template <typename Args>
int32_t launch_kernel(void (*kernel)(Args), int blocks, int threads, bool pdl, cudaStream_t stream,
                      const Args& args, const char* name) {
    return launch_ex(kernel, blocks, threads, 0, pdl, stream, args, name);
}

template <int CAP, int VEC, int ND, bool QZ, bool FAST = false>
int32_t launch_step_vec(const StepArgs<CAP>& a, bool pdl, cudaStream_t stream) {
    const void* k = (const void*)shard_step_kernel<CAP, VEC, ND, QZ, FAST>;
    const int blocks = persistent_blocks(k, kThreads, a.n / VEC > 0 ? a.n / VEC : 1);
    return launch_kernel(shard_step_kernel<CAP, VEC, ND, QZ, FAST>, blocks, kThreads, pdl, stream, a,
                         "shard_step_kernel");
}

// ZS_MATH_FAST runs the FAST instantiation of the vector layouts without a
// qwZ copy where it measured faster: the 8-element layout (N_d = 4: +5.6 %,
// 6.76 TB/s), the 16-element layout compiled for N_d = 16, 32, 64 (+1.3 % at
// 16), and the 16-element layout with a run-time N_d on launches of at most
// kFastRuntimeWideMax elements.  That last kernel measured faster with FAST on
// short launches and slower on long ones (N_d = 8, steps back to back: +5 % at
// 8M and +2.5 % at 15.6M elements; -3 % at 24M and 32M, -2.3 % at 64M and
// 100M, -1.5 % at 200M).  With a qwZ copy the 8-element kernel measured no
// gain (172.4 vs 173.4 Gparams/s at N_d = 4).
constexpr int64_t kFastRuntimeWideMax = (int64_t)1 << 24;

template <int VEC, int ND>
bool fast_pays(int64_t elements) { return VEC == 8 || ND > 0 || elements <= kFastRuntimeWideMax; }

template <int CAP, int VEC, int ND, bool QZ>
int32_t launch_math(const StepArgs<CAP>& a, bool fast, bool pdl, cudaStream_t stream) {
    if constexpr (!QZ && (VEC == 8 || VEC == 16)) {
        if (fast && fast_pays<VEC, ND>(a.n)) return launch_step_vec<CAP, VEC, ND, QZ, true>(a, pdl, stream);
    }
    return launch_step_vec<CAP, VEC, ND, QZ>(a, pdl, stream);
}

// CAP sizes the contribution table; ND > 0 compiles the kernel for exactly ND
// contributions (CAP == ND), ND == 0 reads n_d at run time.
template <int CAP, int ND>
int32_t launch_step_cap(const zs_shard& s, int32_t n_d, int width, const Coef* coef, int32_t cur,
                        const zs_adam& hp, const zs_ctrl* ctrl, int32_t* flag, const LaunchOpts& o,
                        cudaStream_t stream) {
    StepArgs<CAP> a;
    for (int k = 0; k < CAP; ++k) a.grads[k] = k < n_d ? s.grads[k] : nullptr;
    for (int i = 0; i < 2; ++i) {
        a.master[i] = s.master[i];
        a.m[i] = s.m[i];
        a.v[i] = s.v[i];
    }
    a.params = s.params;
    a.n = s.n;
    a.n_d = n_d;
    a.cur = cur;
    if (coef) a.coef = *coef; else a.coef = Coef{};
    a.hp = hp;
    a.ctrl = ctrl;
    a.flag = flag;
    a.commit = o.commit;
    a.qcodes = s.qcodes;
    a.qscales = s.qscales;
    const bool qz = s.qcodes != nullptr;
    const bool fast = hp.math == ZS_MATH_FAST;
    const bool pdl = o.pdl;
    // the wide layout only pays once N_d > 4 (measured); scalar if misaligned
    if constexpr (ND == 0 || ND > 4) {
        if (width == 2 && n_d > 4)
            return qz ? launch_math<CAP, 16, ND, true>(a, fast, pdl, stream)
                      : launch_math<CAP, 16, ND, false>(a, fast, pdl, stream);
    }
    if (width >= 1)
        return qz ? launch_math<CAP, 8, ND, true>(a, fast, pdl, stream)
                  : launch_math<CAP, 8, ND, false>(a, fast, pdl, stream);
    // scalar kernel: the qwZ copy of every block follows in its own pass
    int32_t rc = launch_step_vec<CAP, 1, ND, false>(a, pdl, stream);
    if (rc == ZS_OK && qz)
        rc = launch_qwz(nullptr, s.params, s.n, s.qcodes, s.qscales, 0, (s.n + kQwzBlock - 1) / kQwzBlock, stream);
    return rc;
}

int32_t launch_step(const zs_shard& s, int32_t n_d, int width, const Coef* coef, int32_t cur,
                    const zs_adam& hp, const zs_ctrl* ctrl, int32_t* flag, const LaunchOpts& o,
                    cudaStream_t stream) {
    // A kernel compiled for the exact count pays for 16 or more contributions
    // (measured: +3.4% at N_d = 16, +0.5% at N_d = 64).  For N_d <= 8 the
    // straight-line version issued every contribution load at once and ran
    // 4-7% slower than the run-time loop, so small counts use the latter.
    switch (n_d) {
    case 16: return launch_step_cap<16, 16>(s, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    case 32: return launch_step_cap<32, 32>(s, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    case 64: return launch_step_cap<64, 64>(s, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    default: break;
    }
    if (n_d <= 4) return launch_step_cap<4, 0>(s, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    if (n_d <= 16) return launch_step_cap<16, 0>(s, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    if (n_d <= 64) return launch_step_cap<64, 0>(s, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    return launch_step_cap<ZS_MAX_ND, 0>(s, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
}

// One launch of the grouped kernel over shards[0, count), all with access
// width `width` (1 or 2) and no qwZ copy.
template <int CAP, int ND>
int32_t launch_group_cap(const zs_shard* shards, int count, int32_t n_d, int width, const Coef* coef, int32_t cur,
                         const zs_adam& hp, const zs_ctrl* ctrl, int32_t* flag, const LaunchOpts& o,
                         cudaStream_t stream) {
    GroupArgs<CAP> a;
    const int vec = (width == 2 && n_d > 4) ? 16 : 8;
    const bool qz = shards[0].qcodes != nullptr;   // all or none of the group
    a.vstart[0] = 0;
    for (int g = 0; g < kGroupMax; ++g) {
        const bool on = g < count;
        const bool live = on && shards[g].n > 0;   // an empty shard's table may be NULL
        for (int k = 0; k < CAP; ++k) a.grads[g][k] = live && k < n_d ? shards[g].grads[k] : nullptr;
        for (int i = 0; i < 2; ++i) {
            a.master[g][i] = on ? shards[g].master[i] : nullptr;
            a.m[g][i] = on ? shards[g].m[i] : nullptr;
            a.v[g][i] = on ? shards[g].v[i] : nullptr;
        }
        a.params[g] = on ? shards[g].params : nullptr;
        a.n[g] = on ? shards[g].n : 0;
        a.qcodes[g] = on ? shards[g].qcodes : nullptr;
        a.qscales[g] = on ? shards[g].qscales : nullptr;
        if (g < count) {
            const int64_t nv = shards[g].n / vec;
            a.vstart[g + 1] = a.vstart[g] + (qz ? (nv + 31) / 32 * 32 : nv);   // warp-aligned for qwZ
        }
    }
    for (int g = count + 1; g <= kGroupMax; ++g) a.vstart[g] = a.vstart[count];
    a.n_shards = count;
    a.n_d = n_d;
    a.cur = cur;
    if (coef) a.coef = *coef; else a.coef = Coef{};
    a.hp = hp;
    a.ctrl = ctrl;
    a.flag = flag;
    a.commit = o.commit;
    const bool fast = hp.math == ZS_MATH_FAST;
    auto go = [&](auto kernel) {
        const int blocks = persistent_blocks((const void*)kernel, kThreads, a.vstart[count] > 0 ? a.vstart[count] : 1);
        return launch_kernel(kernel, blocks, kThreads, o.pdl, stream, a, "group_step_kernel");
    };
    // the same kernel choice as for one shard (launch_step_cap / launch_math)
    if constexpr (ND == 0 || ND > 4) {
        if (vec == 16) {
            if (qz) return go(group_step_kernel<CAP, 16, ND, true, false>);
            if (fast && fast_pays<16, ND>(a.vstart[count] * 16)) return go(group_step_kernel<CAP, 16, ND, false, true>);
            return go(group_step_kernel<CAP, 16, ND, false, false>);
        }
    }
    if (qz) return go(group_step_kernel<CAP, 8, ND, true, false>);
    if (fast) return go(group_step_kernel<CAP, 8, ND, false, true>);
    return go(group_step_kernel<CAP, 8, ND, false, false>);
}

int32_t launch_group(const zs_shard* shards, int count, int32_t n_d, int width, const Coef* coef, int32_t cur,
                     const zs_adam& hp, const zs_ctrl* ctrl, int32_t* flag, const LaunchOpts& o,
                     cudaStream_t stream) {
    switch (n_d) {
    case 16: return launch_group_cap<16, 16>(shards, count, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    case 32: return launch_group_cap<32, 32>(shards, count, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    case 64: return launch_group_cap<64, 64>(shards, count, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    default: break;
    }
    if (n_d <= 4) return launch_group_cap<4, 0>(shards, count, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    if (n_d <= 16) return launch_group_cap<16, 0>(shards, count, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
    return launch_group_cap<64, 0>(shards, count, n_d, width, coef, cur, hp, ctrl, flag, o, stream);
}

// The fused launches of one step for shards[0, n_shards), in order: runs of
// consecutive non-empty shards with the same vector width, all with or all
// without a qwZ copy, go up to kGroupMax per launch of the grouped kernel
// (n_d <= 64); every other shard gets its own launch; empty shards launch
// nothing.  plan[k] = {first shard, shard count}; returns the launch count.
struct LaunchRange {
    int32_t first, count;
};
int32_t plan_steps(const zs_shard* shards, int32_t n_shards, int32_t n_d, const int* width, LaunchRange* plan) {
    int32_t np = 0, i = 0;
    while (i < n_shards) {
        if (shards[i].n == 0) { ++i; continue; }
        const bool groupable = n_d <= 64 && width[i] >= 1;
        const bool qz = shards[i].qcodes != nullptr;
        int32_t j = i + 1;
        if (groupable) {
            while (j < n_shards && j - i < kGroupMax && width[j] == width[i] && (shards[j].qcodes != nullptr) == qz &&
                   shards[j].n > 0)
                ++j;
        }
        plan[np++] = LaunchRange{i, j - i};
        i = j;
    }
    return np;
}

// Enqueues the fused launches of one step (see plan_steps).  flag: the
// step's overflow word; with flag_per_launch, launch k writes flag[first
// shard of launch k] instead.  o.commit is given to the last launch only;
// *committed says whether a launch took it (false when nothing launched).
int32_t launch_steps(const zs_shard* shards, int32_t n_shards, int32_t n_d, const int* width, const Coef* coef,
                     int32_t cur, const zs_adam& hp, const zs_ctrl* ctrl, int32_t* flag, bool flag_per_launch,
                     const LaunchOpts& o, bool* committed, cudaStream_t stream) {
    LaunchRange plan[ZS_MAX_SHARDS];
    const int32_t np = plan_steps(shards, n_shards, n_d, width, plan);
    if (committed) *committed = false;
    for (int32_t k = 0; k < np; ++k) {
        LaunchOpts ok = o;
        if (k + 1 < np) ok.commit = nullptr;
        const LaunchRange& L = plan[k];
        int32_t* f = flag_per_launch ? flag + L.first : flag;
        const int32_t rc = L.count > 1
            ? launch_group(shards + L.first, L.count, n_d, width[L.first], coef, cur, hp, ctrl, f, ok, stream)
            : launch_step(shards[L.first], n_d, width[L.first], coef, cur, hp, ctrl, f, ok, stream);
        if (rc != ZS_OK) return rc;
    }
    if (committed) *committed = o.commit != nullptr && np > 0;
    return ZS_OK;
}

// The restore pass after a step that a fused launch finished (restore_kernel),
// with programmatic serialization.
template <int MAXS>
int32_t launch_restore_cap(const zs_shard* shards, int32_t n_shards, zs_ctrl* ctrl, bool early,
                           cudaStream_t stream) {
    CommitArgs<MAXS> a;
    for (int i = 0; i < MAXS; ++i) {
        if (i < n_shards)
            a.shards[i] = CommitShard{shards[i].params, {shards[i].master[0], shards[i].master[1]}, shards[i].n,
                                      nullptr, nullptr};
        else
            a.shards[i] = CommitShard{nullptr, {nullptr, nullptr}, 0, nullptr, nullptr};
    }
    a.n_shards = n_shards;
    a.early_dependents = early ? 1 : 0;
    a.beta1 = 0.0;
    a.beta2 = 0.0;
    a.ctrl = ctrl;
    // one block per SM, as the commit kernel: full bandwidth for the restore
    return launch_kernel(restore_kernel<MAXS>, zs::device_sm_count(), kCommitThreads, true, stream, a,
                         "restore_kernel");
}

int32_t launch_restore(const zs_shard* shards, int32_t n_shards, zs_ctrl* ctrl, cudaStream_t stream,
                       bool early = false) {
    if (n_shards <= 1) return launch_restore_cap<1>(shards, n_shards, ctrl, early, stream);
    if (n_shards <= 16) return launch_restore_cap<16>(shards, n_shards, ctrl, early, stream);
    return launch_restore_cap<ZS_MAX_SHARDS>(shards, n_shards, ctrl, early, stream);
}

}  // namespace

namespace zs {
uint64_t take_fault_shard_step() { return take_fault(); }
int32_t launch_restore_pass(const zs_shard* shards, int32_t n_shards, zs_ctrl* ctrl, cudaStream_t stream,
                            bool early_dependents) {
    return launch_restore(shards, n_shards, ctrl, stream, early_dependents);
}
}  // namespace zs

extern "C" {

ZS_API int32_t zero_shard_step(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                               const zs_adam* hp, double loss_scale, int64_t step, int32_t cur,
                               int32_t* flag_dev, void* stream, int32_t* overflow_out) {
    zs::NvtxRange nvtx_range("zero_shard_step");
    if (n_d < 1 || n_d > ZS_MAX_ND || !valid_hp(hp) || !(loss_scale > 0.0) || loss_scale > 1e300 ||
        step < 1 || (cur != 0 && cur != 1) || flag_dev == nullptr || overflow_out == nullptr)
        return ZS_ERR_ARG;
    if (!zs::aligned_to(flag_dev, 4)) return ZS_ERR_ALIGN;
    int width[ZS_MAX_SHARDS];
    int32_t rc = check_shard_list(shards, n_shards, n_d, width);
    if (rc != ZS_OK) return rc;

    // Adam time t = step: beta^t by repeated multiplication
    double p1 = 1.0, p2 = 1.0;
    for (int64_t i = 0; i < step; ++i) {
        p1 *= hp->beta1;
        p2 *= hp->beta2;
    }
    const Coef coef = coef_host(*hp, p1, p2, n_d, loss_scale);
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t err = cudaMemsetAsync(flag_dev, 0, sizeof(int32_t), st);
    if (err != cudaSuccess) return zs::cuda_fail(err, "zero_shard_step: clear flag");
    rc = launch_steps(shards, n_shards, n_d, width, &coef, cur, *hp, nullptr, flag_dev, false, LaunchOpts{}, nullptr,
                      st);
    if (rc != ZS_OK) return rc;
    int32_t flag = 0;
    err = cudaMemcpyAsync(&flag, flag_dev, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return zs::cuda_fail(err, "zero_shard_step: read flag");
    // overflow: restore the fp16 slices (and qwZ copies); else finish the qwZ tails
    rc = finish_sync_step(shards, n_shards, width, cur, flag != 0, st);
    if (rc != ZS_OK) return rc;
    err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return zs::cuda_fail(err, "zero_shard_step: restore");
    *overflow_out = flag ? 1 : 0;
    return ZS_OK;
}

// ------------------------------------------------ no-allocation entry point ---

// Overflow words of zero_shard_step_noalloc, one per shard of a call.  Lives in
// the library image: every device that loads the library has its own copy for
// the life of the process.  Host code must not use the symbol as an address;
// noalloc_scratch() looks up the device address.
static __device__ __align__(256) int32_t g_noalloc_scratch[ZS_NOALLOC_MAX_SHARDS];

// Device address of g_noalloc_scratch for the current device and context,
// looked up once per (device, context) pair, with that device current, and
// cached.  The context is identified by the driver's context ID, unique for
// the life of the process, so a context made after cudaDeviceReset (which
// reloads the library's module, possibly at another address) gets its own
// lookup instead of a stale pointer, even if its handle repeats.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The calling thread's current context ID (0 if there is no current context
// or the driver cannot say).
static unsigned long long current_context_id() {
    static const std::pair<CtxGetCurrentFn, CtxGetIdFn> fns = [] {
        void* get = nullptr;
        void* id = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        const cudaError_t e1 = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &get, 12000, cudaEnableDefault, &q1);
        const cudaError_t e2 = cudaGetDriverEntryPointByVersion("cuCtxGetId", &id, 12000, cudaEnableDefault, &q2);
        if (e1 != cudaSuccess || e2 != cudaSuccess) cudaGetLastError();  // a failed query leaves nothing behind
        if (e1 != cudaSuccess || q1 != cudaDriverEntryPointSuccess) get = nullptr;
        if (e2 != cudaSuccess || q2 != cudaDriverEntryPointSuccess) id = nullptr;
        return std::make_pair(reinterpret_cast<CtxGetCurrentFn>(get), reinterpret_cast<CtxGetIdFn>(id));
    }();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (fns.first == nullptr || fns.second == nullptr || fns.first(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        fns.second(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

static int32_t* noalloc_scratch(int32_t* status) {
    static std::mutex mu;
    static std::map<std::pair<int, unsigned long long>, int32_t*> cache;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) {
        *status = zs::cuda_fail(err, "zero_shard_step_noalloc: cudaGetDevice");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_context_id();
    if (id != 0) {
        auto it = cache.find(std::make_pair(dev, id));
        if (it != cache.end()) return it->second;
    }
    // first call in this context (the lookup also makes the device's context
    // current if no CUDA call has yet)
    void* addr = nullptr;
    err = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (err != cudaSuccess || addr == nullptr) {
        *status = zs::cuda_fail(err != cudaSuccess ? err : cudaErrorInvalidSymbol,
                                "zero_shard_step_noalloc: cudaGetSymbolAddress");
        return nullptr;
    }
    const unsigned long long id_now = current_context_id();
    if (id_now != 0) cache[std::make_pair(dev, id_now)] = static_cast<int32_t*>(addr);
    return static_cast<int32_t*>(addr);
}

ZS_API int32_t zero_shard_step_noalloc(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                       const zs_adam* hp, double loss_scale, int64_t step,
                                       int32_t cur, void* stream, int32_t* overflow_out) {
    zs::NvtxRange nvtx_range("zero_shard_step_noalloc");
    if (n_d < 1 || n_d > ZS_MAX_ND || !valid_hp(hp) || !(loss_scale > 0.0) || loss_scale > 1e300 ||
        step < 1 || (cur != 0 && cur != 1) || overflow_out == nullptr)
        return ZS_ERR_ARG;
    if (n_shards > ZS_NOALLOC_MAX_SHARDS)
        return zs::fail_with(ZS_ERR_ARG, "zero_shard_step_noalloc: n_shards exceeds ZS_NOALLOC_MAX_SHARDS "
                                         "(the size of its static scratch)");
    int width[ZS_NOALLOC_MAX_SHARDS];
    int32_t rc = check_shard_list(shards, n_shards, n_d, width);
    if (rc != ZS_OK) return rc;
    int32_t* scratch = noalloc_scratch(&rc);
    if (scratch == nullptr) return rc;

    double p1 = 1.0, p2 = 1.0;
    for (int64_t i = 0; i < step; ++i) {
        p1 *= hp->beta1;
        p2 *= hp->beta2;
    }
    const Coef coef = coef_host(*hp, p1, p2, n_d, loss_scale);
    cudaStream_t st = (cudaStream_t)stream;
    // the array keeps the previous call's words: clear the ones this call uses
    cudaError_t err = cudaMemsetAsync(scratch, 0, sizeof(int32_t) * n_shards, st);
    if (err != cudaSuccess) return zs::cuda_fail(err, "zero_shard_step_noalloc: clear scratch");
    // the launches of zero_shard_step (grouped where the shards allow); each
    // launch ORs into the word of its first shard
    rc = launch_steps(shards, n_shards, n_d, width, &coef, cur, *hp, nullptr, scratch, true, LaunchOpts{}, nullptr,
                      st);
    if (rc != ZS_OK) return rc;
    int32_t words[ZS_NOALLOC_MAX_SHARDS];
    err = cudaMemcpyAsync(words, scratch, sizeof(int32_t) * n_shards, cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return zs::cuda_fail(err, "zero_shard_step_noalloc: read scratch");
    int32_t flag = 0;
    for (int32_t i = 0; i < n_shards; ++i) flag |= words[i];
    rc = finish_sync_step(shards, n_shards, width, cur, flag != 0, st);
    if (rc != ZS_OK) return rc;
    err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return zs::cuda_fail(err, "zero_shard_step_noalloc: restore");
    *overflow_out = flag ? 1 : 0;
    return ZS_OK;
}

ZS_API int32_t zero_ctrl_init(zs_ctrl* ctrl_dev, double loss_scale, void* stream) {
    if (ctrl_dev == nullptr || !(loss_scale > 0.0) || loss_scale > 1e300) return ZS_ERR_ARG;
    if (!zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    ctrl_init_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(ctrl_dev, loss_scale);
    return zs::check_launch("zero_ctrl_init");
}

ZS_API int32_t zero_shard_reduce_adam_async(const zs_shard* shard, int32_t n_d, const zs_adam* hp,
                                            zs_ctrl* ctrl_dev, void* stream) {
    if (shard == nullptr || n_d < 1 || n_d > ZS_MAX_ND || !valid_hp(hp) || ctrl_dev == nullptr)
        return ZS_ERR_ARG;
    if (!zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    int width = 0;
    int32_t rc = check_shard(*shard, n_d, &width);
    if (rc != ZS_OK) return rc;
    if (shard->n == 0) return ZS_OK;
    return launch_step(*shard, n_d, width, nullptr, 0, *hp, ctrl_dev, &ctrl_dev->overflow, LaunchOpts{},
                       (cudaStream_t)stream);
}

ZS_API int32_t zero_step_commit_async(const zs_shard* shards, int32_t n_shards, const zs_adam* hp,
                                      zs_ctrl* ctrl_dev, void* stream) {
    if (shards == nullptr || n_shards < 1 || n_shards > ZS_MAX_SHARDS || !valid_hp(hp) || ctrl_dev == nullptr)
        return ZS_ERR_ARG;
    if (!zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    for (int32_t i = 0; i < n_shards; ++i) {
        const zs_shard& s = shards[i];
        if (s.n < 0) return ZS_ERR_ARG;
        if (s.n > 0 && (!s.params || !s.master[0] || !s.master[1])) return ZS_ERR_ARG;
        if (!zs::aligned_to(s.params, 2) || !zs::aligned_to(s.master[0], 4) || !zs::aligned_to(s.master[1], 4))
            return ZS_ERR_ALIGN;
    }
    return launch_commit(shards, n_shards, *hp, ctrl_dev, (cudaStream_t)stream);
}

ZS_API int32_t zero_shard_step_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                     const zs_adam* hp, zs_ctrl* ctrl_dev, void* stream) {
    zs::NvtxRange nvtx_range("zero_shard_step_async");
    if (n_d < 1 || n_d > ZS_MAX_ND || !valid_hp(hp) || ctrl_dev == nullptr) return ZS_ERR_ARG;
    if (!zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    int width[ZS_MAX_SHARDS];
    int32_t rc = check_shard_list(shards, n_shards, n_d, width);
    if (rc != ZS_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    // Without a qwZ copy the step's last fused launch finishes the step in the
    // control block itself and a restore pass follows (it leaves at once unless
    // the step overflowed); with one, the commit kernel ends the step and also
    // writes the qwZ copies' trailing blocks.  Every launch carries
    // programmatic serialization.
    bool any_qwz = false;
    for (int32_t i = 0; i < n_shards; ++i) any_qwz |= shards[i].qcodes != nullptr;
    LaunchOpts o;
    o.commit = any_qwz ? nullptr : ctrl_dev;
    o.pdl = true;
    bool committed = false;
    rc = launch_steps(shards, n_shards, n_d, width, nullptr, 0, *hp, ctrl_dev, &ctrl_dev->overflow, false, o,
                      &committed, st);
    if (rc != ZS_OK) return rc;
    if (committed) return launch_restore(shards, n_shards, ctrl_dev, st);
    return launch_commit(shards, n_shards, *hp, ctrl_dev, st);
}

ZS_API int32_t zero_shard_reduce_adam_all_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                                const zs_adam* hp, zs_ctrl* ctrl_dev, void* stream) {
    if (n_d < 1 || n_d > ZS_MAX_ND || !valid_hp(hp) || ctrl_dev == nullptr) return ZS_ERR_ARG;
    if (!zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    int width[ZS_MAX_SHARDS];
    int32_t rc = check_shard_list(shards, n_shards, n_d, width);
    if (rc != ZS_OK) return rc;
    LaunchOpts o;
    o.pdl = true;   // the commit kernel that ends this split form waits for them
    return launch_steps(shards, n_shards, n_d, width, nullptr, 0, *hp, ctrl_dev, &ctrl_dev->overflow, false, o,
                        nullptr, (cudaStream_t)stream);
}

// Device-usable address of page-locked, mapped host memory (nullptr if the
// pointer is not such memory).
static void* mapped_host_pointer(const void* host) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of a failed query
        return nullptr;
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return nullptr;
    return attr.devicePointer;
}

ZS_API int32_t zero_shard_step_host(const zs_shard* shard, int32_t n_d, const zs_adam* hp,
                                    zs_ctrl* ctrl_dev, void* stream, int32_t* overflow_out) {
    zs::NvtxRange nvtx_range("zero_shard_step_host");
    if (shard == nullptr || n_d < 1 || n_d > ZS_MAX_ND || !valid_hp(hp) || ctrl_dev == nullptr ||
        overflow_out == nullptr)
        return ZS_ERR_ARG;
    if (!zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    int width = 0;
    int32_t rc = check_shard(*shard, n_d, &width);
    if (rc != ZS_OK) return rc;
    const uint16_t* mapped[ZS_MAX_ND];
    zs_shard dev = *shard;
    if (shard->n > 0) {
        for (int k = 0; k < n_d; ++k) {
            mapped[k] = static_cast<const uint16_t*>(mapped_host_pointer(shard->grads[k]));
            if (mapped[k] == nullptr) return ZS_ERR_ARG;
        }
        dev.grads = mapped;
        dev.params = static_cast<uint16_t*>(mapped_host_pointer(shard->params));
        if (dev.params == nullptr) return ZS_ERR_ARG;
        if (shard->qcodes != nullptr) {  // the qwZ copy leaves through host memory too
            dev.qcodes = static_cast<int8_t*>(mapped_host_pointer(shard->qcodes));
            dev.qscales = static_cast<float*>(mapped_host_pointer(shard->qscales));
            if (dev.qcodes == nullptr || dev.qscales == nullptr) return ZS_ERR_ARG;
        }
        // the mapping may shift addresses: recompute the access width
        rc = check_shard(dev, n_d, &width);
        if (rc != ZS_OK) return rc;
    }
    cudaStream_t st = (cudaStream_t)stream;
    if (dev.n > 0) {
        rc = launch_step(dev, n_d, width, nullptr, 0, *hp, ctrl_dev, &ctrl_dev->overflow, LaunchOpts{}, st);
        if (rc != ZS_OK) return rc;
    }
    rc = launch_commit(&dev, 1, *hp, ctrl_dev, st);
    if (rc != ZS_OK) return rc;
    int32_t flag = 0;
    cudaError_t err = cudaMemcpyAsync(&flag, &ctrl_dev->last_overflow, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (err == cudaSuccess) err = cudaStreamSynchronize(st);
    if (err != cudaSuccess) return zs::cuda_fail(err, "zero_shard_step_host");
    *overflow_out = flag ? 1 : 0;
    return ZS_OK;
}

ZS_API int32_t zero_qwz_quantize(const uint16_t* params_dev, int64_t n, int8_t* codes_dev, float* scales_dev,
                                 void* stream) {
    if (n < 0 || (n > 0 && (params_dev == nullptr || codes_dev == nullptr || scales_dev == nullptr)))
        return ZS_ERR_ARG;
    if (!zs::aligned_to(params_dev, 2) || !zs::aligned_to(scales_dev, 4)) return ZS_ERR_ALIGN;
    return launch_qwz(nullptr, const_cast<uint16_t*>(params_dev), n, codes_dev, scales_dev, 0,
                      (n + kQwzBlock - 1) / kQwzBlock, (cudaStream_t)stream);
}

ZS_API int32_t zero_qwz_dequantize(const int8_t* codes_dev, const float* scales_dev, int64_t n,
                                   uint16_t* params_dev, void* stream) {
    if (n < 0 || (n > 0 && (params_dev == nullptr || codes_dev == nullptr || scales_dev == nullptr)))
        return ZS_ERR_ARG;
    if (!zs::aligned_to(params_dev, 2) || !zs::aligned_to(scales_dev, 4)) return ZS_ERR_ALIGN;
    if (n == 0) return ZS_OK;
    const int blocks = persistent_blocks((const void*)dequant_kernel, kCastThreads, (n + 7) / 8);
    dequant_kernel<<<blocks, kCastThreads, 0, (cudaStream_t)stream>>>(codes_dev, scales_dev, n, params_dev);
    return zs::check_launch("dequant_kernel");
}

ZS_API int32_t zero_params_from_master(const float* master_dev, uint16_t* params_dev, int64_t n,
                                       void* stream) {
    if (n < 0 || (n > 0 && (master_dev == nullptr || params_dev == nullptr))) return ZS_ERR_ARG;
    if (!zs::aligned_to(master_dev, 4) || !zs::aligned_to(params_dev, 2)) return ZS_ERR_ALIGN;
    return launch_cast(master_dev, params_dev, n, (cudaStream_t)stream);
}

}  // extern "C"
