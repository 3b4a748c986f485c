// clip.cu -- the shard step with global gradient-norm clipping.
//
// Clipping is the one coupling of coordinates in the step: it needs
// ||g||_2 over every parameter of the model ("DeepSpeed ZeRO Stages",
// sec. 2.1, Fact 1), so the step splits in two passes around one scalar:
//   pass 1  reduce the N_d contributions (same arithmetic as the fused step),
//           test for non-finite values, and add sum_j g_j^2 of the shard to a
//           double accumulator; optionally keep g (fp32) for pass 2;
//   (ranks) sum the accumulators (an all-reduce of one double per rank;
//           shards stepped by the same call are summed in place);
//   pass 2  c = min(1, max_norm / (||g|| + 1e-6)), g' = g * c, Adam / AdamW and
//           the fp16 cast, exactly as the fused step does with g'.
// Pass 2 either re-reduces the contributions (2 N_d bytes per element) or
// reads the fp32 g kept by pass 1 (4 bytes, plus 4 written in pass 1); the
// second is cheaper once N_d > 4.  Per element the clipped step moves
// 4 N_d + 26 bytes (re-reduce) or 2 N_d + 34 bytes (kept g).  Both passes'
// launches carry programmatic serialization; in the one-call step without a
// qwZ copy, pass 2's last launch ends the step in the control block and the
// restore pass follows, as in the unclipped step.
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "zs_internal.h"

namespace {

#include "step_common.cuh"
#include "step_end.cuh"

constexpr int kClipThreads = 256;

// Shards per launch: up to 16 consecutive shards of one access width share a
// launch (their pointer tables travel in the parameter block; 1 for the
// 1024-contribution table, which alone fills it).
template <int CAP>
constexpr int clip_group() { return CAP <= 64 ? 16 : 1; }

template <int CAP>
struct ClipArgs {
    static constexpr int G = clip_group<CAP>();
    const uint16_t* grads[G][CAP];
    float* master[G][2];
    float* m[G][2];
    float* v[G][2];
    uint16_t* params[G];
    float* g[G];          // pass 1 writes / pass 2 reads it; nullptr: re-reduce
    int64_t n[G];
    int64_t vstart[G + 1];  // first vector of each shard in the launch's index space
    int32_t n_shards;
    double* sqnorm;       // pass 1 adds to it, pass 2 reads it
    double max_norm;
    int32_t n_d;
    zs_adam hp;
    const zs_ctrl* ctrl;  // loss scale, t and the ping-pong set
    int32_t* flag;        // &ctrl->overflow
    zs_ctrl* commit;      // pass 2, non-null: this launch ends the step (arrive_and_finish)
};

// Block-wide sum of one double per thread; the result is valid in thread 0.
__device__ double block_sum(double x) {
    __shared__ double s_part[32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) x = __dadd_rn(x, __shfl_down_sync(0xffffffffu, x, d));
    if (lane == 0) s_part[wid] = x;
    __syncthreads();
    x = 0.0;
    if (wid == 0) {
        if (lane < (int)(blockDim.x >> 5)) x = s_part[lane];
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) x = __dadd_rn(x, __shfl_down_sync(0xffffffffu, x, d));
    }
    return x;
}

// g_j for VEC elements of shard s from its contributions; returns the
// non-finite test.
template <int CAP, int VEC, int ND>
__device__ __forceinline__ uint32_t reduced_grad(const ClipArgs<CAP>& p, int s, float inv, int64_t e, float* g) {
    float acc[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.0f;
    sum_contributions<CAP, VEC, ND>(p.grads[s], p.n_d, e, acc);
    uint32_t bad = 0;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        bad |= nonfinite(acc[j]) ? 1u : 0u;
        g[j] = __fmul_rn(acc[j], inv);
    }
    return bad;
}

// Sum of squares of VEC floats, accurate to about 2^-48 relative, in fp32 with
// error-free transformations: g^2 = p + e exactly (p rounded, e = fma(g, g, -p))
// and hi + p = s + err exactly (TwoSum); the rounding errors are carried in
// lo.  Returned as hi + lo in double.  GB300's fp64 rate is a small fraction
// of its fp32 rate, so the double work is one conversion pair and add per
// VEC elements instead of three double operations per element.
template <int VEC>
__device__ __forceinline__ double sum_squares(const float* g) {
    float hi = 0.0f, lo = 0.0f;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        const float p = __fmul_rn(g[j], g[j]);
        const float e = __fmaf_rn(g[j], g[j], -p);
        const float s = __fadd_rn(hi, p);
        const float bp = __fsub_rn(s, hi);
        const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
        hi = s;
        lo = __fadd_rn(lo, __fadd_rn(err, e));
    }
    return __dadd_rn((double)hi, (double)lo);
}

template <int CAP, int VEC, int ND>
__device__ __forceinline__ uint32_t norm_elements(const ClipArgs<CAP>& p, int s, float inv, int64_t e, double& sq) {
    float g[VEC];
    if (!ZS_RANGE_OK(kSiteNorm, e, VEC, p.n[s])) return 0u;
    const uint32_t bad = reduced_grad<CAP, VEC, ND>(p, s, inv, e, g);
    sq = __dadd_rn(sq, sum_squares<VEC>(g));
    if (p.g[s] != nullptr) Mem<VEC>::store_f(p.g[s] + e, g);
    return bad;
}

// Both passes walk the launch's shards as one index space: vector i belongs
// to the shard s with vstart[s] <= i < vstart[s + 1]; the index only grows, so
// each thread's shard cursor only moves forward.  Each shard's tail (fewer
// than VEC elements) is taken by one block.

// Pass 1: non-finite test and sum of squares of the shards' reduced gradient.
template <int CAP, int VEC, int ND>
__global__ void __launch_bounds__(kClipThreads) grad_norm_kernel(const __grid_constant__ ClipArgs<CAP> p) {
    __shared__ float s_inv;
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0)
        s_inv = __double2float_rn(__ddiv_rn(1.0, __dmul_rn((double)p.n_d, p.ctrl->loss_scale)));
    __syncthreads();
    const float inv = s_inv;
    double sq = 0.0;
    uint32_t bad = 0;
    const int64_t total = p.vstart[p.n_shards];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int s = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        while (i >= p.vstart[s + 1]) ++s;
        bad |= norm_elements<CAP, VEC, ND>(p, s, inv, (i - p.vstart[s]) * VEC, sq);
    }
    if (VEC > 1) {
        for (int t = blockIdx.x; t < p.n_shards; t += gridDim.x) {
            const int64_t e = p.n[t] / VEC * VEC + threadIdx.x;
            if (e < p.n[t]) bad |= norm_elements<CAP, 1, ND>(p, t, inv, e, sq);
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(p.flag, 1);
    const double total_sq = block_sum(sq);
    if (threadIdx.x == 0) atomicAdd(p.sqnorm, total_sq);
}

// Pass 2: clipped Adam / AdamW update and fp16 cast.  FAST: ZS_MATH_FAST.
// The 8-element variant is held to 64 registers: four blocks per SM, as the
// unclipped step's 8-element kernel (the shard cursor would otherwise take it
// to 68 registers and three blocks).
template <int CAP, int VEC, int ND, bool FAST>
__global__ void __launch_bounds__(kClipThreads, VEC == 8 ? 4 : 0)
clipped_step_kernel(const __grid_constant__ ClipArgs<CAP> p) {
    __shared__ Coef s_coef;
    __shared__ float s_clip;
    __shared__ int s_cur;
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        const zs_ctrl* ctrl = p.ctrl;
        const double p1 = __dmul_rn(ctrl->beta1_pow, p.hp.beta1);
        const double p2 = __dmul_rn(ctrl->beta2_pow, p.hp.beta2);
        s_coef = coef_device(p.hp, p1, p2, p.n_d, ctrl->loss_scale);
        s_cur = ctrl->cur;
        // c = min(1, max_norm / (||g|| + 1e-6)), formed in double
        double c = 1.0;
        if (p.max_norm > 0.0) {
            c = __ddiv_rn(p.max_norm, __dadd_rn(__dsqrt_rn(*p.sqnorm), 1e-6));
            if (!(c < 1.0)) c = 1.0;
        }
        s_clip = __double2float_rn(c);
    }
    __syncthreads();
    const Coef c = s_coef;
    const float clip = s_clip;
    const int cur = s_cur;

    auto step = [&](auto vec_tag, int s, int64_t e) {
        constexpr int V = decltype(vec_tag)::value;
        float th[V], m[V], v[V], g[V];
        if (!ZS_RANGE_OK(kSiteClipped, e, V, p.n[s])) return;
        Mem<V>::load_f(p.master[s][cur] + e, th);
        Mem<V>::load_f(p.m[s][cur] + e, m);
        Mem<V>::load_f(p.v[s][cur] + e, v);
        if (p.g[s] != nullptr) Mem<V>::load_f(p.g[s] + e, g);
        else reduced_grad<CAP, V, ND>(p, s, c.inv, e, g);
#pragma unroll
        for (int j = 0; j < V; ++j) adam_apply<FAST>(c, __fmul_rn(g[j], clip), th[j], m[j], v[j]);
        Mem<V>::store_f(p.master[s][cur ^ 1] + e, th);
        Mem<V>::store_f(p.m[s][cur ^ 1] + e, m);
        Mem<V>::store_f(p.v[s][cur ^ 1] + e, v);
        Mem<V>::store_h(p.params[s] + e, th);
    };
    const int64_t total = p.vstart[p.n_shards];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int s = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        while (i >= p.vstart[s + 1]) ++s;
        step(std::integral_constant<int, VEC>{}, s, (i - p.vstart[s]) * VEC);
    }
    if (VEC > 1) {
        for (int t = blockIdx.x; t < p.n_shards; t += gridDim.x) {
            const int64_t e = p.n[t] / VEC * VEC + threadIdx.x;
            if (e < p.n[t]) step(std::integral_constant<int, 1>{}, t, e);
        }
    }
    if (p.commit != nullptr) {   // pass 1 has set the step's flag
        __syncthreads();
        if (threadIdx.x == 0) arrive_and_finish(p.commit, gridDim.x, p.hp.beta1, p.hp.beta2);
    }
}

// ------------------------------------------------------------ host side ---

enum class Pass { Norm, Update };

template <int CAP, int VEC, int ND, bool FAST>
int32_t launch_pass_as(Pass pass, const ClipArgs<CAP>& a, cudaStream_t stream) {
    const void* k = pass == Pass::Norm ? (const void*)grad_norm_kernel<CAP, VEC, ND>
                                       : (const void*)clipped_step_kernel<CAP, VEC, ND, FAST>;
    const int64_t work = a.vstart[a.n_shards];
    const int blocks = zs::persistent_blocks(k, kClipThreads, work > 0 ? work : 1);
    if (pass == Pass::Norm)
        return launch_ex(grad_norm_kernel<CAP, VEC, ND>, blocks, kClipThreads, 0, true, stream, a, "grad_norm_kernel");
    return launch_ex(clipped_step_kernel<CAP, VEC, ND, FAST>, blocks, kClipThreads, 0, true, stream, a,
                     "clipped_step_kernel");
}

// ZS_MATH_FAST is taken by the same layouts as in the unclipped step: the
// 8-element one and the 16-element one compiled for N_d = 16, 32, 64.
template <int CAP, int VEC, int ND>
int32_t launch_pass(Pass pass, const ClipArgs<CAP>& a, cudaStream_t stream) {
    if constexpr (VEC == 8 || (VEC == 16 && ND > 0)) {
        if (pass == Pass::Update && a.hp.math == ZS_MATH_FAST) return launch_pass_as<CAP, VEC, ND, true>(pass, a, stream);
    }
    return launch_pass_as<CAP, VEC, ND, false>(pass, a, stream);
}

// One launch of pass 1 or 2 over shards[0, count) (count <= the group size),
// all of access width `width`; g[i]: shard i's kept-g buffer or nullptr.
template <int CAP, int ND>
int32_t launch_cap(Pass pass, const zs_shard* shards, int count, int32_t n_d, int width, float* const* g,
                   double* sqnorm, double max_norm, const zs_adam& hp, zs_ctrl* ctrl, zs_ctrl* commit,
                   cudaStream_t stream) {
    using Args = ClipArgs<CAP>;
    Args a;
    const bool wide = (ND == 0 || ND > 4) && width == 2 && n_d > 4;
    const int vec = wide ? 16 : (width >= 1 ? 8 : 1);
    a.vstart[0] = 0;
    for (int q = 0; q < Args::G; ++q) {
        const bool on = q < count;
        const bool live = on && shards[q].n > 0;   // an empty shard's table may be NULL
        for (int k = 0; k < CAP; ++k) a.grads[q][k] = live && k < n_d ? shards[q].grads[k] : nullptr;
        for (int i = 0; i < 2; ++i) {
            a.master[q][i] = on ? shards[q].master[i] : nullptr;
            a.m[q][i] = on ? shards[q].m[i] : nullptr;
            a.v[q][i] = on ? shards[q].v[i] : nullptr;
        }
        a.params[q] = on ? shards[q].params : nullptr;
        a.g[q] = on && g != nullptr ? g[q] : nullptr;
        a.n[q] = on ? shards[q].n : 0;
        if (on) a.vstart[q + 1] = a.vstart[q] + shards[q].n / vec;
    }
    for (int q = count + 1; q <= Args::G; ++q) a.vstart[q] = a.vstart[count];
    a.n_shards = count;
    a.sqnorm = sqnorm;
    a.max_norm = max_norm;
    a.n_d = n_d;
    a.hp = hp;
    a.ctrl = ctrl;
    a.flag = &ctrl->overflow;
    a.commit = pass == Pass::Update ? commit : nullptr;
    if constexpr (ND == 0 || ND > 4) {
        if (wide) return launch_pass<CAP, 16, ND>(pass, a, stream);
    }
    if (width >= 1) return launch_pass<CAP, 8, ND>(pass, a, stream);
    return launch_pass<CAP, 1, ND>(pass, a, stream);
}

// Largest number of shards one launch takes for this n_d.
int group_size(int32_t n_d) { return n_d <= 64 ? clip_group<64>() : clip_group<ZS_MAX_ND>(); }

int32_t launch_by_nd(Pass pass, const zs_shard* shards, int count, int32_t n_d, int width, float* const* g,
                     double* sqnorm, double max_norm, const zs_adam& hp, zs_ctrl* ctrl, zs_ctrl* commit,
                     cudaStream_t stream) {
    switch (n_d) {
    case 16: return launch_cap<16, 16>(pass, shards, count, n_d, width, g, sqnorm, max_norm, hp, ctrl, commit, stream);
    case 32: return launch_cap<32, 32>(pass, shards, count, n_d, width, g, sqnorm, max_norm, hp, ctrl, commit, stream);
    case 64: return launch_cap<64, 64>(pass, shards, count, n_d, width, g, sqnorm, max_norm, hp, ctrl, commit, stream);
    default: break;
    }
    if (n_d <= 4) return launch_cap<4, 0>(pass, shards, count, n_d, width, g, sqnorm, max_norm, hp, ctrl, commit, stream);
    if (n_d <= 16) return launch_cap<16, 0>(pass, shards, count, n_d, width, g, sqnorm, max_norm, hp, ctrl, commit, stream);
    if (n_d <= 64) return launch_cap<64, 0>(pass, shards, count, n_d, width, g, sqnorm, max_norm, hp, ctrl, commit, stream);
    return launch_cap<ZS_MAX_ND, 0>(pass, shards, count, n_d, width, g, sqnorm, max_norm, hp, ctrl, commit, stream);
}

// Pass 1 or 2 for shards[0, n_shards): consecutive non-empty shards of one
// access width share a launch (up to the group size); after pass 2 each
// shard's qwZ copy (if any) is rebuilt from its new fp16 slice in its own pass
// (3 + 4/256 bytes per element).  commit (pass 2 only): given to the last
// launch, which then ends the step; *launched says whether anything ran.
int32_t launch_all(Pass pass, const zs_shard* shards, int32_t n_shards, int32_t n_d, const int* width,
                   float* const* g, double* sqnorm, double max_norm, const zs_adam& hp, zs_ctrl* ctrl,
                   cudaStream_t stream, zs_ctrl* commit = nullptr, bool* launched = nullptr) {
    const int gmax = group_size(n_d);
    struct Range { int32_t first, count; };
    Range plan[ZS_MAX_SHARDS];
    int32_t np = 0, i = 0;
    while (i < n_shards) {
        if (shards[i].n == 0) { ++i; continue; }
        int32_t j = i + 1;
        while (j < n_shards && j - i < gmax && width[j] == width[i] && shards[j].n > 0) ++j;
        plan[np++] = Range{i, j - i};
        i = j;
    }
    for (int32_t k = 0; k < np; ++k) {
        const int32_t first = plan[k].first, last = first + plan[k].count;
        int32_t rc = launch_by_nd(pass, shards + first, plan[k].count, n_d, width[first], g ? g + first : nullptr,
                                  sqnorm, max_norm, hp, ctrl, k + 1 == np ? commit : nullptr, stream);
        if (rc != ZS_OK) return rc;
        if (pass == Pass::Update) {
            for (int32_t q = first; q < last; ++q) {
                const zs_shard& s = shards[q];
                if (s.qcodes == nullptr) continue;
                rc = zs::launch_qwz(nullptr, s.params, s.n, s.qcodes, s.qscales, 0, (s.n + kQwzBlock - 1) / kQwzBlock,
                                    stream);
                if (rc != ZS_OK) return rc;
            }
        }
    }
    if (launched) *launched = np > 0;
    return ZS_OK;
}

// Width allowed by the shard together with its kept-g buffer (fp32 like the state).
int32_t check_with_g(const zs_shard& s, int32_t n_d, const float* g, int* width) {
    int32_t rc = zs::check_shard(s, n_d, width);
    if (rc != ZS_OK || g == nullptr || s.n == 0) return rc;
    if (!zs::aligned_to(g, 4)) return ZS_ERR_ALIGN;
    if (!zs::aligned_to(g, 16)) *width = 0;
    else if (!zs::aligned_to(g, 32) && *width > 1) *width = 1;
    return ZS_OK;
}

// Argument checks shared by the entry points; *width gets each shard's width.
int32_t check_list(const zs_shard* shards, int32_t n_shards, int32_t n_d, float* const* g, const double* sqnorm,
                   const zs_ctrl* ctrl, int* width) {
    if (shards == nullptr || n_shards < 1 || n_shards > ZS_MAX_SHARDS || n_d < 1 || n_d > ZS_MAX_ND ||
        sqnorm == nullptr || ctrl == nullptr)
        return ZS_ERR_ARG;
    if (!zs::aligned_to(sqnorm, 8) || !zs::aligned_to(ctrl, 8)) return ZS_ERR_ALIGN;
    for (int32_t i = 0; i < n_shards; ++i) {
        int32_t rc = check_with_g(shards[i], n_d, g ? g[i] : nullptr, &width[i]);
        if (rc != ZS_OK) return rc;
    }
    return ZS_OK;
}

}  // namespace

namespace zs {
uint64_t take_fault_clip() { return take_fault(); }
}  // namespace zs

extern "C" {

ZS_API int32_t zero_shard_grad_sqnorm_all_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                                float* const* g_dev, double* sqnorm_dev, zs_ctrl* ctrl_dev,
                                                void* stream) {
    int width[ZS_MAX_SHARDS];
    int32_t rc = check_list(shards, n_shards, n_d, g_dev, sqnorm_dev, ctrl_dev, width);
    if (rc != ZS_OK) return rc;
    const zs_adam none{0.0, 0.0, 0.0, 0.0, 0.0, 0, 0};
    return launch_all(Pass::Norm, shards, n_shards, n_d, width, g_dev, sqnorm_dev, 0.0, none, ctrl_dev,
                      (cudaStream_t)stream);
}

ZS_API int32_t zero_shard_clipped_adam_all_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                                 const zs_adam* hp, double max_norm, float* const* g_dev,
                                                 const double* sqnorm_dev, zs_ctrl* ctrl_dev, void* stream) {
    if (!zs::valid_hp(hp) || !(max_norm == max_norm)) return ZS_ERR_ARG;
    int width[ZS_MAX_SHARDS];
    int32_t rc = check_list(shards, n_shards, n_d, g_dev, sqnorm_dev, ctrl_dev, width);
    if (rc != ZS_OK) return rc;
    return launch_all(Pass::Update, shards, n_shards, n_d, width, g_dev, const_cast<double*>(sqnorm_dev), max_norm,
                      *hp, ctrl_dev, (cudaStream_t)stream);
}

ZS_API int32_t zero_shard_grad_sqnorm_async(const zs_shard* shard, int32_t n_d, float* g_dev,
                                            double* sqnorm_dev, zs_ctrl* ctrl_dev, void* stream) {
    float* const g[1] = {g_dev};
    return zero_shard_grad_sqnorm_all_async(shard, 1, n_d, g_dev ? g : nullptr, sqnorm_dev, ctrl_dev, stream);
}

ZS_API int32_t zero_shard_clipped_adam_async(const zs_shard* shard, int32_t n_d, const zs_adam* hp,
                                             double max_norm, const float* g_dev, const double* sqnorm_dev,
                                             zs_ctrl* ctrl_dev, void* stream) {
    float* const g[1] = {const_cast<float*>(g_dev)};
    return zero_shard_clipped_adam_all_async(shard, 1, n_d, hp, max_norm, g_dev ? g : nullptr, sqnorm_dev,
                                             ctrl_dev, stream);
}

ZS_API int32_t zero_shard_step_clipped_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                             const zs_adam* hp, double max_norm, float* const* g_dev,
                                             double* sqnorm_dev, zs_ctrl* ctrl_dev, void* stream) {
    zs::NvtxRange nvtx_range("zero_shard_step_clipped_async");
    if (!zs::valid_hp(hp) || !(max_norm == max_norm)) return ZS_ERR_ARG;
    int width[ZS_MAX_SHARDS];
    int32_t rc = check_list(shards, n_shards, n_d, g_dev, sqnorm_dev, ctrl_dev, width);
    if (rc != ZS_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t err = cudaMemsetAsync(sqnorm_dev, 0, sizeof(double), st);
    if (err != cudaSuccess) return zs::cuda_fail(err, "zero_shard_step_clipped_async: clear sqnorm");
    const zs_adam none{0.0, 0.0, 0.0, 0.0, 0.0, 0, 0};
    rc = launch_all(Pass::Norm, shards, n_shards, n_d, width, g_dev, sqnorm_dev, 0.0, none, ctrl_dev, st);
    if (rc != ZS_OK) return rc;
    // Without a qwZ copy, pass 2's last launch ends the step in the control
    // block and the restore pass follows; with one (rebuilt after pass 2), or
    // with nothing launched, the commit kernel ends it.
    bool any_qwz = false;
    for (int32_t i = 0; i < n_shards; ++i) any_qwz |= shards[i].qcodes != nullptr;
    bool launched = false;
    rc = launch_all(Pass::Update, shards, n_shards, n_d, width, g_dev, sqnorm_dev, max_norm, *hp, ctrl_dev, st,
                    any_qwz ? nullptr : ctrl_dev, &launched);
    if (rc != ZS_OK) return rc;
    if (!any_qwz && launched) return zs::launch_restore_pass(shards, n_shards, ctrl_dev, st);
    return zs::launch_commit(shards, n_shards, *hp, ctrl_dev, st);
}

}  // extern "C"
