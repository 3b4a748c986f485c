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
// 4 N_d + 26 bytes (re-reduce) or 2 N_d + 34 bytes (kept g).
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "zs_internal.h"

namespace {

#include "step_common.cuh"

constexpr int kClipThreads = 256;

template <int CAP>
struct ClipArgs {
    const uint16_t* grads[CAP];
    float* master[2];
    float* m[2];
    float* v[2];
    uint16_t* params;
    float* g;             // pass 1 writes / pass 2 reads it; nullptr: re-reduce
    double* sqnorm;       // pass 1 adds to it, pass 2 reads it
    double max_norm;
    int64_t n;
    int32_t n_d;
    zs_adam hp;
    const zs_ctrl* ctrl;  // loss scale, t and the ping-pong set
    int32_t* flag;        // &ctrl->overflow
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

// g_j for VEC elements from the contributions; returns the non-finite test.
template <int CAP, int VEC, int ND>
__device__ __forceinline__ uint32_t reduced_grad(const ClipArgs<CAP>& p, float inv, int64_t e, float* g) {
    float acc[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.0f;
    sum_contributions<CAP, VEC, ND>(p.grads, p.n_d, e, acc);
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
__device__ __forceinline__ uint32_t norm_elements(const ClipArgs<CAP>& p, float inv, int64_t e, double& sq) {
    float g[VEC];
    if (!ZS_RANGE_OK(kSiteNorm, e, VEC, p.n)) return 0u;
    const uint32_t bad = reduced_grad<CAP, VEC, ND>(p, inv, e, g);
    sq = __dadd_rn(sq, sum_squares<VEC>(g));
    if (p.g != nullptr) Mem<VEC>::store_f(p.g + e, g);
    return bad;
}

// Pass 1: non-finite test and sum of squares of the shard's reduced gradient.
template <int CAP, int VEC, int ND>
__global__ void __launch_bounds__(kClipThreads) grad_norm_kernel(const __grid_constant__ ClipArgs<CAP> p) {
    __shared__ float s_inv;
    if (threadIdx.x == 0)
        s_inv = __double2float_rn(__ddiv_rn(1.0, __dmul_rn((double)p.n_d, p.ctrl->loss_scale)));
    __syncthreads();
    const float inv = s_inv;
    double sq = 0.0;
    uint32_t bad = 0;
    const int64_t nvec = p.n / VEC;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride)
        bad |= norm_elements<CAP, VEC, ND>(p, inv, i * VEC, sq);
    if (VEC > 1) {
        const int64_t e = nvec * VEC + threadIdx.x;
        if (blockIdx.x == 0 && e < p.n) bad |= norm_elements<CAP, 1, ND>(p, inv, e, sq);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(p.flag, 1);
    const double total = block_sum(sq);
    if (threadIdx.x == 0) atomicAdd(p.sqnorm, total);
}

// Pass 2: clipped Adam / AdamW update and fp16 cast.  FAST: ZS_MATH_FAST.
template <int CAP, int VEC, int ND, bool FAST>
__global__ void __launch_bounds__(kClipThreads) clipped_step_kernel(const __grid_constant__ ClipArgs<CAP> p) {
    __shared__ Coef s_coef;
    __shared__ float s_clip;
    __shared__ int s_cur;
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
    const float* th_in = p.master[cur];
    const float* m_in = p.m[cur];
    const float* v_in = p.v[cur];
    float* th_out = p.master[cur ^ 1];
    float* m_out = p.m[cur ^ 1];
    float* v_out = p.v[cur ^ 1];

    auto step = [&](auto vec_tag, int64_t e) {
        constexpr int V = decltype(vec_tag)::value;
        float th[V], m[V], v[V], g[V];
        if (!ZS_RANGE_OK(kSiteClipped, e, V, p.n)) return;
        Mem<V>::load_f(th_in + e, th);
        Mem<V>::load_f(m_in + e, m);
        Mem<V>::load_f(v_in + e, v);
        if (p.g != nullptr) Mem<V>::load_f(p.g + e, g);
        else reduced_grad<CAP, V, ND>(p, c.inv, e, g);
#pragma unroll
        for (int j = 0; j < V; ++j) adam_apply<FAST>(c, __fmul_rn(g[j], clip), th[j], m[j], v[j]);
        Mem<V>::store_f(th_out + e, th);
        Mem<V>::store_f(m_out + e, m);
        Mem<V>::store_f(v_out + e, v);
        Mem<V>::store_h(p.params + e, th);
    };
    const int64_t nvec = p.n / VEC;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride)
        step(std::integral_constant<int, VEC>{}, i * VEC);
    if (VEC > 1) {
        const int64_t e = nvec * VEC + threadIdx.x;
        if (blockIdx.x == 0 && e < p.n) step(std::integral_constant<int, 1>{}, e);
    }
}

// ------------------------------------------------------------ host side ---

enum class Pass { Norm, Update };

template <int CAP, int VEC, int ND, bool FAST>
int32_t launch_pass_as(Pass pass, const ClipArgs<CAP>& a, cudaStream_t stream) {
    const void* k = pass == Pass::Norm ? (const void*)grad_norm_kernel<CAP, VEC, ND>
                                       : (const void*)clipped_step_kernel<CAP, VEC, ND, FAST>;
    const int blocks = zs::persistent_blocks(k, kClipThreads, a.n / VEC > 0 ? a.n / VEC : 1);
    if (pass == Pass::Norm)
        grad_norm_kernel<CAP, VEC, ND><<<blocks, kClipThreads, 0, stream>>>(a);
    else
        clipped_step_kernel<CAP, VEC, ND, FAST><<<blocks, kClipThreads, 0, stream>>>(a);
    return zs::check_launch(pass == Pass::Norm ? "grad_norm_kernel" : "clipped_step_kernel");
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

template <int CAP, int ND>
int32_t launch_cap(Pass pass, const zs_shard& s, int32_t n_d, int width, float* g, double* sqnorm,
                   double max_norm, const zs_adam& hp, zs_ctrl* ctrl, cudaStream_t stream) {
    ClipArgs<CAP> a;
    for (int k = 0; k < CAP; ++k) a.grads[k] = k < n_d ? s.grads[k] : nullptr;
    for (int i = 0; i < 2; ++i) {
        a.master[i] = s.master[i];
        a.m[i] = s.m[i];
        a.v[i] = s.v[i];
    }
    a.params = s.params;
    a.g = g;
    a.sqnorm = sqnorm;
    a.max_norm = max_norm;
    a.n = s.n;
    a.n_d = n_d;
    a.hp = hp;
    a.ctrl = ctrl;
    a.flag = &ctrl->overflow;
    if constexpr (ND == 0 || ND > 4) {
        if (width == 2 && n_d > 4) return launch_pass<CAP, 16, ND>(pass, a, stream);
    }
    if (width >= 1) return launch_pass<CAP, 8, ND>(pass, a, stream);
    return launch_pass<CAP, 1, ND>(pass, a, stream);
}

int32_t launch_by_nd(Pass pass, const zs_shard& s, int32_t n_d, int width, float* g, double* sqnorm,
                     double max_norm, const zs_adam& hp, zs_ctrl* ctrl, cudaStream_t stream) {
    switch (n_d) {
    case 16: return launch_cap<16, 16>(pass, s, n_d, width, g, sqnorm, max_norm, hp, ctrl, stream);
    case 32: return launch_cap<32, 32>(pass, s, n_d, width, g, sqnorm, max_norm, hp, ctrl, stream);
    case 64: return launch_cap<64, 64>(pass, s, n_d, width, g, sqnorm, max_norm, hp, ctrl, stream);
    default: break;
    }
    if (n_d <= 4) return launch_cap<4, 0>(pass, s, n_d, width, g, sqnorm, max_norm, hp, ctrl, stream);
    if (n_d <= 16) return launch_cap<16, 0>(pass, s, n_d, width, g, sqnorm, max_norm, hp, ctrl, stream);
    if (n_d <= 64) return launch_cap<64, 0>(pass, s, n_d, width, g, sqnorm, max_norm, hp, ctrl, stream);
    return launch_cap<ZS_MAX_ND, 0>(pass, s, n_d, width, g, sqnorm, max_norm, hp, ctrl, stream);
}

// Pass 1 or 2 for one shard; after pass 2 the shard's qwZ copy (if any) is
// rebuilt from the new fp16 slice in its own pass (3 + 4/256 bytes per element).
int32_t launch(Pass pass, const zs_shard& s, int32_t n_d, int width, float* g, double* sqnorm, double max_norm,
               const zs_adam& hp, zs_ctrl* ctrl, cudaStream_t stream) {
    int32_t rc = launch_by_nd(pass, s, n_d, width, g, sqnorm, max_norm, hp, ctrl, stream);
    if (rc == ZS_OK && pass == Pass::Update && s.qcodes != nullptr)
        rc = zs::launch_qwz(nullptr, s.params, s.n, s.qcodes, s.qscales, 0, (s.n + kQwzBlock - 1) / kQwzBlock,
                            stream);
    return rc;
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

}  // namespace

namespace zs {
uint64_t take_fault_clip() { return take_fault(); }
}  // namespace zs

extern "C" {

ZS_API int32_t zero_shard_grad_sqnorm_async(const zs_shard* shard, int32_t n_d, float* g_dev,
                                            double* sqnorm_dev, zs_ctrl* ctrl_dev, void* stream) {
    if (shard == nullptr || n_d < 1 || n_d > ZS_MAX_ND || sqnorm_dev == nullptr || ctrl_dev == nullptr)
        return ZS_ERR_ARG;
    if (!zs::aligned_to(sqnorm_dev, 8) || !zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    int width = 0;
    int32_t rc = check_with_g(*shard, n_d, g_dev, &width);
    if (rc != ZS_OK) return rc;
    if (shard->n == 0) return ZS_OK;
    const zs_adam none{0.0, 0.0, 0.0, 0.0, 0.0};
    return launch(Pass::Norm, *shard, n_d, width, g_dev, sqnorm_dev, 0.0, none, ctrl_dev, (cudaStream_t)stream);
}

ZS_API int32_t zero_shard_clipped_adam_async(const zs_shard* shard, int32_t n_d, const zs_adam* hp,
                                             double max_norm, const float* g_dev, const double* sqnorm_dev,
                                             zs_ctrl* ctrl_dev, void* stream) {
    if (shard == nullptr || n_d < 1 || n_d > ZS_MAX_ND || !zs::valid_hp(hp) || sqnorm_dev == nullptr ||
        ctrl_dev == nullptr || !(max_norm == max_norm))
        return ZS_ERR_ARG;
    if (!zs::aligned_to(sqnorm_dev, 8) || !zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    int width = 0;
    int32_t rc = check_with_g(*shard, n_d, g_dev, &width);
    if (rc != ZS_OK) return rc;
    if (shard->n == 0) return ZS_OK;
    return launch(Pass::Update, *shard, n_d, width, const_cast<float*>(g_dev), const_cast<double*>(sqnorm_dev),
                  max_norm, *hp, ctrl_dev, (cudaStream_t)stream);
}

ZS_API int32_t zero_shard_step_clipped_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                             const zs_adam* hp, double max_norm, float* const* g_dev,
                                             double* sqnorm_dev, zs_ctrl* ctrl_dev, void* stream) {
    zs::NvtxRange nvtx_range("zero_shard_step_clipped_async");
    if (n_d < 1 || n_d > ZS_MAX_ND || !zs::valid_hp(hp) || sqnorm_dev == nullptr || ctrl_dev == nullptr ||
        !(max_norm == max_norm))
        return ZS_ERR_ARG;
    if (!zs::aligned_to(sqnorm_dev, 8) || !zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    if (shards == nullptr || n_shards < 1 || n_shards > ZS_MAX_SHARDS) return ZS_ERR_ARG;
    int width[ZS_MAX_SHARDS];
    for (int32_t i = 0; i < n_shards; ++i) {
        int32_t rc = check_with_g(shards[i], n_d, g_dev ? g_dev[i] : nullptr, &width[i]);
        if (rc != ZS_OK) return rc;
    }
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t err = cudaMemsetAsync(sqnorm_dev, 0, sizeof(double), st);
    if (err != cudaSuccess) return zs::cuda_fail(err, "zero_shard_step_clipped_async: clear sqnorm");
    const zs_adam none{0.0, 0.0, 0.0, 0.0, 0.0};
    for (int32_t i = 0; i < n_shards; ++i) {
        if (shards[i].n == 0) continue;
        int32_t rc = launch(Pass::Norm, shards[i], n_d, width[i], g_dev ? g_dev[i] : nullptr, sqnorm_dev, 0.0,
                            none, ctrl_dev, st);
        if (rc != ZS_OK) return rc;
    }
    for (int32_t i = 0; i < n_shards; ++i) {
        if (shards[i].n == 0) continue;
        int32_t rc = launch(Pass::Update, shards[i], n_d, width[i], g_dev ? g_dev[i] : nullptr, sqnorm_dev,
                            max_norm, *hp, ctrl_dev, st);
        if (rc != ZS_OK) return rc;
    }
    return zs::launch_commit(shards, n_shards, *hp, ctrl_dev, st);
}

}  // extern "C"
