// sgd.cu -- the shard step with mixed-precision SGD with momentum.
//
// The other optimizer the pages name through its state multiplier K
// ("DeepSpeed ZeRO Stages", sec. 1.2).  Same structure as the Adam step: the
// N_d fp16 contributions are summed in rank order in fp32, averaged and
// unscaled, tested for non-finite values, and the update
//   d = g + wd theta,  b' = mu b + d,  theta' = theta - lr b'
// runs on the fp32 master and momentum (ping-pong, read set cur, write cur ^ 1)
// with the fp16 cast, every fp32 operation rounded once.  The step ends as the
// Adam step does: the last block of the step's last launch commits or skips
// in the control block (its beta^t bookkeeping is unused here), and the
// restore pass follows; the launches carry programmatic serialization.
// Per element: 2 N_d + 8 bytes read, 8 + 2 written.
#include <cuda_fp16.h>
#include <stdint.h>

#include "zs_internal.h"

namespace {

#include "step_common.cuh"
#include "step_end.cuh"

// Threads per block: 512 for the 16-element layout with 32 or more
// contributions (CAP >= 32), which at its ~80 registers puts exactly one block
// (512 threads) on each SM -- measured on the N_d = 64 shard: 7.13 TB/s
// against 5.97 TB/s for three 256-thread blocks per SM; 256 otherwise (at
// N_d = 16 the 512-thread block was 2.6 % slower).  A persistent grid must
// also fill the SMs' capacity exactly: capping it below lets the scheduler
// stack blocks on some SMs and leave others idle (4.65 TB/s).
template <int VEC, int CAP>
constexpr int sgd_threads() { return (VEC == 16 && CAP >= 32) ? 512 : 256; }

template <int CAP>
struct SgdArgs {
    const uint16_t* grads[CAP];
    float* master[2];
    float* mom[2];
    uint16_t* params;
    int64_t n;
    int32_t n_d;
    double lr, momentum, weight_decay;
    const zs_ctrl* ctrl;  // loss scale and the ping-pong set
    int32_t* flag;        // &ctrl->overflow
    zs_ctrl* commit;      // non-null: this launch ends the step (arrive_and_finish)
};

// VEC elements of one shard starting at element e (grads / n_d: its
// contribution table; params, n: its fp16 slice and length).
template <int CAP, int VEC, int ND>
__device__ __forceinline__ uint32_t sgd_elements(const uint16_t* const (&grads)[CAP], int32_t n_d, uint16_t* params,
                                                 int64_t n, float inv, float lr, float mu, float wd, int64_t e,
                                                 const float* th_in, const float* b_in, float* th_out, float* b_out) {
    float th[VEC], b[VEC], acc[VEC];
    if (!ZS_RANGE_OK(kSiteSgd, e, VEC, n)) return 0u;
    Mem<VEC>::load_f(th_in + e, th);
    Mem<VEC>::load_f(b_in + e, b);
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.0f;
    sum_contributions<CAP, VEC, ND>(grads, n_d, e, acc);
    uint32_t bad = 0;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        bad |= nonfinite(acc[j]) ? 1u : 0u;
        const float g = __fmul_rn(acc[j], inv);
        const float d = __fadd_rn(g, __fmul_rn(wd, th[j]));
        b[j] = __fadd_rn(__fmul_rn(mu, b[j]), d);
        th[j] = __fsub_rn(th[j], __fmul_rn(lr, b[j]));
    }
    Mem<VEC>::store_f(th_out + e, th);
    Mem<VEC>::store_f(b_out + e, b);
    Mem<VEC>::store_h(params + e, th);
    return bad;
}

template <int CAP, int VEC, int ND>
__global__ void __launch_bounds__(sgd_threads<VEC, CAP>()) sgd_step_kernel(const __grid_constant__ SgdArgs<CAP> p) {
    __shared__ float s_inv;
    __shared__ int s_cur;
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        s_inv = __double2float_rn(__ddiv_rn(1.0, __dmul_rn((double)p.n_d, p.ctrl->loss_scale)));
        s_cur = p.ctrl->cur;
    }
    __syncthreads();
    const float inv = s_inv;
    const int cur = s_cur;
    const float lr = __double2float_rn(p.lr), mu = __double2float_rn(p.momentum), wd = __double2float_rn(p.weight_decay);
    const float* th_in = p.master[cur];
    const float* b_in = p.mom[cur];
    float* th_out = p.master[cur ^ 1];
    float* b_out = p.mom[cur ^ 1];
    uint32_t bad = 0;
    const int64_t nvec = p.n / VEC;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride)
        bad |= sgd_elements<CAP, VEC, ND>(p.grads, p.n_d, p.params, p.n, inv, lr, mu, wd, i * VEC, th_in, b_in, th_out,
                                          b_out);
    if (VEC > 1) {
        const int64_t e = nvec * VEC + threadIdx.x;
        if (blockIdx.x == 0 && e < p.n)
            bad |= sgd_elements<CAP, 1, ND>(p.grads, p.n_d, p.params, p.n, inv, lr, mu, wd, e, th_in, b_in, th_out, b_out);
    }
    const int any_bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        if (any_bad) atomicOr(p.flag, 1);
        if (p.commit != nullptr) arrive_and_finish(p.commit, gridDim.x, 0.0, 0.0);
    }
}

// Several shards of one step in one launch, as the Adam step's grouped kernel:
// the grid walks the shards' concatenated vectors with a forward-only shard
// cursor; each shard's tail is taken by one block.
constexpr int kSgdGroupMax = 16;

template <int CAP>
struct SgdGroupArgs {
    const uint16_t* grads[kSgdGroupMax][CAP];
    float* master[kSgdGroupMax][2];
    float* mom[kSgdGroupMax][2];
    uint16_t* params[kSgdGroupMax];
    int64_t n[kSgdGroupMax];
    int64_t vstart[kSgdGroupMax + 1];
    int32_t n_shards;
    int32_t n_d;
    double lr, momentum, weight_decay;
    const zs_ctrl* ctrl;
    int32_t* flag;
    zs_ctrl* commit;      // non-null: this launch ends the step (arrive_and_finish)
};

template <int CAP, int VEC, int ND>
__global__ void __launch_bounds__(sgd_threads<VEC, CAP>())
sgd_group_kernel(const __grid_constant__ SgdGroupArgs<CAP> a) {
    __shared__ float s_inv;
    __shared__ int s_cur;
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        s_inv = __double2float_rn(__ddiv_rn(1.0, __dmul_rn((double)a.n_d, a.ctrl->loss_scale)));
        s_cur = a.ctrl->cur;
    }
    __syncthreads();
    const float inv = s_inv;
    const int cur = s_cur;
    const float lr = __double2float_rn(a.lr), mu = __double2float_rn(a.momentum), wd = __double2float_rn(a.weight_decay);
    uint32_t bad = 0;
    const int64_t total = a.vstart[a.n_shards];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int s = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        while (i >= a.vstart[s + 1]) ++s;
        bad |= sgd_elements<CAP, VEC, ND>(a.grads[s], a.n_d, a.params[s], a.n[s], inv, lr, mu, wd,
                                          (i - a.vstart[s]) * VEC, a.master[s][cur], a.mom[s][cur],
                                          a.master[s][cur ^ 1], a.mom[s][cur ^ 1]);
    }
    if (VEC > 1) {
        for (int t = blockIdx.x; t < a.n_shards; t += gridDim.x) {
            const int64_t e = a.n[t] / VEC * VEC + threadIdx.x;
            if (e < a.n[t])
                bad |= sgd_elements<CAP, 1, ND>(a.grads[t], a.n_d, a.params[t], a.n[t], inv, lr, mu, wd, e,
                                                a.master[t][cur], a.mom[t][cur], a.master[t][cur ^ 1],
                                                a.mom[t][cur ^ 1]);
        }
    }
    const int any_bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        if (any_bad) atomicOr(a.flag, 1);
        if (a.commit != nullptr) arrive_and_finish(a.commit, gridDim.x, 0.0, 0.0);
    }
}

template <int CAP, int ND>
int32_t launch_group_cap(const zs_shard* shards, int count, int32_t n_d, int width, const zs_sgd& hp, zs_ctrl* ctrl,
                         zs_ctrl* commit, cudaStream_t stream) {
    SgdGroupArgs<CAP> a;
    const bool wide = width == 2 && n_d > 4;
    const int vec = wide ? 16 : 8;
    a.vstart[0] = 0;
    for (int g = 0; g < kSgdGroupMax; ++g) {
        const bool on = g < count;
        const bool live = on && shards[g].n > 0;   // an empty shard's table may be NULL
        for (int k = 0; k < CAP; ++k) a.grads[g][k] = live && k < n_d ? shards[g].grads[k] : nullptr;
        for (int i = 0; i < 2; ++i) {
            a.master[g][i] = on ? shards[g].master[i] : nullptr;
            a.mom[g][i] = on ? shards[g].m[i] : nullptr;
        }
        a.params[g] = on ? shards[g].params : nullptr;
        a.n[g] = on ? shards[g].n : 0;
        if (on) a.vstart[g + 1] = a.vstart[g] + shards[g].n / vec;
    }
    for (int g = count + 1; g <= kSgdGroupMax; ++g) a.vstart[g] = a.vstart[count];
    a.n_shards = count;
    a.n_d = n_d;
    a.lr = hp.lr;
    a.momentum = hp.momentum;
    a.weight_decay = hp.weight_decay;
    a.ctrl = ctrl;
    a.flag = &ctrl->overflow;
    a.commit = commit;
    auto go = [&](auto kernel, int threads) {
        const int blocks = zs::persistent_blocks((const void*)kernel, threads, a.vstart[count] > 0 ? a.vstart[count] : 1);
        return launch_ex(kernel, blocks, threads, 0, true, stream, a, "sgd_group_kernel");
    };
    if constexpr (ND == 0 || ND > 4) {
        if (wide) return go(sgd_group_kernel<CAP, 16, ND>, sgd_threads<16, CAP>());
    }
    return go(sgd_group_kernel<CAP, 8, ND>, sgd_threads<8, CAP>());
}

int32_t launch_group(const zs_shard* shards, int count, int32_t n_d, int width, const zs_sgd& hp, zs_ctrl* ctrl,
                     zs_ctrl* commit, cudaStream_t stream) {
    switch (n_d) {
    case 16: return launch_group_cap<16, 16>(shards, count, n_d, width, hp, ctrl, commit, stream);
    case 32: return launch_group_cap<32, 32>(shards, count, n_d, width, hp, ctrl, commit, stream);
    case 64: return launch_group_cap<64, 64>(shards, count, n_d, width, hp, ctrl, commit, stream);
    default: break;
    }
    if (n_d <= 4) return launch_group_cap<4, 0>(shards, count, n_d, width, hp, ctrl, commit, stream);
    if (n_d <= 16) return launch_group_cap<16, 0>(shards, count, n_d, width, hp, ctrl, commit, stream);
    return launch_group_cap<64, 0>(shards, count, n_d, width, hp, ctrl, commit, stream);
}

template <int CAP, int VEC, int ND>
int32_t launch_vec(const SgdArgs<CAP>& a, cudaStream_t stream) {
    const void* k = (const void*)sgd_step_kernel<CAP, VEC, ND>;
    constexpr int threads = sgd_threads<VEC, CAP>();
    const int blocks = zs::persistent_blocks(k, threads, a.n / VEC > 0 ? a.n / VEC : 1);
    return launch_ex(sgd_step_kernel<CAP, VEC, ND>, blocks, threads, 0, true, stream, a, "sgd_step_kernel");
}

template <int CAP, int ND>
int32_t launch_cap(const zs_shard& s, int32_t n_d, int width, const zs_sgd& hp, zs_ctrl* ctrl, zs_ctrl* commit,
                   cudaStream_t stream) {
    SgdArgs<CAP> a;
    for (int k = 0; k < CAP; ++k) a.grads[k] = k < n_d ? s.grads[k] : nullptr;
    for (int i = 0; i < 2; ++i) {
        a.master[i] = s.master[i];
        a.mom[i] = s.m[i];
    }
    a.params = s.params;
    a.n = s.n;
    a.n_d = n_d;
    a.lr = hp.lr;
    a.momentum = hp.momentum;
    a.weight_decay = hp.weight_decay;
    a.ctrl = ctrl;
    a.flag = &ctrl->overflow;
    a.commit = commit;
    if constexpr (ND == 0 || ND > 4) {
        if (width == 2 && n_d > 4) return launch_vec<CAP, 16, ND>(a, stream);
    }
    if (width >= 1) return launch_vec<CAP, 8, ND>(a, stream);
    return launch_vec<CAP, 1, ND>(a, stream);
}

int32_t launch(const zs_shard& s, int32_t n_d, int width, const zs_sgd& hp, zs_ctrl* ctrl, zs_ctrl* commit,
               cudaStream_t stream) {
    switch (n_d) {
    case 16: return launch_cap<16, 16>(s, n_d, width, hp, ctrl, commit, stream);
    case 32: return launch_cap<32, 32>(s, n_d, width, hp, ctrl, commit, stream);
    case 64: return launch_cap<64, 64>(s, n_d, width, hp, ctrl, commit, stream);
    default: break;
    }
    if (n_d <= 4) return launch_cap<4, 0>(s, n_d, width, hp, ctrl, commit, stream);
    if (n_d <= 16) return launch_cap<16, 0>(s, n_d, width, hp, ctrl, commit, stream);
    if (n_d <= 64) return launch_cap<64, 0>(s, n_d, width, hp, ctrl, commit, stream);
    return launch_cap<ZS_MAX_ND, 0>(s, n_d, width, hp, ctrl, commit, stream);
}

// Checks one SGD shard (v unused, no qwZ copy); *width as for the Adam step.
int32_t check_sgd_shard(const zs_shard& s, int32_t n_d, int* width) {
    if (s.n < 0) return ZS_ERR_ARG;
    if (s.qcodes != nullptr || s.qscales != nullptr) return ZS_ERR_ARG;
    *width = 2;
    if (s.n == 0) return ZS_OK;
    if (s.grads == nullptr || s.params == nullptr) return ZS_ERR_ARG;
    auto narrow_to = [width](int w) { if (w < *width) *width = w; };
    for (int k = 0; k < n_d; ++k) {
        if (s.grads[k] == nullptr) return ZS_ERR_ARG;
        if (!zs::aligned_to(s.grads[k], 2)) return ZS_ERR_ALIGN;
        if (!zs::aligned_to(s.grads[k], 16)) narrow_to(0);
    }
    if (!zs::aligned_to(s.params, 2)) return ZS_ERR_ALIGN;
    if (!zs::aligned_to(s.params, 16)) narrow_to(0);
    for (int i = 0; i < 2; ++i) {
        const void* st[] = {s.master[i], s.m[i]};
        for (const void* q : st) {
            if (q == nullptr) return ZS_ERR_ARG;
            if (!zs::aligned_to(q, 4)) return ZS_ERR_ALIGN;
            if (!zs::aligned_to(q, 16)) narrow_to(0);
            else if (!zs::aligned_to(q, 32)) narrow_to(1);
        }
    }
    return ZS_OK;
}

bool valid_sgd(const zs_sgd* hp) {
    if (hp == nullptr) return false;
    const double v[] = {hp->lr, hp->momentum, hp->weight_decay};
    for (double x : v)
        if (!(x == x) || x > 1e300 || x < -1e300) return false;
    return hp->momentum >= 0.0;
}

}  // namespace

namespace zs {
uint64_t take_fault_sgd() { return take_fault(); }
}  // namespace zs

extern "C" {

ZS_API int32_t zero_shard_step_sgd_async(const zs_shard* shards, int32_t n_shards, int32_t n_d, const zs_sgd* hp,
                                         zs_ctrl* ctrl_dev, void* stream) {
    zs::NvtxRange nvtx_range("zero_shard_step_sgd_async");
    if (shards == nullptr || n_shards < 1 || n_shards > ZS_MAX_SHARDS || n_d < 1 || n_d > ZS_MAX_ND ||
        !valid_sgd(hp) || ctrl_dev == nullptr)
        return ZS_ERR_ARG;
    if (!zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    int width[ZS_MAX_SHARDS];
    for (int32_t i = 0; i < n_shards; ++i) {
        int32_t rc = check_sgd_shard(shards[i], n_d, &width[i]);
        if (rc != ZS_OK) return rc;
    }
    cudaStream_t st = (cudaStream_t)stream;
    // consecutive shards with one vector width: up to 16 per grouped launch
    struct Range { int32_t first, count; bool group; };
    Range plan[ZS_MAX_SHARDS];
    int32_t np = 0, i = 0;
    while (i < n_shards) {
        if (shards[i].n == 0) { ++i; continue; }
        const bool groupable = n_d <= 64 && width[i] >= 1;
        int32_t j = i + 1;
        if (groupable)
            while (j < n_shards && j - i < kSgdGroupMax && width[j] == width[i]) ++j;
        plan[np++] = Range{i, j - i, groupable && j - i > 1};
        i = j;
    }
    // the last launch finishes the step in the control block, then the
    // restore pass follows; a step with nothing to launch ends in the commit
    // kernel (its beta^t products are unused by SGD)
    for (int32_t k = 0; k < np; ++k) {
        const Range& r = plan[k];
        zs_ctrl* commit = k + 1 == np ? ctrl_dev : nullptr;
        const int32_t rc = r.group ? launch_group(shards + r.first, r.count, n_d, width[r.first], *hp, ctrl_dev, commit, st)
                                   : launch(shards[r.first], n_d, width[r.first], *hp, ctrl_dev, commit, st);
        if (rc != ZS_OK) return rc;
    }
    if (np > 0) return zs::launch_restore_pass(shards, n_shards, ctrl_dev, st);
    const zs_adam no_adam{hp->lr, 0.0, 0.0, 0.0, 0.0};
    return zs::launch_commit(shards, n_shards, no_adam, ctrl_dev, st);
}

}  // extern "C"
