// layout.cu -- partition of the flat parameter buffer into N_d shards, on the
// host and as a single-block CUDA kernel.
//
// "DeepSpeed ZeRO Stages", sec. 2: the scalar index set {1..Psi} is split into
// disjoint sets P_1..P_Nd that cover it, |P_i| ~ Psi / N_d, rank i owning P_i.
// Sec. 3.2: gradients live in one pre-allocated flat contiguous buffer.  The
// tensors are therefore packed back to back in list order; the flat index set
// is padded to the least multiple of N_d * align and cut into N_d equal,
// contiguous shards.  A fragment is one tensor's overlap with one shard; a
// tensor may straddle any number of shard boundaries.
#include <stdint.h>

#include "zs_internal.h"

namespace {

inline bool is_pow2(int32_t x) { return x > 0 && (x & (x - 1)) == 0; }

// ---------------------------------------------------------------- device ---

constexpr int kLayoutThreads = 1024;

// Inclusive scan of one int64 per thread over the whole block; *total gets the
// block-wide sum.  Every thread of the block must call it.
__device__ int64_t block_inclusive_scan(int64_t x, int64_t* s_warp, int64_t* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int64_t w = (lane < nwarps) ? s_warp[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += y;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    if (wid > 0) x += s_warp[wid - 1];
    *total = s_warp[nwarps - 1];
    __syncthreads();  // s_warp is reused by the next call
    return x;
}

__global__ void __launch_bounds__(kLayoutThreads)
layout_kernel(const int64_t* __restrict__ numels, int32_t n_tensors, int32_t n_d, int32_t align,
              int64_t* __restrict__ scalars, int64_t* __restrict__ tensor_offsets,
              int64_t* __restrict__ shard_offsets, zs_fragment* __restrict__ frags, int64_t frag_cap) {
    __shared__ int64_t s_warp[32];
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();

    // flat offset of every tensor: exclusive scan of the sizes
    int64_t carry = 0;
    for (int64_t base = 0; base < n_tensors; base += blockDim.x) {
        const int64_t i = base + threadIdx.x;
        int64_t x = (i < n_tensors) ? numels[i] : 0;
        if (x < 0) {
            s_bad = 1;
            x = 0;
        }
        int64_t total;
        const int64_t incl = block_inclusive_scan(x, s_warp, &total);
        if (i < n_tensors) tensor_offsets[i] = carry + incl - x;
        carry += total;
    }
    __syncthreads();
    if (s_bad) {
        if (threadIdx.x == 0) scalars[4] = ZS_ERR_ARG;
        return;
    }

    const int64_t psi = carry;
    const int64_t unit = (int64_t)n_d * align;
    const int64_t psi_pad = (psi + unit - 1) / unit * unit;
    const int64_t s = psi_pad / n_d;
    for (int64_t i = threadIdx.x; i <= n_d; i += blockDim.x) shard_offsets[i] = i * s;

    // fragments: tensor t covers shards first..last; its pieces go to
    // consecutive slots after the pieces of tensors 0..t-1
    int64_t frag_carry = 0;
    for (int64_t base = 0; base < n_tensors; base += blockDim.x) {
        const int64_t i = base + threadIdx.x;
        int64_t cnt = 0, lo = 0, hi = 0, first = 0;
        if (i < n_tensors) {
            const int64_t numel = numels[i];
            if (numel > 0) {
                lo = tensor_offsets[i];
                hi = lo + numel;
                first = lo / s;
                cnt = (hi - 1) / s - first + 1;
            }
        }
        int64_t total;
        const int64_t pos = frag_carry + block_inclusive_scan(cnt, s_warp, &total) - cnt;
        if (frags != nullptr) {
            for (int64_t c = 0; c < cnt; ++c) {
                const int64_t sh = first + c;
                if (pos + c >= frag_cap) break;
                const int64_t a = lo > sh * s ? lo : sh * s;
                const int64_t b = hi < (sh + 1) * s ? hi : (sh + 1) * s;
                zs_fragment f;
                f.tensor = (int32_t)i;
                f.shard = (int32_t)sh;
                f.tensor_offset = a - lo;
                f.shard_offset = a - sh * s;
                f.length = b - a;
                frags[pos + c] = f;
            }
        }
        frag_carry += total;
    }
    if (threadIdx.x == 0) {
        scalars[0] = psi;
        scalars[1] = psi_pad;
        scalars[2] = s;
        scalars[3] = frag_carry;
        scalars[4] = ZS_OK;
    }
}

}  // namespace

extern "C" {

ZS_API int32_t zero_partition_layout(const int64_t* numels, int32_t n_tensors, int32_t n_d,
                                     int32_t align, int64_t* psi_out, int64_t* psi_padded_out,
                                     int64_t* shard_numel_out, int64_t* tensor_offsets,
                                     int64_t* shard_offsets, zs_fragment* frags, int64_t frag_cap,
                                     int64_t* n_frags_out) {
    if (n_tensors < 0 || n_d < 1 || n_d > ZS_MAX_ND || !is_pow2(align) || frag_cap < 0)
        return ZS_ERR_ARG;
    if (n_tensors > 0 && numels == nullptr) return ZS_ERR_ARG;
    int64_t psi = 0;
    for (int32_t t = 0; t < n_tensors; ++t) {
        if (numels[t] < 0) return ZS_ERR_ARG;
        psi += numels[t];
    }
    const int64_t unit = (int64_t)n_d * align;
    const int64_t psi_pad = (psi + unit - 1) / unit * unit;
    const int64_t s = psi_pad / n_d;
    if (psi_out) *psi_out = psi;
    if (psi_padded_out) *psi_padded_out = psi_pad;
    if (shard_numel_out) *shard_numel_out = s;
    if (shard_offsets)
        for (int32_t i = 0; i <= n_d; ++i) shard_offsets[i] = (int64_t)i * s;

    int64_t count = 0, off = 0;
    for (int32_t t = 0; t < n_tensors; ++t) {
        const int64_t lo = off, hi = off + numels[t];
        if (tensor_offsets) tensor_offsets[t] = lo;
        off = hi;
        if (hi == lo) continue;
        for (int64_t sh = lo / s; sh * s < hi; ++sh) {
            if (frags && count < frag_cap) {
                const int64_t a = lo > sh * s ? lo : sh * s;
                const int64_t b = hi < (sh + 1) * s ? hi : (sh + 1) * s;
                frags[count].tensor = t;
                frags[count].shard = (int32_t)sh;
                frags[count].tensor_offset = a - lo;
                frags[count].shard_offset = a - sh * s;
                frags[count].length = b - a;
            }
            ++count;
        }
    }
    if (n_frags_out) *n_frags_out = count;
    if (frags && count > frag_cap) return ZS_ERR_ARG;
    return ZS_OK;
}

ZS_API int32_t zero_partition_layout_device(const int64_t* numels_dev, int32_t n_tensors,
                                            int32_t n_d, int32_t align, int64_t* scalars_dev,
                                            int64_t* tensor_offsets_dev, int64_t* shard_offsets_dev,
                                            zs_fragment* frags_dev, int64_t frag_cap, void* stream) {
    zs::NvtxRange nvtx_range("zero_partition_layout_device");
    if (n_tensors < 0 || n_d < 1 || n_d > ZS_MAX_ND || !is_pow2(align) || frag_cap < 0)
        return ZS_ERR_ARG;
    if (scalars_dev == nullptr || shard_offsets_dev == nullptr) return ZS_ERR_ARG;
    if (n_tensors > 0 && (numels_dev == nullptr || tensor_offsets_dev == nullptr)) return ZS_ERR_ARG;
    const void* ptrs[] = {numels_dev, scalars_dev, tensor_offsets_dev, shard_offsets_dev, frags_dev};
    for (const void* p : ptrs)
        if (!zs::aligned_to(p, 8)) return ZS_ERR_ALIGN;
    layout_kernel<<<1, kLayoutThreads, 0, (cudaStream_t)stream>>>(
        numels_dev, n_tensors, n_d, align, scalars_dev, tensor_offsets_dev, shard_offsets_dev, frags_dev,
        frag_cap);
    return zs::check_launch("zero_partition_layout_device");
}

}  // extern "C"
