// adam8.cu -- the shard step with 8-bit Adam: m and v kept as one byte per
// element with an fp32 scale per block of 2048 elements.
//
// The optimizer the pages name through its state multiplier K = 6 ("DeepSpeed
// ZeRO Stages", sec. 1.2), after the block-wise 8-bit Adam of Dettmers et al.,
// "8-bit Optimizers via Block-wise Quantization".  One fused pass per element:
// the N_d fp16 contributions are summed in rank order in fp32, averaged,
// unscaled and tested for non-finite values (as in the fp32 step); m and v are
// dequantized from their codes and the block scale; the fp32 Adam update and
// the fp16 cast run as in the fp32 step; and m', v' are quantized again
// against the block's new largest magnitude.
//
// One CTA owns one 2048-element block per loop iteration (256 threads x 8
// elements, or 128 x 16 when N_d > 4), so the block's absmax is one warp
// shuffle reduction plus one CTA barrier, and the quantization happens in
// registers: every state byte is read once and written once.  Per element
// 2 N_d + 6 bytes are read and 8 written (+ 16 bytes per block for the scales).
//
// The nearest-code search: the map values, and for each pair of neighbours the
// largest float not above their midpoint (so `x > t` decides "nearer to the
// upper one", ties to the smaller), sit in shared memory with a bucket table
// indexed by the top bits of the float x: 128 buckets per octave over
// [2^-26, 1], each holding the number of thresholds below it.  Every bucket
// holds at most one threshold (checked when the tables are built), so a code
// costs one byte lookup, one threshold lookup and one compare.
#include <cuda_fp16.h>
#include <stdint.h>

#include <cmath>
#include <cstring>

#include "zs_internal.h"

namespace {

#include "step_common.cuh"

// index-check sites of this file (the shared ones are 1-9)
constexpr uint32_t kSiteAdam8 = 10, kSiteAdam8Scale = 11;

constexpr int kA8Block = ZS_ADAM8_BLOCK;
constexpr int kMantBits = 7;                        // buckets per octave: 2^7
constexpr int kLowOctave = 26;                      // buckets cover [2^-26, 1]; below: bucket 0
constexpr int kBucketShift = 23 - kMantBits;
constexpr int kBucketBase = (127 - kLowOctave) << kMantBits;
constexpr int kBuckets = (kLowOctave << kMantBits) + 1;   // the last one holds 1.0

// The two code maps, their decision thresholds and bucket tables.  Passed to
// the kernel by value (about 9.7 KB of the 32 KB parameter space) and copied
// to shared memory by each CTA.
struct Maps {
    float mag7[128];        // signed map (m): magnitudes
    float mag8[256];        // unsigned map (v)
    float thr7[128];        // thr7[k]: largest float <= (mag7[k] + mag7[k+1]) / 2; thr7[127] = +inf
    float thr8[256];
    uint8_t bucket7[kBuckets];   // number of thr7 entries below the bucket's first value
    uint8_t bucket8[kBuckets];
};

// ------------------------------------------------------------- host tables ---

// Value of code k of the dynamic map with `bits` bits: 0 for k = 0; otherwise
// decimal exponent E = leading zero bits of k in the field, f = bits - E - 1
// fraction bits j under the leading one: 10^-E (0.1 + 0.9 (j + 1) / 2^f), in
// double, rounded once to float.
float map_value(int k, int bits) {
    if (k == 0) return 0.0f;
    int len = 0;
    while ((k >> len) != 0) ++len;
    const int f = len - 1;
    double pow10 = 1.0;
    for (int i = 0; i < bits - len; ++i) pow10 *= 10.0;
    const double frac = 0.1 + 0.9 * ((double)(k - (1 << f) + 1) / (double)(1 << f));
    return (float)(frac / pow10);
}

// Largest float not above the midpoint of two neighbouring map values.  The
// double sum of two floats within a factor of ten of each other is exact.
float threshold(float lo, float hi) {
    const double mid = ((double)lo + (double)hi) * 0.5;
    float t = (float)mid;
    if ((double)t > mid) t = std::nextafter(t, 0.0f);
    return t;
}

// Fills the thresholds and the bucket table of one map of `count` values;
// false if some bucket would hold two thresholds.
bool build_search(const float* mag, int count, float* thr, uint8_t* bucket) {
    for (int k = 0; k + 1 < count; ++k) thr[k] = threshold(mag[k], mag[k + 1]);
    thr[count - 1] = INFINITY;
    int below = 0;  // thresholds below the current bucket's first value
    for (int b = 0; b < kBuckets; ++b) {
        const uint32_t lo_bits = (uint32_t)(b + kBucketBase) << kBucketShift;
        const uint32_t hi_bits = (uint32_t)(b + 1 + kBucketBase) << kBucketShift;
        float lo, hi;
        std::memcpy(&lo, &lo_bits, 4);
        std::memcpy(&hi, &hi_bits, 4);
        if (b == 0) lo = 0.0f;  // bucket 0 also takes every x below 2^-26
        while (below < count - 1 && thr[below] < lo) ++below;
        int inside = 0;
        for (int k = below; k < count - 1 && thr[k] < hi; ++k) ++inside;
        if (inside > 1) return false;
        bucket[b] = (uint8_t)below;
    }
    return true;
}

struct HostMaps {
    Maps maps;
    bool ok;
};

const HostMaps& host_maps() {
    static const HostMaps built = [] {
        HostMaps h;
        std::memset(&h, 0, sizeof(h));
        for (int k = 0; k < 128; ++k) h.maps.mag7[k] = map_value(k, 7);
        for (int k = 0; k < 256; ++k) h.maps.mag8[k] = map_value(k, 8);
        h.ok = build_search(h.maps.mag7, 128, h.maps.thr7, h.maps.bucket7) &&
               build_search(h.maps.mag8, 256, h.maps.thr8, h.maps.bucket8);
        return h;
    }();
    return built;
}

// ----------------------------------------------------------- device helpers ---

// Index of the map value nearest to a (0 <= a <= 1), ties to the smaller.
// A NaN a (only from a non-finite step, which the commit drops) gives 0.
__device__ __forceinline__ uint32_t nearest_code(float a, const float* thr, const uint8_t* bucket) {
    a = (a <= 1.0f) ? a : 0.0f;
    int b = (int)(__float_as_uint(a) >> kBucketShift) - kBucketBase;
    b = min(max(b, 0), kBuckets - 1);
    const uint32_t k = bucket[b];
    return k + (a > thr[k] ? 1u : 0u);
}

// VEC one-byte codes per thread: one 8- or 16-byte access.
template <int VEC> struct Codes;
template <> struct Codes<8> {
    static __device__ __forceinline__ void load(const uint8_t* p, uint32_t* c) {
        const uint2 r = __ldcs(reinterpret_cast<const uint2*>(p));
        const uint32_t w[2] = {r.x, r.y};
#pragma unroll
        for (int j = 0; j < 8; ++j) c[j] = (w[j / 4] >> (8 * (j % 4))) & 0xffu;
    }
    static __device__ __forceinline__ void store(uint8_t* p, const uint32_t* c) {
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j / 4] |= c[j] << (8 * (j % 4));
        __stcs(reinterpret_cast<uint2*>(p), make_uint2(w[0], w[1]));
    }
};
template <> struct Codes<16> {
    static __device__ __forceinline__ void load(const uint8_t* p, uint32_t* c) {
        const uint4 r = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int j = 0; j < 16; ++j) c[j] = (w[j / 4] >> (8 * (j % 4))) & 0xffu;
    }
    static __device__ __forceinline__ void store(uint8_t* p, const uint32_t* c) {
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j / 4] |= c[j] << (8 * (j % 4));
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Threads per CTA: one 2048-element block per CTA and iteration.
template <int VEC>
constexpr int a8_threads() { return kA8Block / VEC; }

template <int CAP>
struct A8Args {
    const uint16_t* grads[CAP];
    float* master[2];
    uint8_t* mq[2];
    uint8_t* vq[2];
    float* ms[2];
    float* vs[2];
    uint16_t* params;
    int64_t n;
    int32_t n_d;
    zs_adam hp;
    const zs_ctrl* ctrl;  // loss scale, t and the ping-pong set
    int32_t* flag;        // &ctrl->overflow
    Maps maps;
};

// One CTA iteration's share of a block: VEC consecutive elements from e, the
// first `valid` of them real.  Dequantizes, updates, stores master and params,
// and leaves m', v' (0 past valid) in m, v.  VECLOAD: vector accesses for a
// full share (the buffers are aligned for them).
template <int CAP, int VEC, int ND, bool FAST, bool VECLOAD>
__device__ __forceinline__ uint32_t a8_update(const A8Args<CAP>& p, const Maps& sm, const Coef& c, int cur, int64_t e,
                                              int valid, float scale_m, float scale_v, float* m, float* v) {
    float th[VEC], acc[VEC];
    uint32_t cm[VEC], cv[VEC];
    const float* th_in = p.master[cur];
    const bool full = VECLOAD && valid == VEC;
    if (full) {
        Mem<VEC>::load_f(th_in + e, th);
        Codes<VEC>::load(p.mq[cur] + e, cm);
        Codes<VEC>::load(p.vq[cur] + e, cv);
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[j] = 0.0f;
        sum_contributions<CAP, VEC, ND>(p.grads, p.n_d, e, acc);
    } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            th[j] = 0.0f;
            acc[j] = 0.0f;
            cm[j] = cv[j] = 0u;
            if (j < valid) {
                th[j] = __ldcs(th_in + e + j);
                cm[j] = p.mq[cur][e + j];
                cv[j] = p.vq[cur][e + j];
                sum_contributions<CAP, 1, ND>(p.grads, p.n_d, e + j, &acc[j]);
            }
        }
    }
    uint32_t bad = 0;
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        const float mag = sm.mag7[cm[j] & 0x7fu];
        float mj = __fmul_rn((cm[j] & 0x80u) ? -mag : mag, scale_m);
        float vj = __fmul_rn(sm.mag8[cv[j]], scale_v);
        if (j < valid) bad |= nonfinite(acc[j]) ? 1u : 0u;
        adam_update<FAST>(c, acc[j], th[j], mj, vj);
        m[j] = j < valid ? mj : 0.0f;
        v[j] = j < valid ? vj : 0.0f;
    }
    float* th_out = p.master[cur ^ 1];
    if (full) {
        Mem<VEC>::store_f(th_out + e, th);
        Mem<VEC>::store_h(p.params + e, th);
    } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j)
            if (j < valid) {
                Mem<1>::store_f(th_out + e + j, &th[j]);
                Mem<1>::store_h(p.params + e + j, &th[j]);
            }
    }
    return bad;
}

template <int CAP, int VEC, int ND, bool FAST, bool VECLOAD>
__global__ void __launch_bounds__(a8_threads<VEC>()) adam8_step_kernel(const __grid_constant__ A8Args<CAP> p) {
    constexpr int kThr = a8_threads<VEC>();
    constexpr int kWarps = kThr / 32;
    __shared__ Maps sm;
    __shared__ Coef s_coef;
    __shared__ int s_cur;
    __shared__ float s_red[2][2][kWarps];  // [iteration parity][m, v][warp]
    {
        // the tables: word copy of the parameter block into shared memory
        constexpr int kWords = (int)(sizeof(Maps) / 4);
        static_assert(sizeof(Maps) % 4 == 0, "Maps is copied by words");
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&p.maps);
        uint32_t* dst = reinterpret_cast<uint32_t*>(&sm);
        for (int i = threadIdx.x; i < kWords; i += kThr) dst[i] = src[i];
    }
    if (threadIdx.x == 0) {
        const zs_ctrl* ctrl = p.ctrl;
        const double p1 = __dmul_rn(ctrl->beta1_pow, p.hp.beta1);  // beta^(t+1)
        const double p2 = __dmul_rn(ctrl->beta2_pow, p.hp.beta2);
        s_coef = coef_device(p.hp, p1, p2, p.n_d, ctrl->loss_scale);
        s_cur = ctrl->cur;
    }
    __syncthreads();
    const Coef c = s_coef;
    const int cur = s_cur;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nq = (p.n + kA8Block - 1) / kA8Block;
    uint32_t bad = 0;
    int par = 0;
    for (int64_t q = blockIdx.x; q < nq; q += gridDim.x, par ^= 1) {
        const int64_t e = q * kA8Block + (int64_t)threadIdx.x * VEC;
        const int64_t rem = p.n - e;
        const int valid = rem >= VEC ? VEC : (rem > 0 ? (int)rem : 0);
        if (!ZS_RANGE_OK(kSiteAdam8Scale, q, 1, nq)) continue;   // (uniform over the CTA)
        const bool in_range = valid == 0 || ZS_RANGE_OK(kSiteAdam8, e, valid, p.n);
        const float scale_m = p.ms[cur][q], scale_v = p.vs[cur][q];
        float m[VEC], v[VEC];
        if (in_range) {
            bad |= a8_update<CAP, VEC, ND, FAST, VECLOAD>(p, sm, c, cur, e, valid, scale_m, scale_v, m, v);
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) m[j] = v[j] = 0.0f;
        }
        // the block's largest |m'| and v'
        float am = 0.0f, av = 0.0f;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            am = fmaxf(am, fabsf(m[j]));
            av = fmaxf(av, v[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
            av = fmaxf(av, __shfl_xor_sync(0xffffffffu, av, o));
        }
        if (lane == 0) {
            s_red[par][0][warp] = am;
            s_red[par][1][warp] = av;
        }
        __syncthreads();   // one barrier per block: the parity slot is not rewritten before every warp read it
        am = s_red[par][0][0];
        av = s_red[par][1][0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            am = fmaxf(am, s_red[par][0][w]);
            av = fmaxf(av, s_red[par][1][w]);
        }
        // codes of m' / am and v' / av
        uint32_t cm[VEC], cv[VEC];
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float xm = am > 0.0f ? __fdiv_rn(m[j], am) : 0.0f;
            const float xv = av > 0.0f ? __fdiv_rn(v[j], av) : 0.0f;
            const uint32_t k = nearest_code(fabsf(xm), sm.thr7, sm.bucket7);
            cm[j] = (xm < 0.0f && k > 0u) ? (k | 0x80u) : k;
            cv[j] = nearest_code(fabsf(xv), sm.thr8, sm.bucket8);
        }
        if (in_range && valid > 0) {
            if (VECLOAD && valid == VEC) {
                Codes<VEC>::store(p.mq[cur ^ 1] + e, cm);
                Codes<VEC>::store(p.vq[cur ^ 1] + e, cv);
            } else {
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    if (j < valid) {
                        p.mq[cur ^ 1][e + j] = (uint8_t)cm[j];
                        p.vq[cur ^ 1][e + j] = (uint8_t)cv[j];
                    }
            }
        }
        if (threadIdx.x == 0) {
            p.ms[cur ^ 1][q] = am;
            p.vs[cur ^ 1][q] = av;
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(p.flag, 1);
}

// ------------------------------------------------------------------ launch ---

// Access width a shard allows: 2 = 16 elements per thread, 1 = 8, 0 = element-wise.
int32_t check_a8_shard(const zs_adam8_shard& s, int32_t n_d, int* width) {
    if (s.n < 0) return ZS_ERR_ARG;
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
        if (s.master[i] == nullptr || s.m_codes[i] == nullptr || s.v_codes[i] == nullptr ||
            s.m_scale[i] == nullptr || s.v_scale[i] == nullptr)
            return ZS_ERR_ARG;
        if (!zs::aligned_to(s.master[i], 4) || !zs::aligned_to(s.m_scale[i], 4) || !zs::aligned_to(s.v_scale[i], 4))
            return ZS_ERR_ALIGN;
        if (!zs::aligned_to(s.master[i], 16)) narrow_to(0);
        else if (!zs::aligned_to(s.master[i], 32)) narrow_to(1);
        for (const uint8_t* q : {s.m_codes[i], s.v_codes[i]}) {
            if (!zs::aligned_to(q, 8)) narrow_to(0);
            else if (!zs::aligned_to(q, 16)) narrow_to(1);
        }
    }
    return ZS_OK;
}

template <int CAP, int VEC, int ND, bool FAST, bool VECLOAD>
int32_t launch_a8(const A8Args<CAP>& a, cudaStream_t stream) {
    const void* k = (const void*)adam8_step_kernel<CAP, VEC, ND, FAST, VECLOAD>;
    constexpr int threads = a8_threads<VEC>();
    const int64_t nq = (a.n + kA8Block - 1) / kA8Block;
    const int blocks = zs::persistent_blocks(k, threads, nq * threads);
    adam8_step_kernel<CAP, VEC, ND, FAST, VECLOAD><<<blocks, threads, 0, stream>>>(a);
    return zs::check_launch("adam8_step_kernel");
}

template <int CAP, int ND>
int32_t launch_a8_cap(const zs_adam8_shard& s, int32_t n_d, int width, const zs_adam& hp, zs_ctrl* ctrl,
                      cudaStream_t stream) {
    A8Args<CAP> a;
    for (int k = 0; k < CAP; ++k) a.grads[k] = k < n_d ? s.grads[k] : nullptr;
    for (int i = 0; i < 2; ++i) {
        a.master[i] = s.master[i];
        a.mq[i] = s.m_codes[i];
        a.vq[i] = s.v_codes[i];
        a.ms[i] = s.m_scale[i];
        a.vs[i] = s.v_scale[i];
    }
    a.params = s.params;
    a.n = s.n;
    a.n_d = n_d;
    a.hp = hp;
    a.ctrl = ctrl;
    a.flag = &ctrl->overflow;
    a.maps = host_maps().maps;
    const bool fast = hp.math == ZS_MATH_FAST;
    if constexpr (ND == 0 || ND > 4) {
        if (width == 2 && n_d > 4)
            return fast ? launch_a8<CAP, 16, ND, true, true>(a, stream) : launch_a8<CAP, 16, ND, false, true>(a, stream);
    }
    if (width >= 1)
        return fast ? launch_a8<CAP, 8, ND, true, true>(a, stream) : launch_a8<CAP, 8, ND, false, true>(a, stream);
    return launch_a8<CAP, 8, ND, false, false>(a, stream);
}

int32_t launch_a8_shard(const zs_adam8_shard& s, int32_t n_d, int width, const zs_adam& hp, zs_ctrl* ctrl,
                        cudaStream_t stream) {
    switch (n_d) {
    case 16: return launch_a8_cap<16, 16>(s, n_d, width, hp, ctrl, stream);
    case 32: return launch_a8_cap<32, 32>(s, n_d, width, hp, ctrl, stream);
    case 64: return launch_a8_cap<64, 64>(s, n_d, width, hp, ctrl, stream);
    default: break;
    }
    if (n_d <= 4) return launch_a8_cap<4, 0>(s, n_d, width, hp, ctrl, stream);
    if (n_d <= 16) return launch_a8_cap<16, 0>(s, n_d, width, hp, ctrl, stream);
    if (n_d <= 64) return launch_a8_cap<64, 0>(s, n_d, width, hp, ctrl, stream);
    return launch_a8_cap<ZS_MAX_ND, 0>(s, n_d, width, hp, ctrl, stream);
}

}  // namespace

namespace zs {
uint64_t take_fault_adam8() { return take_fault(); }
}  // namespace zs

extern "C" {

ZS_API int32_t zero_adam8_maps(float* mag7, float* mag8) {
    if (mag7 == nullptr || mag8 == nullptr) return ZS_ERR_ARG;
    const HostMaps& h = host_maps();
    if (!h.ok) return zs::fail_with(ZS_ERR_ARG, "zero_adam8_maps: a bucket of the code search holds two thresholds");
    std::memcpy(mag7, h.maps.mag7, sizeof(h.maps.mag7));
    std::memcpy(mag8, h.maps.mag8, sizeof(h.maps.mag8));
    return ZS_OK;
}

ZS_API int32_t zero_shard_step_adam8_async(const zs_adam8_shard* shards, int32_t n_shards, int32_t n_d,
                                           const zs_adam* hp, zs_ctrl* ctrl_dev, void* stream) {
    zs::NvtxRange nvtx_range("zero_shard_step_adam8_async");
    if (shards == nullptr || n_shards < 1 || n_shards > ZS_MAX_SHARDS || n_d < 1 || n_d > ZS_MAX_ND ||
        !zs::valid_hp(hp) || ctrl_dev == nullptr)
        return ZS_ERR_ARG;
    if (!zs::aligned_to(ctrl_dev, 8)) return ZS_ERR_ALIGN;
    if (!host_maps().ok)
        return zs::fail_with(ZS_ERR_ARG, "zero_shard_step_adam8_async: a bucket of the code search holds two thresholds");
    int width[ZS_MAX_SHARDS];
    for (int32_t i = 0; i < n_shards; ++i) {
        const int32_t rc = check_a8_shard(shards[i], n_d, &width[i]);
        if (rc != ZS_OK) return rc;
    }
    cudaStream_t st = (cudaStream_t)stream;
    zs_shard commit[ZS_MAX_SHARDS];
    for (int32_t i = 0; i < n_shards; ++i) {
        if (shards[i].n > 0) {
            const int32_t rc = launch_a8_shard(shards[i], n_d, width[i], *hp, ctrl_dev, st);
            if (rc != ZS_OK) return rc;
        }
        // the commit restores params from master[cur] on an overflow; it reads nothing else
        std::memset(&commit[i], 0, sizeof(zs_shard));
        commit[i].master[0] = shards[i].master[0];
        commit[i].master[1] = shards[i].master[1];
        commit[i].params = shards[i].params;
        commit[i].n = shards[i].n;
    }
    return zs::launch_commit(commit, n_shards, *hp, ctrl_dev, st);
}

}  // extern "C"
