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
// elements, or 128 x 16 when N_d > 16), so the block's absmax is one warp
// shuffle reduction plus one CTA barrier, and the quantization happens in
// registers: every state byte is read once and written once.  Per element
// 2 N_d + 6 bytes are read and 8 written (+ 16 bytes per block for the scales).
// One launch steps up to 16 shards of a step, their blocks back to back; up to
// N_d = 4 each thread prefetches its share of the next block with cp.async.
// The step ends as the fp32 step does: the last block of the step's last
// launch commits or skips in the control block and the restore pass follows;
// the launches carry programmatic serialization, and each CTA copies the code
// tables to shared memory before it waits for the kernel ahead of it.
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
#include <map>
#include <mutex>
#include <utility>

#include "zs_internal.h"

namespace {

#include "step_common.cuh"
#include "step_end.cuh"

// index-check sites of this file (the shared ones are 1-9)
[[maybe_unused]] constexpr uint32_t kSiteAdam8 = 10, kSiteAdam8Scale = 11;

constexpr int kA8Block = ZS_ADAM8_BLOCK;
#include "adam8_math.cuh"

struct HostMaps {
    float mag7[128];        // the signed map's magnitudes
    Maps maps;
    bool ok;
};

const HostMaps& host_maps() {
    static const HostMaps built = [] {
        HostMaps h;
        std::memset(&h, 0, sizeof(h));
        for (int k = 0; k < 128; ++k) h.mag7[k] = map_value(k, 7);
        for (int c = 0; c < 256; ++c) h.maps.dec7[c] = (c & 0x80) ? -h.mag7[c & 0x7f] : h.mag7[c & 0x7f];
        for (int k = 0; k < 256; ++k) h.maps.mag8[k] = map_value(k, 8);
        h.ok = build_search(h.mag7, 128, h.maps.thr7, h.maps.bucket7) &&
               build_search(h.maps.mag8, 256, h.maps.thr8, h.maps.bucket8);
        return h;
    }();
    return built;
}

// Byte j of w, zero-extended; and four codes (each < 256) packed into a word
// (byte permutes: one instruction per byte out, three per word in).
__device__ __forceinline__ uint32_t byte_of(uint32_t w, int j) { return __byte_perm(w, 0u, 0x4440u + (uint32_t)j); }
__device__ __forceinline__ uint32_t pack4(const uint32_t* c) {
    return __byte_perm(__byte_perm(c[0], c[1], 0x0040u), __byte_perm(c[2], c[3], 0x0040u), 0x5410u);
}
template <> struct Codes<8> {
    static __device__ __forceinline__ void unpack(uint2 r, uint32_t* c) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            c[j] = byte_of(r.x, j);
            c[4 + j] = byte_of(r.y, j);
        }
    }
    static __device__ __forceinline__ void load(const uint8_t* p, uint32_t* c) {
        unpack(__ldcs(reinterpret_cast<const uint2*>(p)), c);
    }
    static __device__ __forceinline__ void store(uint8_t* p, const uint32_t* c) {
        __stcs(reinterpret_cast<uint2*>(p), make_uint2(pack4(c), pack4(c + 4)));
    }
};
template <> struct Codes<16> {
    static __device__ __forceinline__ void load(const uint8_t* p, uint32_t* c) {
        const uint4 r = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int j = 0; j < 16; ++j) c[j] = byte_of(w[j / 4], j % 4);
    }
    static __device__ __forceinline__ void store(uint8_t* p, const uint32_t* c) {
        *reinterpret_cast<uint4*>(p) = make_uint4(pack4(c), pack4(c + 4), pack4(c + 8), pack4(c + 12));
    }
};

// Threads per CTA: one 2048-element block per CTA and iteration.
template <int VEC>
constexpr int a8_threads() { return kA8Block / VEC; }

// Shards one launch steps: consecutive shards of one step with one access
// width walk their blocks back to back (one ramp and one tail per launch
// instead of one per shard).
constexpr int kA8GroupMax = 16;

// Kernel parameters for up to G shards.  bstart[s] is the launch's first block
// of shard s; bstart[n_shards .. G] hold the launch's block count.
template <int CAP, int G>
struct A8Args {
    const uint16_t* grads[G][CAP];
    float* master[G][2];
    uint8_t* mq[G][2];
    uint8_t* vq[G][2];
    float* ms[G][2];
    float* vs[G][2];
    uint16_t* params[G];
    int64_t n[G];
    int64_t bstart[G + 1];
    int32_t n_shards;
    int32_t n_d;
    zs_adam hp;
    const zs_ctrl* ctrl;  // loss scale, t and the ping-pong set
    int32_t* flag;        // &ctrl->overflow
    zs_ctrl* commit;      // non-null: this launch ends the step (arrive_and_finish)
    Maps maps;
};

// ------------------------------------------------------------------ loads ---

// One thread's share of a block: VEC consecutive elements from element e of
// shard sh.  The loaders fill th (master), acc (the summed contributions, rank
// order) and the codes cm, cv.

// all VEC elements exist and the buffers are aligned for vector accesses
template <int CAP, int G, int VEC, int ND>
__device__ __forceinline__ void a8_load_global(const A8Args<CAP, G>& p, int sh, int cur, int64_t e, float* th,
                                               float* acc, uint32_t* cm, uint32_t* cv) {
    Mem<VEC>::load_f(p.master[sh][cur] + e, th);
    Codes<VEC>::load(p.mq[sh][cur] + e, cm);
    Codes<VEC>::load(p.vq[sh][cur] + e, cv);
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.0f;
    sum_contributions<CAP, VEC, ND, true>(p.grads[sh], p.n_d, e, acc);
}

// the first `valid` (0..VEC) elements, one at a time; zeros past them (which
// give m' = v' = 0, so they change no block maximum)
template <int CAP, int G, int VEC, int ND>
__device__ __forceinline__ void a8_load_partial(const A8Args<CAP, G>& p, int sh, int cur, int64_t e, int valid,
                                                float* th, float* acc, uint32_t* cm, uint32_t* cv) {
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
        th[j] = 0.0f;
        acc[j] = 0.0f;
        cm[j] = cv[j] = 0u;
        if (j < valid) {
            th[j] = __ldcs(p.master[sh][cur] + e + j);
            cm[j] = p.mq[sh][cur][e + j];
            cv[j] = p.vq[sh][cur][e + j];
            sum_contributions<CAP, 1, ND, true>(p.grads[sh], p.n_d, e + j, &acc[j]);
        }
    }
}

// ------------------------------------------------ staged (prefetched) loads ---

// The staged kernel (8 elements per thread, 256 threads) copies each thread's
// share of the CTA's next block into shared memory with cp.async while it
// computes the current one.  Each thread reads back only what it copied
// itself, after waiting for its own copy groups: no barrier, flag or spin is
// involved.  Stage layout (bytes), for n_d contributions:
//   [k * 4096 + 16 t]           contribution k, thread t (8 fp16)
//   [G + 16 t], [G + 4096 + 16 t] master, elements 0-3 and 4-7 (G = n_d * 4096)
//   [G + 8192 + 8 t]            m codes;  [G + 10240 + 8 t]  v codes
constexpr int kStageThreads = 256;

__host__ __device__ constexpr int64_t stage_bytes(int n_d) { return (int64_t)n_d * 4096 + 12288; }

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void copy16_async(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void copy8_async(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void copies_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// returns once at most N of this thread's committed copy groups are in flight
template <int N>
__device__ __forceinline__ void copies_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int CAP, int G, int ND>
__device__ __forceinline__ void a8_prefetch(const A8Args<CAP, G>& p, int sh, int cur, int64_t e, unsigned char* st) {
    const int t = threadIdx.x;
    const int nd = ND > 0 ? ND : p.n_d;
#pragma unroll 4
    for (int k = 0; k < nd; ++k) copy16_async(st + ((int64_t)k * kStageThreads + t) * 16, p.grads[sh][k] + e);
    unsigned char* s = st + (int64_t)nd * kStageThreads * 16;
    copy16_async(s + t * 16, p.master[sh][cur] + e);
    copy16_async(s + 4096 + t * 16, p.master[sh][cur] + e + 4);
    copy8_async(s + 8192 + t * 8, p.mq[sh][cur] + e);
    copy8_async(s + 10240 + t * 8, p.vq[sh][cur] + e);
}

template <int CAP, int G, int ND>
__device__ __forceinline__ void a8_load_staged(const A8Args<CAP, G>& p, const unsigned char* st, float* th,
                                               float* acc, uint32_t* cm, uint32_t* cv) {
    const int t = threadIdx.x;
    const int nd = ND > 0 ? ND : p.n_d;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
#pragma unroll 4
    for (int k = 0; k < nd; ++k) {   // rank order, as sum_contributions
        const uint4 r = *reinterpret_cast<const uint4*>(st + ((int64_t)k * kStageThreads + t) * 16);
        add_f16x2(r.x, acc[0], acc[1]);
        add_f16x2(r.y, acc[2], acc[3]);
        add_f16x2(r.z, acc[4], acc[5]);
        add_f16x2(r.w, acc[6], acc[7]);
    }
    const unsigned char* s = st + (int64_t)nd * kStageThreads * 16;
    const float4 a = *reinterpret_cast<const float4*>(s + t * 16);
    const float4 b = *reinterpret_cast<const float4*>(s + 4096 + t * 16);
    th[0] = a.x; th[1] = a.y; th[2] = a.z; th[3] = a.w;
    th[4] = b.x; th[5] = b.y; th[6] = b.z; th[7] = b.w;
    Codes<8>::unpack(*reinterpret_cast<const uint2*>(s + 8192 + t * 8), cm);
    Codes<8>::unpack(*reinterpret_cast<const uint2*>(s + 10240 + t * 8), cv);
}

// ------------------------------------------------------------------ kernel ---

// One CTA steps one 2048-element block per loop iteration (persistent grid)
// over the blocks of the launch's shards, taken back to back: block q is
// block q - bstart[s] of shard s, found by a forward-only cursor (each CTA's
// q only grows).  VECLOAD: vector accesses for full shares; STAGED: the
// cp.async pipeline above (VEC = 8 with VECLOAD only).
// Minimum resident CTAs per SM promised to the compiler.  Four for the
// 16-element kernel (128 threads, at most 128 registers): measured on the
// 7.5B-parameter N_d = 64 shard, 47.6 Gparams/s (6.76 TB/s) against 28.9 with
// no promise (the compiler then took 124 registers and ran slower) and 32.3
// with five CTAs (102 registers, spills).  Three for the 8-element kernels
// (256 threads, at most 85 registers), the most the staged kernel's shared
// memory allows anyway.
template <int VEC, bool STAGED>
constexpr int a8_min_blocks() { return VEC == 16 ? 4 : 3; }

template <int CAP, int G, int VEC, int ND, bool FAST, bool VECLOAD, bool STAGED>
__global__ void __launch_bounds__(a8_threads<VEC>(), a8_min_blocks<VEC, STAGED>())
adam8_step_kernel(const __grid_constant__ A8Args<CAP, G> p) {
    static_assert(!STAGED || (VEC == 8 && VECLOAD), "the staged kernel moves 8 aligned elements per thread");
    constexpr int kThr = a8_threads<VEC>();
    constexpr int kWarps = kThr / 32;
    extern __shared__ __align__(16) unsigned char stages[];  // STAGED: two stages
    __shared__ Maps sm;
    __shared__ Coef s_coef;
    __shared__ int s_cur;
    static_assert(kWarps % 4 == 0, "the warps' maxima are read four at a time");
    __shared__ __align__(16) uint32_t s_red[2][2][kWarps];  // [iteration parity][m, v][warp]: bit patterns
    {
        // the tables: word copy of the parameter block into shared memory
        constexpr int kWords = (int)(sizeof(Maps) / 4);
        static_assert(sizeof(Maps) % 4 == 0, "Maps is copied by words");
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&p.maps);
        uint32_t* dst = reinterpret_cast<uint32_t*>(&sm);
        for (int i = threadIdx.x; i < kWords; i += kThr) dst[i] = src[i];
    }
    // the tables come from the kernel parameters; global memory only from here
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        const zs_ctrl* ctrl = p.ctrl;
        const double p1 = __dmul_rn(ctrl->beta1_pow, p.hp.beta1);  // beta^(t+1)
        const double p2 = __dmul_rn(ctrl->beta2_pow, p.hp.beta2);
        s_coef = coef_device(p.hp, p1, p2, p.n_d, ctrl->loss_scale);
        s_cur = ctrl->cur;
    }
    __syncthreads();
    const Coef c = s_coef;
    const float rcp_bc1 = __frcp_rn(c.bc1), rcp_bc2 = __frcp_rn(c.bc2);
    const int cur = s_cur;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t total = p.bstart[p.n_shards];
    const int64_t stage_sz = STAGED ? stage_bytes(ND > 0 ? ND : p.n_d) : 0;
    // the shard of launch block qq (qq < total), advancing *cursor
    auto shard_of = [&](int64_t qq, int* cursor) {
        while (*cursor + 1 < G && qq >= p.bstart[*cursor + 1]) ++*cursor;
        return *cursor;
    };
    int cur_shard = 0, next_shard = 0;
    // this thread's share of launch block qq: all VEC elements exist (sets
    // *sh and *e to its shard and first element)
    auto share_full = [&](int64_t qq, int* sh, int64_t* e) {
        if (qq >= total) return false;
        *sh = shard_of(qq, &next_shard);
        *e = (qq - p.bstart[*sh]) * kA8Block + (int64_t)threadIdx.x * VEC;
        return *e + VEC <= p.n[*sh] && ZS_RANGE_OK(kSiteAdam8, *e, VEC, p.n[*sh]);
    };
    bool staged = false;
    if constexpr (STAGED) {
        int sh0 = 0;
        int64_t e0 = 0;
        staged = share_full(blockIdx.x, &sh0, &e0);
        if (staged) a8_prefetch<CAP, G, ND>(p, sh0, cur, e0, stages);
        copies_commit();
    }
    uint32_t bad = 0;
    int par = 0;
    for (int64_t q = blockIdx.x; q < total; q += gridDim.x, par ^= 1) {
        const int sh = shard_of(q, &cur_shard);
        const int64_t n = p.n[sh];
        const int64_t lq = q - p.bstart[sh];  // the block within its shard
        const int64_t e = lq * kA8Block + (int64_t)threadIdx.x * VEC;
        const int64_t rem = n - e;
        const int valid = rem >= VEC ? VEC : (rem > 0 ? (int)rem : 0);
        const bool scale_ok = ZS_RANGE_OK(kSiteAdam8Scale, lq, 1, (n + kA8Block - 1) / kA8Block);
        const float scale_m = scale_ok ? p.ms[sh][cur][lq] : 0.0f, scale_v = scale_ok ? p.vs[sh][cur][lq] : 0.0f;
        float th[VEC], acc[VEC];
        uint32_t cm[VEC], cv[VEC];
        bool full;  // this share moves by vector accesses
        if constexpr (STAGED) {
            int shn = 0;
            int64_t en = 0;
            const bool next = share_full(q + gridDim.x, &shn, &en);
            if (next) a8_prefetch<CAP, G, ND>(p, shn, cur, en, stages + (par ^ 1) * stage_sz);
            copies_commit();
            copies_wait<1>();  // this block's copies have landed
            full = staged;
            if (full) a8_load_staged<CAP, G, ND>(p, stages + par * stage_sz, th, acc, cm, cv);
            staged = next;
        } else {
            full = VECLOAD && valid == VEC && ZS_RANGE_OK(kSiteAdam8, e, VEC, n);
            if (full) a8_load_global<CAP, G, VEC, ND>(p, sh, cur, e, th, acc, cm, cv);
        }
        const int live = full ? VEC : ((valid == 0 || ZS_RANGE_OK(kSiteAdam8, e, valid, n)) ? valid : 0);
        if (!full) a8_load_partial<CAP, G, VEC, ND>(p, sh, cur, e, live, th, acc, cm, cv);
        // dequantize, update, cast
        // the Adam update of the fp32 step, operation for operation, in two
        // phases so that the bias corrections can use the exact division below
        float m[VEC], v[VEC];
        float low = 1.0f;  // smallest |m'|, v' of this thread's share
        float nfs = 0.0f;  // sum of acc * 0: NaN once some acc is +-inf or NaN, else 0
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float g = __fmul_rn(acc[j], c.inv);
            nfs = __fmaf_rn(acc[j], 0.0f, nfs);
            m[j] = __fadd_rn(__fmul_rn(c.b1, __fmul_rn(sm.dec7[cm[j]], scale_m)), __fmul_rn(c.c1, g));
            v[j] = __fadd_rn(__fmul_rn(c.b2, __fmul_rn(sm.mag8[cv[j]], scale_v)), __fmul_rn(c.c2, __fmul_rn(g, g)));
            low = fminf(low, fminf(fabsf(m[j]), v[j]));
        }
        // m' / (1 - beta1^t), v' / (1 - beta2^t): exact by two corrections,
        // unless a warp holds a value below 2^-100 (or 0): then IEEE divisions
        bad |= (nfs != nfs) ? 1u : 0u;  // the non-finite test of this share
        float mh[VEC], vh[VEC];
        if (__any_sync(0xffffffffu, !(low >= 0x1p-100f))) {  // (warp-uniform)
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                mh[j] = __fdiv_rn(m[j], c.bc1);
                vh[j] = __fdiv_rn(v[j], c.bc2);
            }
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                mh[j] = div_by_constant(m[j], c.bc1, rcp_bc1);
                vh[j] = div_by_constant(v[j], c.bc2, rcp_bc2);
            }
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const float den = __fadd_rn(__fsqrt_rn(vh[j]), c.eps);
            const float u = FAST ? div_corrected(mh[j], den) : __fdiv_rn(mh[j], den);
            th[j] = __fsub_rn(th[j], __fmul_rn(c.lr, __fadd_rn(u, __fmul_rn(c.wd, th[j]))));
        }
        float* th_out = p.master[sh][cur ^ 1];
        if (full) {
            Mem<VEC>::store_f(th_out + e, th);
            Mem<VEC>::store_h(p.params[sh] + e, th);
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (j < live) {
                    Mem<1>::store_f(th_out + e + j, &th[j]);
                    Mem<1>::store_h(p.params[sh] + e + j, &th[j]);
                }
        }
        // the block's largest |m'| and v': the thread's maxima (fmaxf, which
        // passes over a NaN), then one warp reduction each on their bit
        // patterns (for floats >= 0 the largest pattern is the largest value),
        // then the warps' maxima from shared memory, read as 16-byte vectors
        float am = 0.0f, av = 0.0f;
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            am = fmaxf(am, fabsf(m[j]));
            av = fmaxf(av, v[j]);
        }
        const uint32_t am_w = __reduce_max_sync(0xffffffffu, __float_as_uint(am));
        const uint32_t av_w = __reduce_max_sync(0xffffffffu, __float_as_uint(av));
        if (lane == 0) {
            s_red[par][0][warp] = am_w;
            s_red[par][1][warp] = av_w;
        }
        __syncthreads();  // one barrier per block: a parity slot is not rewritten before every warp read it
        uint32_t am_b = 0u, av_b = 0u;
#pragma unroll
        for (int w = 0; w < kWarps; w += 4) {
            const uint4 a = *reinterpret_cast<const uint4*>(&s_red[par][0][w]);
            const uint4 b = *reinterpret_cast<const uint4*>(&s_red[par][1][w]);
            am_b = max(am_b, max(max(a.x, a.y), max(a.z, a.w)));
            av_b = max(av_b, max(max(b.x, b.y), max(b.z, b.w)));
        }
        am = __uint_as_float(am_b);
        av = __uint_as_float(av_b);
        // codes of x = m' / am and v' / av, each quotient rounded once: by the
        // constant-divisor division when both scales allow it (the block's
        // scales are the same in every thread, so the branch is uniform), else
        // by IEEE divisions; x = 0 for a zero scale
        float xm[VEC], xv[VEC];
        if (scale_divisor_ok(am) && scale_divisor_ok(av)) {
            const float rm = __frcp_rn(am), rv = __frcp_rn(av);
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                xm[j] = div_by_constant(m[j], am, rm);
                xv[j] = div_by_constant(v[j], av, rv);
            }
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j) {
                xm[j] = am > 0.0f ? __fdiv_rn(m[j], am) : 0.0f;
                xv[j] = av > 0.0f ? __fdiv_rn(v[j], av) : 0.0f;
            }
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
            const uint32_t k = nearest_code(fabsf(xm[j]), sm.thr7, sm.bucket7);
            cm[j] = (xm[j] < 0.0f && k > 0u) ? (k | 0x80u) : k;
            cv[j] = nearest_code(fabsf(xv[j]), sm.thr8, sm.bucket8);
        }
        if (full) {
            Codes<VEC>::store(p.mq[sh][cur ^ 1] + e, cm);
            Codes<VEC>::store(p.vq[sh][cur ^ 1] + e, cv);
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (j < live) {
                    p.mq[sh][cur ^ 1][e + j] = (uint8_t)cm[j];
                    p.vq[sh][cur ^ 1][e + j] = (uint8_t)cv[j];
                }
        }
        if (threadIdx.x == 0 && scale_ok) {
            p.ms[sh][cur ^ 1][lq] = am;
            p.vs[sh][cur ^ 1][lq] = av;
        }
    }
    if constexpr (STAGED) copies_wait<0>();  // (the last group is empty) nothing in flight at exit
    const int any_bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        if (any_bad) atomicOr(p.flag, 1);
        if (p.commit != nullptr) arrive_and_finish(p.commit, gridDim.x, p.hp.beta1, p.hp.beta2);
    }
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

// Persistent grid of a kernel with `smem` bytes of dynamic shared memory:
// every SM filled at the kernel's occupancy, at most one CTA per block.
int a8_blocks(const void* kernel, int threads, size_t smem, int64_t nq) {
    static std::mutex mu;
    static std::map<std::pair<const void*, size_t>, int> per_sm;
    int bps = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = per_sm.find({kernel, smem});
        if (it != per_sm.end()) bps = it->second;
    }
    if (bps == 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kernel, threads, smem) != cudaSuccess || bps < 1)
            bps = 1;
        std::lock_guard<std::mutex> lock(mu);
        per_sm[{kernel, smem}] = bps;
    }
    const int64_t full = (int64_t)bps * zs::device_sm_count();
    return (int)(nq < full ? (nq < 1 ? 1 : nq) : full);
}

// Contributions up to which the staged kernel is used: its two stages take
// 2 (4096 N_d + 12288) bytes of shared memory per CTA, 57 KB at N_d = 4 (three
// CTAs per SM).  At N_d = 8 they would allow only two, and the direct kernel
// measured faster (gpt2s workload: 134.6 against 129.9 Gparams/s).
constexpr int kStagedMaxNd = 4;

template <int CAP, int G, int VEC, int ND, bool FAST, bool VECLOAD, bool STAGED>
int32_t launch_a8(const A8Args<CAP, G>& a, cudaStream_t stream) {
    const void* k = (const void*)adam8_step_kernel<CAP, G, VEC, ND, FAST, VECLOAD, STAGED>;
    constexpr int threads = a8_threads<VEC>();
    size_t smem = 0;
    if constexpr (STAGED) {
        static const cudaError_t attr = cudaFuncSetAttribute(
            k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(2 * stage_bytes(ND > 0 ? ND : kStagedMaxNd)));
        if (attr != cudaSuccess) return zs::cuda_fail(attr, "adam8_step_kernel: shared memory attribute");
        smem = (size_t)(2 * stage_bytes(ND > 0 ? ND : a.n_d));
    }
    const int blocks = a8_blocks(k, threads, smem, a.bstart[a.n_shards]);
    return launch_ex(adam8_step_kernel<CAP, G, VEC, ND, FAST, VECLOAD, STAGED>, blocks, threads, smem, true, stream, a,
                     "adam8_step_kernel");
}

// One launch for `count` (<= G) consecutive shards of one access width.
template <int CAP, int G, int ND>
int32_t launch_a8_cap(const zs_adam8_shard* shards, int count, int32_t n_d, int width, const zs_adam& hp,
                      zs_ctrl* ctrl, zs_ctrl* commit, cudaStream_t stream) {
    A8Args<CAP, G> a;
    a.bstart[0] = 0;
    for (int g = 0; g < G; ++g) {
        const bool on = g < count;
        const bool live = on && shards[g].n > 0;  // an empty shard's table may be NULL
        for (int k = 0; k < CAP; ++k) a.grads[g][k] = live && k < n_d ? shards[g].grads[k] : nullptr;
        for (int i = 0; i < 2; ++i) {
            a.master[g][i] = on ? shards[g].master[i] : nullptr;
            a.mq[g][i] = on ? shards[g].m_codes[i] : nullptr;
            a.vq[g][i] = on ? shards[g].v_codes[i] : nullptr;
            a.ms[g][i] = on ? shards[g].m_scale[i] : nullptr;
            a.vs[g][i] = on ? shards[g].v_scale[i] : nullptr;
        }
        a.params[g] = on ? shards[g].params : nullptr;
        a.n[g] = on ? shards[g].n : 0;
        if (on) a.bstart[g + 1] = a.bstart[g] + (a.n[g] + kA8Block - 1) / kA8Block;
    }
    for (int g = count + 1; g <= G; ++g) a.bstart[g] = a.bstart[count];
    a.n_shards = count;
    a.n_d = n_d;
    a.hp = hp;
    a.ctrl = ctrl;
    a.flag = &ctrl->overflow;
    a.commit = commit;
    a.maps = host_maps().maps;
    const bool fast = hp.math == ZS_MATH_FAST;
    // Up to 4 contributions: the staged 8-element kernel.  5-16: the direct
    // 8-element kernel, whose contribution loads already keep enough bytes in
    // flight (ragged workload, N_d = 16: 128.0 Gparams/s against 124.9 for the
    // 16-element kernel).  Above 16: the 16-element kernel.
    if constexpr (ND == 0 && CAP <= kStagedMaxNd) {
        if (width >= 1 && n_d <= kStagedMaxNd)
            return fast ? launch_a8<CAP, G, 8, ND, true, true, true>(a, stream)
                        : launch_a8<CAP, G, 8, ND, false, true, true>(a, stream);
    }
    if constexpr (ND == 0 || ND > 16) {
        if (width == 2 && n_d > 16)
            return fast ? launch_a8<CAP, G, 16, ND, true, true, false>(a, stream)
                        : launch_a8<CAP, G, 16, ND, false, true, false>(a, stream);
    }
    if (width >= 1)
        return fast ? launch_a8<CAP, G, 8, ND, true, true, false>(a, stream)
                    : launch_a8<CAP, G, 8, ND, false, true, false>(a, stream);
    return launch_a8<CAP, G, 8, ND, false, false, false>(a, stream);
}

// Shards per launch: up to kA8GroupMax with at most 64 contributions (the
// pointer tables stay within the kernel parameter space), one above.
int32_t launch_a8_group(const zs_adam8_shard* shards, int count, int32_t n_d, int width, const zs_adam& hp,
                        zs_ctrl* ctrl, zs_ctrl* commit, cudaStream_t stream) {
    switch (n_d) {
    case 16: return launch_a8_cap<16, kA8GroupMax, 16>(shards, count, n_d, width, hp, ctrl, commit, stream);
    case 32: return launch_a8_cap<32, kA8GroupMax, 32>(shards, count, n_d, width, hp, ctrl, commit, stream);
    case 64: return launch_a8_cap<64, kA8GroupMax, 64>(shards, count, n_d, width, hp, ctrl, commit, stream);
    default: break;
    }
    // a lone shard with up to 16 contributions: the one-slot kernel, whose
    // block walk needs no shard lookup (xl, N_d = 4: 203.5 Gparams/s against
    // 193.6 for the 16-slot kernel stepping one shard)
    if (n_d <= 4)
        return count == 1 ? launch_a8_cap<4, 1, 0>(shards, count, n_d, width, hp, ctrl, commit, stream)
                          : launch_a8_cap<4, kA8GroupMax, 0>(shards, count, n_d, width, hp, ctrl, commit, stream);
    if (n_d <= 16)
        return count == 1 ? launch_a8_cap<16, 1, 0>(shards, count, n_d, width, hp, ctrl, commit, stream)
                          : launch_a8_cap<16, kA8GroupMax, 0>(shards, count, n_d, width, hp, ctrl, commit, stream);
    if (n_d <= 64) return launch_a8_cap<64, kA8GroupMax, 0>(shards, count, n_d, width, hp, ctrl, commit, stream);
    return launch_a8_cap<ZS_MAX_ND, 1, 0>(shards, count, n_d, width, hp, ctrl, commit, stream);
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
    std::memcpy(mag7, h.mag7, sizeof(h.mag7));
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
    // consecutive shards of one access width (empty ones join any group): up
    // to kA8GroupMax per launch with n_d <= 64, one per launch above
    const int group_max = n_d <= 64 ? kA8GroupMax : 1;
    struct Range { int32_t first, count; };
    Range plan[ZS_MAX_SHARDS];
    int32_t np = 0, i = 0;
    while (i < n_shards) {
        if (shards[i].n == 0) { ++i; continue; }
        int32_t j = i + 1;
        while (j < n_shards && j - i < group_max && (shards[j].n == 0 || width[j] == width[i])) ++j;
        plan[np++] = Range{i, j - i};
        i = j;
    }
    // the last launch finishes the step in the control block
    for (int32_t k = 0; k < np; ++k) {
        const int32_t rc = launch_a8_group(shards + plan[k].first, plan[k].count, n_d, width[plan[k].first], *hp,
                                           ctrl_dev, k + 1 == np ? ctrl_dev : nullptr, st);
        if (rc != ZS_OK) return rc;
    }
    zs_shard ends[ZS_MAX_SHARDS];
    for (int32_t s = 0; s < n_shards; ++s) {
        // the restore pass (and the commit kernel) re-cast params from
        // master[cur] after an overflow; they read nothing else
        std::memset(&ends[s], 0, sizeof(zs_shard));
        ends[s].master[0] = shards[s].master[0];
        ends[s].master[1] = shards[s].master[1];
        ends[s].params = shards[s].params;
        ends[s].n = shards[s].n;
    }
    if (np > 0) return zs::launch_restore_pass(ends, n_shards, ctrl_dev, st, true);
    return zs::launch_commit(ends, n_shards, *hp, ctrl_dev, st);  // nothing launched: the commit kernel ends it
}

}  // extern "C"
