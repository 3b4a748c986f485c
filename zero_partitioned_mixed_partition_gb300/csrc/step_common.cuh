// step_common.cuh -- device code shared by the kernels of libzeroshard.so:
// the step coefficients, the element update and the vector memory accesses.
// Each CUDA translation unit includes it inside its anonymous namespace, after
// <cuda_fp16.h>, <stdint.h> and zero_shard.h.
#pragma once

// ------------------------------------------------------------ index checks ---

// Debug build (compiled with ZS_CHECKED=1, libzeroshard_checked.so): before an
// access of `count` elements starting at element `first`, ZS_RANGE_OK tests
// 0 <= first and first + count <= limit, the extent the call was given (the
// shard's n, or its qwZ block count).  A failed test records
// (site << 48) | first in this translation unit's fault word -- the first
// failure wins -- and the caller skips the access; nothing traps or asserts.
// In the ordinary build ZS_RANGE_OK is the constant true.
constexpr uint32_t kSiteStep = 1, kSiteQwzFused = 2, kSiteCast = 3, kSiteQwz = 4, kSiteDequant = 5,
                   kSiteNorm = 6, kSiteClipped = 7, kSiteSgd = 8, kSiteScale = 9;

#if ZS_CHECKED
__device__ unsigned long long g_fault;

__device__ __forceinline__ bool zs_range_ok(uint32_t site, int64_t first, int64_t count, int64_t limit) {
    if (first >= 0 && count >= 0 && first + count <= limit) return true;
    atomicCAS(&g_fault, 0ull, ((unsigned long long)site << 48) | ((unsigned long long)first & 0xffffffffffffull));
    return false;
}
#define ZS_RANGE_OK(site, first, count, limit) zs_range_ok((site), (first), (count), (limit))

// The recorded failure (0: none), cleared; synchronises the device.
uint64_t take_fault() {
    unsigned long long v = 0, zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return ~0ull;
    if (cudaMemcpyFromSymbol(&v, g_fault, sizeof(v)) != cudaSuccess) return ~0ull;
    if (cudaMemcpyToSymbol(g_fault, &zero, sizeof(zero)) != cudaSuccess) return ~0ull;
    return v;
}
#else
#define ZS_RANGE_OK(site, first, count, limit) true
uint64_t take_fault() { return 0; }
#endif

// ------------------------------------------------------------ coefficients ---

// Scalar coefficients of one step, each formed in double and rounded once to
// float, so host and device agree bit for bit.
struct Coef {
    float b1, c1, b2, c2;  // beta1, 1 - beta1, beta2, 1 - beta2
    float bc1, bc2;        // 1 - beta1^t, 1 - beta2^t
    float lr, eps, wd;
    float inv;             // 1 / (N_d L)
};

Coef coef_host(const zs_adam& hp, double p1, double p2, int n_d, double loss_scale) {
    Coef c;
    c.b1 = (float)hp.beta1;
    c.c1 = (float)(1.0 - hp.beta1);
    c.b2 = (float)hp.beta2;
    c.c2 = (float)(1.0 - hp.beta2);
    c.bc1 = (float)(1.0 - p1);
    c.bc2 = (float)(1.0 - p2);
    c.lr = (float)hp.lr;
    c.eps = (float)hp.eps;
    c.wd = (float)hp.weight_decay;
    c.inv = (float)(1.0 / ((double)n_d * loss_scale));
    return c;
}

__device__ Coef coef_device(const zs_adam& hp, double p1, double p2, int n_d, double loss_scale) {
    Coef c;
    c.b1 = __double2float_rn(hp.beta1);
    c.c1 = __double2float_rn(__dsub_rn(1.0, hp.beta1));
    c.b2 = __double2float_rn(hp.beta2);
    c.c2 = __double2float_rn(__dsub_rn(1.0, hp.beta2));
    c.bc1 = __double2float_rn(__dsub_rn(1.0, p1));
    c.bc2 = __double2float_rn(__dsub_rn(1.0, p2));
    c.lr = __double2float_rn(hp.lr);
    c.eps = __double2float_rn(hp.eps);
    c.wd = __double2float_rn(hp.weight_decay);
    c.inv = __double2float_rn(__ddiv_rn(1.0, __dmul_rn((double)n_d, loss_scale)));
    return c;
}

// ------------------------------------------------------------ element math ---

__device__ __forceinline__ bool nonfinite(float x) {
    return (__float_as_uint(x) & 0x7f800000u) == 0x7f800000u;
}

// a / b for ZS_MATH_FAST: the hardware reciprocal estimate y ~ 1/b (PTX
// rcp.approx, at most 1 ulp off), the quotient q0 = a * y, and one residual
// correction q0 + (a - b q0) y with the residual formed exactly by a fused
// multiply-add (the Newton-Raphson / Markstein correction step of FMA-based
// division).  The result is within 1 ulp of a / b and equals the correctly
// rounded quotient except when a / b lies extremely close to a rounding
// midpoint.  b = sqrt(vh) + eps >= eps > 0 here.
__device__ __forceinline__ float div_corrected(float a, float b) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(b));
    const float q0 = __fmul_rn(a, y);
    const float r = __fmaf_rn(-q0, b, a);
    return __fmaf_rn(r, y, q0);
}

// One Adam / AdamW update of one coordinate from its reduced gradient g.
// FAST (ZS_MATH_FAST) forms u with div_corrected instead of the IEEE divide;
// everything else, m and v included, is the same in both modes.
template <bool FAST>
__device__ __forceinline__ void adam_apply(const Coef& c, float g, float& th, float& m, float& v) {
    m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.c1, g));
    v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.c2, __fmul_rn(g, g)));
    const float mh = __fdiv_rn(m, c.bc1);
    const float vh = __fdiv_rn(v, c.bc2);
    const float den = __fadd_rn(__fsqrt_rn(vh), c.eps);
    const float u = FAST ? div_corrected(mh, den) : __fdiv_rn(mh, den);
    th = __fsub_rn(th, __fmul_rn(c.lr, __fadd_rn(u, __fmul_rn(c.wd, th))));
}

// The same from the summed contributions gs: g = gs * (float)(1 / (N_d L)).
template <bool FAST>
__device__ __forceinline__ void adam_update(const Coef& c, float gs, float& th, float& m, float& v) {
    adam_apply<FAST>(c, __fmul_rn(gs, c.inv), th, m, v);
}

// --------------------------------------------------------- vector memory ---

// How a thread moves its VEC consecutive elements per loop iteration.
//   Mem<8>   "narrow": one 16-byte fp16 access per contribution, two 16-byte
//            fp32 accesses per state array, all with evict-first (.cs) hints.
//            Needs 16-byte aligned buffers.  Best measured layout for small
//            N_d (N_d <= 4: 6.65 TB/s on a 375M-param shard).
//   Mem<16>  "wide": two 16-byte fp16 accesses per contribution and one
//            256-bit (v8) fp32 access per 8 state values, default caching.
//            Twice the contribution bytes in flight per thread, which large
//            N_d needs (N_d = 64: 7.06 TB/s vs 4.98 TB/s narrow).  Needs
//            32-byte aligned fp32 buffers and 16-byte aligned fp16 buffers.
//   Mem<1>   scalar, any naturally aligned buffer.
template <int VEC> struct Mem;

template <> struct Mem<8> {
    // the 8 fp16 values as raw words (two per word, the lower address in the low half)
    static __device__ __forceinline__ void load_h_words(const uint16_t* p, uint32_t* w) {
        const uint4 r = __ldcs(reinterpret_cast<const uint4*>(p));
        w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
    }
    static __device__ __forceinline__ void load_h(const uint16_t* p, float* out) {
        const uint4 r = __ldcs(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void load_f(const float* p, float* out) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
        const float4 b = __ldcs(reinterpret_cast<const float4*>(p + 4));
        out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
        out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    }
    static __device__ __forceinline__ void store_f(float* p, const float* in) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(in[0], in[1], in[2], in[3]));
        __stcs(reinterpret_cast<float4*>(p + 4), make_float4(in[4], in[5], in[6], in[7]));
    }
    static __device__ __forceinline__ void store_h(uint16_t* p, const float* in) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h = __floats2half2_rn(in[2 * i], in[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        __stcs(reinterpret_cast<uint4*>(p), make_uint4(w[0], w[1], w[2], w[3]));
    }
};

template <> struct Mem<16> {
    static __device__ __forceinline__ void load_h_words(const uint16_t* p, uint32_t* w) {
        const uint4 a = *reinterpret_cast<const uint4*>(p);
        const uint4 b = *reinterpret_cast<const uint4*>(p + 8);
        w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
        w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    }
    static __device__ __forceinline__ void load_h8(const uint16_t* p, float* out) {
        const uint4 r = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
            out[2 * i] = f.x;
            out[2 * i + 1] = f.y;
        }
    }
    static __device__ __forceinline__ void load_h(const uint16_t* p, float* out) {
        load_h8(p, out);
        load_h8(p + 8, out + 8);
    }
    static __device__ __forceinline__ void load_f8(const float* p, float* o) {
        asm volatile("ld.global.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=f"(o[0]), "=f"(o[1]), "=f"(o[2]), "=f"(o[3]), "=f"(o[4]), "=f"(o[5]), "=f"(o[6]),
                       "=f"(o[7])
                     : "l"(p));
    }
    static __device__ __forceinline__ void load_f(const float* p, float* out) {
        load_f8(p, out);
        load_f8(p + 8, out + 8);
    }
    static __device__ __forceinline__ void store_f8(float* p, const float* v) {
        asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                     :: "l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
                        "f"(v[7])
                     : "memory");
    }
    static __device__ __forceinline__ void store_f(float* p, const float* in) {
        store_f8(p, in);
        store_f8(p + 8, in + 8);
    }
    static __device__ __forceinline__ void store_h(uint16_t* p, const float* in) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const __half2 h = __floats2half2_rn(in[2 * i], in[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(p + 8) = make_uint4(w[4], w[5], w[6], w[7]);
    }
};

template <> struct Mem<1> {
    static __device__ __forceinline__ void load_h(const uint16_t* p, float* out) {
        out[0] = __half2float(__ushort_as_half(__ldcs(reinterpret_cast<const unsigned short*>(p))));
    }
    static __device__ __forceinline__ void load_f(const float* p, float* out) { out[0] = __ldcs(p); }
    static __device__ __forceinline__ void store_f(float* p, const float* in) { __stcs(p, in[0]); }
    static __device__ __forceinline__ void store_h(uint16_t* p, const float* in) {
        __stcs(reinterpret_cast<unsigned short*>(p), __half_as_ushort(__float2half_rn(in[0])));
    }
};

// acc0 += fp16 value in the low half of w, acc1 += the one in the high half,
// each as one mixed-precision add (PTX add.rn.f32.f16, sm_100 and later): the
// fp16 operand is widened exactly and the sum rounded once to fp32, the
// result of widening first and adding with __fadd_rn, without the separate
// conversion instruction.
__device__ __forceinline__ void add_f16x2(uint32_t w, float& acc0, float& acc1) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(w));
}
__device__ __forceinline__ void add_f16(uint16_t h, float& acc) {
    asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(acc) : "h"(h));
}

// Unroll of the contribution loop when N_d is a compile-time constant above 16.
constexpr int kUnrollLargeNd = 8;

// Sum of the N_d contributions of VEC consecutive elements, in rank order.
// MIXED: each contribution added by the mixed-precision add (add_f16x2), the
// same sums; the issue-bound 8-bit Adam kernel takes it (+1.5 % on the 1.5B
// shard), the HBM-bound kernels do not (the fp32 step measured 9-11 % slower
// with it at N_d = 4 and 64).
// ND > 0: exactly ND contributions, known at compile time (fully unrolled for
// ND <= 16, unrolled by kUnrollLargeNd above); ND == 0: p.n_d of them (<= CAP),
// unrolled by 4.
template <int CAP, int VEC, int ND, bool MIXED = false>
__device__ __forceinline__ void sum_contributions(const uint16_t* const (&grads)[CAP], int n_d, int64_t e,
                                                  float* acc) {
    auto add = [&](int k) {
        if constexpr (MIXED && VEC == 1) {
            add_f16(__ldcs(reinterpret_cast<const unsigned short*>(grads[k] + e)), acc[0]);
        } else if constexpr (MIXED) {
            uint32_t w[VEC / 2];
            Mem<VEC>::load_h_words(grads[k] + e, w);
#pragma unroll
            for (int j = 0; j < VEC / 2; ++j) add_f16x2(w[j], acc[2 * j], acc[2 * j + 1]);
        } else {
            float h[VEC];
            Mem<VEC>::load_h(grads[k] + e, h);
#pragma unroll
            for (int j = 0; j < VEC; ++j) acc[j] = __fadd_rn(acc[j], h[j]);
        }
    };
    if constexpr (ND > 0 && ND <= 16) {
#pragma unroll
        for (int k = 0; k < ND; ++k) add(k);
    } else if constexpr (ND > 16) {
#pragma unroll kUnrollLargeNd
        for (int k = 0; k < ND; ++k) add(k);
    } else {
#pragma unroll 4
        for (int k = 0; k < n_d; ++k) add(k);
    }
}


// ------------------------------------------------ quantized weights (qwZ) ---

// Parameters per quantization block of the int8 copy of the fp16 shard.
constexpr int kQwzBlock = ZS_QWZ_BLOCK;

// x / s rounded once, for the codes of the 16-element layout: with the
// correctly rounded reciprocal y = 1/s, q0 = x y and one exact-residual
// correction q0 + (x - s q0) y (Markstein's theorem: the result is the
// correctly rounded quotient when y is, and nothing under- or overflows).
// Checked exhaustively on the domain it serves -- every fp16 x with |x| <= a
// against every positive finite fp16 block maximum a, s = fp32(a / 127):
// 1,007,713,278 pairs, all equal to the IEEE quotient.  Cheaper than a
// divide per element in the 16-element kernels (+2.4 % on the ragged
// workload's qwZ step, +6.5 % at N_d = 8); the 8-element kernel measured
// faster with the IEEE divide and keeps it.
__device__ __forceinline__ float div_by_scale(float x, float s, float y) {
    const float q0 = __fmul_rn(x, y);
    return __fmaf_rn(__fmaf_rn(-q0, s, x), y, q0);
}

// One quantization block held by an aligned group of G lanes, V consecutive
// values per lane (G * V == kQwzBlock): the block's scale max|x| / 127 and this
// lane's V codes rint(x / scale), ties to even, all in fp32.  Lanes past the
// data pass valid = 0.  Every lane of the warp must call it (it shuffles).
template <int V, int G>
__device__ __forceinline__ float qwz_group_codes(const float* x, int valid, int8_t* q) {
    static_assert(V * G == kQwzBlock, "a group holds one block");
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < V; ++j)
        if (j < valid) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(amax, 127.0f);
    if constexpr (V == 16) {
        const float y = scale > 0.0f ? __frcp_rn(scale) : 0.0f;
#pragma unroll
        for (int j = 0; j < V; ++j) {
            float r = scale > 0.0f ? rintf(div_by_scale(x[j], scale, y)) : 0.0f;
            r = fminf(fmaxf(r, -127.0f), 127.0f);
            q[j] = (int8_t)(int)r;
        }
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j) {
            float r = scale > 0.0f ? rintf(__fdiv_rn(x[j], scale)) : 0.0f;
            r = fminf(fmaxf(r, -127.0f), 127.0f);
            q[j] = (int8_t)(int)r;
        }
    }
    return scale;
}

// Packs V int8 codes (V = 8 or 16) and stores them with one 8- or 16-byte access.
template <int V>
__device__ __forceinline__ void store_codes(int8_t* dst, const int8_t* q) {
    uint32_t w[V / 4];
#pragma unroll
    for (int k = 0; k < V / 4; ++k)
        w[k] = (uint32_t)(uint8_t)q[4 * k] | ((uint32_t)(uint8_t)q[4 * k + 1] << 8) |
               ((uint32_t)(uint8_t)q[4 * k + 2] << 16) | ((uint32_t)(uint8_t)q[4 * k + 3] << 24);
    if constexpr (V == 8) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    } else {
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// fp16 rounding of a float, back in float: the value the fp16 shard holds.
__device__ __forceinline__ float as_fp16_value(float x) { return __half2float(__float2half_rn(x)); }
