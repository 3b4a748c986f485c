// Exhaustive GPU checks of the 8-bit Adam step's own arithmetic
// (csrc/adam8_math.cuh), run by tests/test_gpu_adam8_math.py:
//
//  1. nearest_code, for every float a in [0, 1] and both code maps, against an
//     independent search written here from the definition: find the two map
//     values around a (binary search over the values), then take the nearer
//     one, distances compared exactly in double, a tie going to the smaller;
//     plus values just above 1 (top code) and NaN (code 0).
//  2. div_by_constant, for every float x with 2^-100 <= |x| < 2^100 (both
//     signs) and 40 divisors d = 1 - beta^t formed as the step forms them,
//     against CUDA's IEEE division __fdiv_rn(x, d), bit for bit.
//  3. the normalization of a block by its scale: for 40 scales d with
//     scale_divisor_ok(d) (ends of the range, 1 and its neighbours, two
//     scales from the oracle's pins, 33 spread over [2^-64, 2^64]) and every
//     float x with |x| <= d (both signs), the codes of div_by_constant(x, d,
//     RN(1/d)) under both maps equal the codes of __fdiv_rn(x, d), and the two
//     quotients are equal bit for bit wherever |x / d| >= 2^-27.
//  4. the mixed-precision accumulation of a contribution (add_f16x2 in
//     csrc/step_common.cuh: PTX add.rn.f32.f16 on each half of a word) against
//     widening with __half2float and adding with __fadd_rn, bit for bit (NaN
//     against NaN), for every fp16 value in both halves and 4096 fp32
//     accumulators (zeros of both signs, fp16 extremes, subnormals, values
//     near the fp16 range and spread over the fp32 range).
//
// Every loop is a grid-stride loop over a fixed range; nothing waits.  Prints
// one line per check and exits 1 if any value differs.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <cmath>
#include <cstring>

#include "zero_shard.h"

namespace {

#include "adam8_math.cuh"
#include "step_common.cuh"

struct Result {
    unsigned long long bad;
    unsigned long long first;  // smallest bit pattern that differed
};

__global__ void nearest_check(const float* values, const float* thr, const uint8_t* bucket, int count, uint32_t lo,
                              uint32_t hi, Result* out) {
    __shared__ float s_val[256], s_thr[256];
    __shared__ uint8_t s_bucket[kBuckets];
    for (int i = threadIdx.x; i < count; i += blockDim.x) {
        s_val[i] = values[i];
        s_thr[i] = thr[i];
    }
    for (int i = threadIdx.x; i < kBuckets; i += blockDim.x) s_bucket[i] = bucket[i];
    __syncthreads();
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t b = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b <= hi; b += stride) {
        const float a = __uint_as_float((uint32_t)b);
        const uint32_t got = nearest_code(a, s_thr, s_bucket);
        // the map values around a: largest k with values[k] <= a
        int l = 0, h = count - 1;
        while (l < h) {
            const int mid = (l + h + 1) / 2;
            if (s_val[mid] <= a) l = mid; else h = mid - 1;
        }
        uint32_t want = (uint32_t)l;
        if (l + 1 < count) {
            const double below = (double)a - (double)s_val[l];
            const double above = (double)s_val[l + 1] - (double)a;
            if (above < below) want = (uint32_t)(l + 1);
        }
        if (got != want) {
            atomicAdd(&out->bad, 1ull);
            atomicMin(&out->first, (unsigned long long)b);
        }
    }
}

__global__ void div_check(float d, uint32_t lo, uint32_t hi, Result* out) {
    const float y = __frcp_rn(d);
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t b = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b < hi; b += stride) {
        const float x = __uint_as_float((uint32_t)b);
        const float q1 = div_by_constant(x, d, y), r1 = __fdiv_rn(x, d);
        const float q2 = div_by_constant(-x, d, y), r2 = __fdiv_rn(-x, d);
        if (__float_as_uint(q1) != __float_as_uint(r1) || __float_as_uint(q2) != __float_as_uint(r2)) {
            atomicAdd(&out->bad, 1ull);
            atomicMin(&out->first, (unsigned long long)b);
        }
    }
}

// the sign-and-magnitude code of the signed map, as the step forms it
__device__ __forceinline__ uint32_t signed_code(float x, const float* thr, const uint8_t* bucket) {
    const uint32_t k = nearest_code(fabsf(x), thr, bucket);
    return (x < 0.0f && k > 0u) ? (k | 0x80u) : k;
}

__global__ void scale_check(float d, const float* thr7, const uint8_t* b7, const float* thr8, const uint8_t* b8,
                            Result* out) {
    __shared__ float s_thr7[128], s_thr8[256];
    __shared__ uint8_t s_b7[kBuckets], s_b8[kBuckets];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) {
        if (i < 128) s_thr7[i] = thr7[i];
        s_thr8[i] = thr8[i];
    }
    for (int i = threadIdx.x; i < kBuckets; i += blockDim.x) {
        s_b7[i] = b7[i];
        s_b8[i] = b8[i];
    }
    __syncthreads();
    const float y = __frcp_rn(d);
    const uint64_t hi = __float_as_uint(d);  // every float in [0, d]
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t b = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b <= hi; b += stride) {
        const float x = __uint_as_float((uint32_t)b);
        bool bad = false;
        for (int sgn = 0; sgn < 2; ++sgn) {
            const float xs = sgn ? -x : x;
            const float q = div_by_constant(xs, d, y), r = __fdiv_rn(xs, d);
            if (fabsf(r) >= 0x1p-27f && __float_as_uint(q) != __float_as_uint(r)) bad = true;
            if (signed_code(q, s_thr7, s_b7) != signed_code(r, s_thr7, s_b7)) bad = true;
            if (nearest_code(fabsf(q), s_thr8, s_b8) != nearest_code(fabsf(r), s_thr8, s_b8)) bad = true;
        }
        if (bad) {
            atomicAdd(&out->bad, 1ull);
            atomicMin(&out->first, (unsigned long long)b);
        }
    }
}

__global__ void mixed_add_check(const float* accs, int na, Result* out) {
    const uint32_t hb = blockIdx.x * blockDim.x + threadIdx.x;  // every fp16 bit pattern
    if (hb > 0xffffu) return;
    unsigned long long bad = 0;
    for (int i = 0; i < na; ++i) {
        float a0 = accs[i], a1 = accs[(i + 7) % na];
        const uint32_t h1 = hb ^ 0x8000u;  // the other sign in the high half
        const float r0 = __fadd_rn(a0, __half2float(__ushort_as_half((unsigned short)hb)));
        const float r1 = __fadd_rn(a1, __half2float(__ushort_as_half((unsigned short)h1)));
        add_f16x2(hb | (h1 << 16), a0, a1);
        const bool nan0 = r0 != r0 && a0 != a0, nan1 = r1 != r1 && a1 != a1;
        if ((__float_as_uint(a0) != __float_as_uint(r0) && !nan0) || (__float_as_uint(a1) != __float_as_uint(r1) && !nan1))
            ++bad;
    }
    if (bad) {
        atomicAdd(&out->bad, bad);
        atomicMin(&out->first, (unsigned long long)hb);
    }
}

}  // namespace

static int fail(const char* what) {
    printf("CUDA error: %s: %s\n", what, cudaGetErrorString(cudaGetLastError()));
    return 2;
}

int main() {
    // the tables, built by the library's host code
    float mag7[128], mag8[256], thr7[128], thr8[256];
    static uint8_t b7[kBuckets], b8[kBuckets];
    for (int k = 0; k < 128; ++k) mag7[k] = map_value(k, 7);
    for (int k = 0; k < 256; ++k) mag8[k] = map_value(k, 8);
    if (!build_search(mag7, 128, thr7, b7) || !build_search(mag8, 256, thr8, b8)) {
        printf("bucket table: a bucket holds two thresholds\n");
        return 1;
    }
    float *d_val, *d_thr;
    uint8_t* d_bucket;
    Result* d_res;
    if (cudaMalloc(&d_val, 256 * 4) || cudaMalloc(&d_thr, 256 * 4) || cudaMalloc(&d_bucket, kBuckets) ||
        cudaMalloc(&d_res, sizeof(Result)))
        return fail("cudaMalloc");
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    const int blocks = sms * 8, threads = 256;
    int status = 0;
    auto run = [&](const char* name, auto launch) {
        const Result zero{0ull, ~0ull};
        cudaMemcpy(d_res, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        launch();
        Result r;
        if (cudaMemcpy(&r, d_res, sizeof(r), cudaMemcpyDeviceToHost) != cudaSuccess) {
            status = fail(name);
            return;
        }
        printf("%s: %llu mismatches%s", name, r.bad, r.bad ? "" : "\n");
        if (r.bad) {
            printf(" (first at bit pattern 0x%08llx)\n", r.first);
            status = 1;
        }
    };
    const uint32_t one = 0x3f800000u;
    for (int map = 0; map < 2; ++map) {
        const int count = map == 0 ? 128 : 256;
        cudaMemcpy(d_val, map == 0 ? mag7 : mag8, count * 4, cudaMemcpyHostToDevice);
        cudaMemcpy(d_thr, map == 0 ? thr7 : thr8, count * 4, cudaMemcpyHostToDevice);
        cudaMemcpy(d_bucket, map == 0 ? b7 : b8, kBuckets, cudaMemcpyHostToDevice);
        char name[96];
        snprintf(name, sizeof(name), "nearest_code, %s map, every float in [0, 1]", map == 0 ? "signed" : "unsigned");
        run(name, [&] { nearest_check<<<blocks, threads>>>(d_val, d_thr, d_bucket, count, 0u, one, d_res); });
        snprintf(name, sizeof(name), "nearest_code, %s map, 1 < a < 1.0078 (top code)", map == 0 ? "signed" : "unsigned");
        run(name, [&] { nearest_check<<<blocks, threads>>>(d_val, d_thr, d_bucket, count, one + 1, one + 65535, d_res); });
    }
    // divisors as the step forms them: p = beta^t by repeated double
    // multiplication, d = (float)(1 - p)
    const double betas[] = {0.9, 0.95, 0.99, 0.999, 0.9999};
    const int ts[] = {1, 2, 3, 5, 10, 100, 1000, 10000};
    const uint32_t lo = (uint32_t)(127 - 100) << 23, hi = (uint32_t)(127 + 100) << 23;
    for (double beta : betas)
        for (int t : ts) {
            double p = 1.0;
            for (int i = 0; i < t; ++i) p *= beta;
            const float d = (float)(1.0 - p);
            char name[96];
            snprintf(name, sizeof(name), "div_by_constant, d = 1 - %g^%d = %.9g, 2^-100 <= |x| < 2^100", beta, t, d);
            run(name, [&] { div_check<<<blocks, threads>>>(d, lo, hi, d_res); });
        }
    // block scales: the range ends, 1 and its neighbours, two scales of the
    // oracle's normalization pins, and 33 spread over the range with
    // mantissas from a fixed linear congruential sequence
    float *d_thr7, *d_thr8;
    uint8_t *d_b7, *d_b8;
    if (cudaMalloc(&d_thr7, 128 * 4) || cudaMalloc(&d_thr8, 256 * 4) || cudaMalloc(&d_b7, kBuckets) ||
        cudaMalloc(&d_b8, kBuckets))
        return fail("cudaMalloc");
    cudaMemcpy(d_thr7, thr7, 128 * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(d_thr8, thr8, 256 * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(d_b7, b7, kBuckets, cudaMemcpyHostToDevice);
    cudaMemcpy(d_b8, b8, kBuckets, cudaMemcpyHostToDevice);
    uint32_t scales[40] = {(127u - 64u) << 23, (127u + 64u) << 23, 0x3f800000u, 0x3f800001u, 0x3f7fffffu,
                           0x3c0185d6u, 0x35f0cc4du};
    uint32_t lcg = 12345u;
    for (int i = 7; i < 40; ++i) {
        lcg = lcg * 1664525u + 1013904223u;
        const uint32_t e = (uint32_t)(127 - 64 + (i - 7) * 127 / 32);   // exponents -64 .. 63
        scales[i] = (e << 23) | (lcg >> 9);
    }
    for (uint32_t bits : scales) {
        float d;
        std::memcpy(&d, &bits, 4);
        char name[96];
        snprintf(name, sizeof(name), "block quotient, scale 0x%08x = %.9g, every |x| <= scale", bits, d);
        run(name, [&] { scale_check<<<blocks, threads>>>(d, d_thr7, d_b7, d_thr8, d_b8, d_res); });
    }
    // accumulators for the mixed add: special values, then a fixed linear
    // congruential sequence (every fourth near the fp16 range)
    {
        constexpr int na = 4096;
        static float accs[na];
        const float special[] = {0.0f, -0.0f, 1.0f, -1.0f, 65504.0f, -65504.0f, 1e-8f, -1e-8f, 3.0e38f, 1e-40f,
                                 -1e-40f, 5.96e-8f, 0.5f};
        int k = 0;
        for (float v : special) accs[k++] = v;
        uint32_t r = 12345u;
        for (; k < na; ++k) {
            r = r * 1664525u + 1013904223u;
            uint32_t bits = r;
            if ((k & 3) == 0) bits = (bits & 0x80FFFFFFu) | (((112u + (r >> 27)) & 0xFFu) << 23);
            float f;
            std::memcpy(&f, &bits, 4);
            if (!std::isfinite(f)) f = 1.0f;
            accs[k] = f;
        }
        float* d_accs;
        if (cudaMalloc(&d_accs, sizeof(accs))) return fail("cudaMalloc");
        cudaMemcpy(d_accs, accs, sizeof(accs), cudaMemcpyHostToDevice);
        run("mixed-precision add, every fp16 value x 4096 accumulators",
            [&] { mixed_add_check<<<256, 256>>>(d_accs, na, d_res); });
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("kernels");
    printf("%s\n", status == 0 ? "all equal" : "MISMATCH");
    return status;
}
