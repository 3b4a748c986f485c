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
//
// Every loop is a grid-stride loop over a fixed range; nothing waits.  Prints
// one line per check and exits 1 if any value differs.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <cmath>
#include <cstring>

namespace {

#include "adam8_math.cuh"

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
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("kernels");
    printf("%s\n", status == 0 ? "all equal" : "MISMATCH");
    return status;
}
