// adam8_math.cuh -- the arithmetic of the 8-bit Adam step that is not the
// fp32 Adam update: the two code maps and their nearest-code search, and the
// exact division by a divisor used many times (a per-step bias correction, a
// block's scale).  Included inside an anonymous
// namespace by adam8.cu (and by the test program that checks these functions
// exhaustively against a plain search and the IEEE division), after <cmath>,
// <cstring> and <stdint.h>.
#pragma once

constexpr int kMantBits = 7;                        // buckets per octave: 2^7
constexpr int kLowOctave = 26;                      // buckets cover [2^-26, 1]; below: bucket 0
constexpr int kBucketShift = 23 - kMantBits;
constexpr int kBucketBase = (127 - kLowOctave) << kMantBits;
constexpr int kBuckets = (kLowOctave << kMantBits) + 1;   // the last one holds 1.0

// What the kernel needs of the two code maps: the signed map's 256 code
// values (sign bit applied), the unsigned map, their decision thresholds and
// bucket tables.  Passed to the kernel by value (about 10 KB of the 32 KB
// parameter space) and copied to shared memory by each CTA.
struct Maps {
    float dec7[256];        // value of each m code: +-mag7[code & 127]
    float mag8[256];        // value of each v code
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

// ----------------------------------------------------------- device helpers ---

// Index of the map value nearest to min(a, 1) for a >= 0, ties to the
// smaller; a NaN (inf / inf, only on a step that overflowed and is dropped)
// gives 0, as a nearest search does.  Raising a to 2^-26 moves nothing across
// a threshold (the lowest is 5e-8); with the clamp to 1 it keeps the bucket
// index inside the table for every input.
__device__ __forceinline__ uint32_t nearest_code(float a, const float* thr, const uint8_t* bucket) {
    a = fminf(fmaxf(a, 0x1p-26f), 1.0f);
    const uint32_t k = bucket[(__float_as_uint(a) >> kBucketShift) - (uint32_t)kBucketBase];
    return k + (a > thr[k] ? 1u : 0u);
}

// VEC one-byte codes per thread: one 8- or 16-byte access.
template <int VEC> struct Codes;
// x / d rounded once to nearest, for a divisor d used many times (1 - beta^t
// in a step, a block's scale) with y = RN(1 / d) formed once: q = x y, then two corrections
// q <- q + (x - d q) y whose residuals the fused multiply-add forms exactly.
// After the first, q is within one ulp of x / d (a faithful quotient); then
// its residual is exact and, y being the correctly rounded reciprocal, the
// second correction yields the correctly rounded quotient (Markstein's
// theorem; P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", 1990; also Cornea, Harrison and Tang, "Scientific
// Computing on Itanium-based Systems", 2002).  For d = 1 - beta^t in (0, 1]:
// valid for x = 0 and for |x| >= 2^-100, where no quotient, product or
// residual leaves the normal range; the caller sends smaller values to the
// IEEE division.  For a block's scale, see scale_divisor_ok.
__device__ __forceinline__ float div_by_constant(float x, float d, float y) {
    float q = __fmul_rn(x, y);
    q = __fmaf_rn(__fmaf_rn(-q, d, x), y, q);
    return __fmaf_rn(__fmaf_rn(-q, d, x), y, q);
}

// Whether div_by_constant gives the codes of the IEEE quotient x / d for
// every |x| <= d when d is a block's largest magnitude (the normalization of
// m' and v' before their codes are looked up).  For d in [2^-64, 2^64]:
//   - where x / d >= 2^-27 in magnitude, 1 / d and every quotient, product
//     and residual of div_by_constant are normal floats (the residual's unit,
//     ulp(q) ulp(d) >= 2^-137, stays above the subnormal unit), so the result
//     is the correctly rounded quotient;
//   - where x / d < 2^-27, both results lie far below the lowest code
//     threshold (5e-8), so both take code 0.
// Outside that range the caller divides with __fdiv_rn.
__device__ __forceinline__ bool scale_divisor_ok(float d) { return d >= 0x1p-64f && d <= 0x1p64f; }
