// cpu_step.cpp -- the shard step on the host CPU cores (ZeRO-Offload).
//
// ZeRO-Offload keeps the fp32 optimizer state on the CPU and runs the Adam
// update there with SIMD and threads ("DeepSpeed ZeRO Stages", sec. 5.1: a
// hand-tuned CPU Adam using SIMD and OpenMP; the step is elementwise, O(1) work
// per parameter, so it is memory-bound and the host's bandwidth decides).  On
// Grace-Blackwell the host is the Grace CPU, coherent with the GPU over
// NVLink-C2C.  This is the same step as the GPU kernel -- rank-order fp32 sum
// of the N_d fp16 contributions, one multiply by (float)(1 / (N_d L)), the
// non-finite test, Adam / AdamW with bias correction, the fp16 cast, ping-pong
// state with skip-on-overflow -- with every fp32 operation rounded once (the
// file is compiled with -ffp-contract=off), so it agrees with the GPU bit for
// bit.
//
// Layout for the vector units: each thread takes a contiguous chunk of the
// shard and walks it in tiles of kTile elements; per tile the contributions
// are summed contribution by contribution into a tile accumulator (the inner
// loop runs over elements, so the compiler vectorises it), then the update
// runs over the tile.  Rank order per element is kept.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <thread>
#include <vector>

#include "zs_internal.h"

namespace {

constexpr int64_t kTile = 2048;

struct CpuCoef {
    float b1, c1, b2, c2, bc1, bc2, lr, eps, wd, inv;
};

inline bool nonfinite_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof(u));
    return (u & 0x7f800000u) == 0x7f800000u;
}

inline float f16_to_f32(uint16_t h) {
    _Float16 v;
    memcpy(&v, &h, sizeof(v));
    return (float)v;
}

inline uint16_t f32_to_f16(float x) {
    const _Float16 v = (_Float16)x;  // IEEE round to nearest even
    uint16_t h;
    memcpy(&h, &v, sizeof(h));
    return h;
}

// Steps [lo, hi) of the shard; returns 1 if a reduced gradient was not finite.
int step_chunk(const zs_shard& s, int n_d, const CpuCoef& c, int cur, int64_t lo, int64_t hi) {
    float acc[kTile];
    int bad = 0;
    const float* th_in = s.master[cur];
    const float* m_in = s.m[cur];
    const float* v_in = s.v[cur];
    float* th_out = s.master[cur ^ 1];
    float* m_out = s.m[cur ^ 1];
    float* v_out = s.v[cur ^ 1];
    for (int64_t t0 = lo; t0 < hi; t0 += kTile) {
        const int64_t len = std::min(kTile, hi - t0);
        for (int64_t j = 0; j < len; ++j) acc[j] = 0.0f;
        for (int k = 0; k < n_d; ++k) {  // rank order
            const uint16_t* h = s.grads[k] + t0;
            for (int64_t j = 0; j < len; ++j) acc[j] = acc[j] + f16_to_f32(h[j]);
        }
        for (int64_t j = 0; j < len; ++j) bad |= nonfinite_bits(acc[j]) ? 1 : 0;
        for (int64_t j = 0; j < len; ++j) {
            const int64_t e = t0 + j;
            const float g = acc[j] * c.inv;
            const float m = c.b1 * m_in[e] + c.c1 * g;
            const float v = c.b2 * v_in[e] + c.c2 * (g * g);
            const float mh = m / c.bc1;
            const float vh = v / c.bc2;
            const float u = mh / (std::sqrt(vh) + c.eps);
            const float th = th_in[e];
            const float th_new = th - c.lr * (u + c.wd * th);
            m_out[e] = m;
            v_out[e] = v;
            th_out[e] = th_new;
            s.params[e] = f32_to_f16(th_new);
        }
    }
    return bad;
}

void restore_chunk(const zs_shard& s, int cur, int64_t lo, int64_t hi) {
    const float* th = s.master[cur];
    for (int64_t e = lo; e < hi; ++e) s.params[e] = f32_to_f16(th[e]);
}

template <typename F>
void parallel_chunks(int64_t n, int threads, F&& f) {
    if (threads <= 1 || n < 2 * kTile) {
        f(0, (int64_t)0, n);
        return;
    }
    std::vector<std::thread> pool;
    pool.reserve(threads);
    for (int t = 0; t < threads; ++t) {
        // chunks aligned to 16 elements so vector loads stay aligned
        const int64_t lo = (n * t / threads) & ~(int64_t)15;
        const int64_t hi = t == threads - 1 ? n : ((n * (t + 1) / threads) & ~(int64_t)15);
        pool.emplace_back([&f, t, lo, hi] { f(t, lo, hi); });
    }
    for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

ZS_API int32_t zero_shard_step_cpu(const zs_shard* shards, int32_t n_shards, int32_t n_d, const zs_adam* hp,
                                   double loss_scale, int64_t step, int32_t cur, int32_t n_threads,
                                   int32_t* overflow_out) {
    zs::NvtxRange nvtx_range("zero_shard_step_cpu");
    if (shards == nullptr || n_shards < 1 || n_shards > ZS_MAX_SHARDS || n_d < 1 || n_d > ZS_MAX_ND ||
        !zs::valid_hp(hp) || !(loss_scale > 0.0) || loss_scale > 1e300 || step < 1 || (cur != 0 && cur != 1) ||
        overflow_out == nullptr || n_threads < 0)
        return ZS_ERR_ARG;
    for (int32_t i = 0; i < n_shards; ++i) {
        const zs_shard& s = shards[i];
        if (s.n < 0) return ZS_ERR_ARG;
        if (s.qcodes != nullptr || s.qscales != nullptr) return ZS_ERR_ARG;  // no qwZ copy on the host step
        if (s.n == 0) continue;
        if (s.grads == nullptr || s.params == nullptr) return ZS_ERR_ARG;
        for (int k = 0; k < n_d; ++k)
            if (s.grads[k] == nullptr || !zs::aligned_to(s.grads[k], 2)) return ZS_ERR_ARG;
        for (int b = 0; b < 2; ++b)
            if (!s.master[b] || !s.m[b] || !s.v[b] || !zs::aligned_to(s.master[b], 4) ||
                !zs::aligned_to(s.m[b], 4) || !zs::aligned_to(s.v[b], 4))
                return ZS_ERR_ARG;
        if (!zs::aligned_to(s.params, 2)) return ZS_ERR_ALIGN;
    }
    int threads = n_threads > 0 ? n_threads : (int)std::thread::hardware_concurrency();
    if (threads < 1) threads = 1;

    // coefficients formed in double, rounded once to float (as on the GPU)
    double p1 = 1.0, p2 = 1.0;
    for (int64_t t = 0; t < step; ++t) {
        p1 *= hp->beta1;
        p2 *= hp->beta2;
    }
    CpuCoef c;
    c.b1 = (float)hp->beta1;
    c.c1 = (float)(1.0 - hp->beta1);
    c.b2 = (float)hp->beta2;
    c.c2 = (float)(1.0 - hp->beta2);
    c.bc1 = (float)(1.0 - p1);
    c.bc2 = (float)(1.0 - p2);
    c.lr = (float)hp->lr;
    c.eps = (float)hp->eps;
    c.wd = (float)hp->weight_decay;
    c.inv = (float)(1.0 / ((double)n_d * loss_scale));

    std::atomic<int> flag{0};
    for (int32_t i = 0; i < n_shards; ++i) {
        const zs_shard& s = shards[i];
        parallel_chunks(s.n, threads, [&](int, int64_t lo, int64_t hi) {
            if (step_chunk(s, n_d, c, cur, lo, hi)) flag.store(1, std::memory_order_relaxed);
        });
    }
    const int ovf = flag.load();
    if (ovf) {
        for (int32_t i = 0; i < n_shards; ++i)
            parallel_chunks(shards[i].n, threads,
                            [&](int, int64_t lo, int64_t hi) { restore_chunk(shards[i], cur, lo, hi); });
    }
    *overflow_out = ovf;
    return ZS_OK;
}

}  // extern "C"
