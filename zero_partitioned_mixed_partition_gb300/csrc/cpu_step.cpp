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
// runs over the tile.  Rank order per element is kept.  The step is bound by
// how fast one core streams its eleven arrays (with every division and the
// square root replaced by multiplies it ran only 4 % faster on 16 Grace
// cores), and longer runs per array stream faster: 65,536-element tiles (the
// accumulator, 256 KB, stays in the core's L2) measured 5.34-5.49 Gparams/s
// on 16 Grace cores against 4.80-4.85 with 2,048-element tiles.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <memory>
#include <thread>
#include <vector>

#include "zs_internal.h"

#if defined(__aarch64__)
#include <arm_neon.h>
#endif

namespace {

constexpr int64_t kTile = 65536;
constexpr int64_t kMinThreadChunk = 2048;  // below 2 x this many elements one thread steps them all

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


// fp16 of len floats, round to nearest even.  On aarch64 four at a time with
// the NEON narrowing conversion (the same IEEE rounding as the scalar
// conversion, under the default FPCR mode), which the compiler does not
// generate from the scalar loop for the baseline architecture; elsewhere the
// scalar loop.
inline void cast_tile(const float* src, _Float16* dst, int64_t len) {
    int64_t j = 0;
#if defined(__aarch64__)
    for (; j + 4 <= len; j += 4) vst1_f16(reinterpret_cast<float16_t*>(dst + j), vcvt_f16_f32(vld1q_f32(src + j)));
#endif
    for (; j < len; ++j) dst[j] = (_Float16)src[j];  // IEEE round to nearest even
}

// The Adam update of one tile of len elements from its reduced gradient
// sums acc: the element loop of step_chunk.  The buffers are declared
// non-overlapping (restrict) so the compiler vectorizes the loop without
// run-time overlap checks (seven arrays are more pairs than it checks);
// step_chunk takes the restrict form only when the state sets are distinct
// buffers, and the same loop without the promise for in-place state.  fp16
// parameters are written through a _Float16 view.
template <bool RESTRICT>
struct TilePtrs;
template <>
struct TilePtrs<true> {
    using CF = const float* __restrict__;
    using F = float* __restrict__;
    using H = _Float16* __restrict__;
};
template <>
struct TilePtrs<false> {
    using CF = const float*;
    using F = float*;
    using H = _Float16*;
};

template <bool RESTRICT>
void update_tile(typename TilePtrs<RESTRICT>::CF acc, typename TilePtrs<RESTRICT>::CF th_in,
                 typename TilePtrs<RESTRICT>::CF m_in, typename TilePtrs<RESTRICT>::CF v_in,
                 typename TilePtrs<RESTRICT>::F th_out, typename TilePtrs<RESTRICT>::F m_out,
                 typename TilePtrs<RESTRICT>::F v_out, typename TilePtrs<RESTRICT>::H params, int64_t len,
                 const CpuCoef cf) {
    const float inv = cf.inv, b1 = cf.b1, c1 = cf.c1, b2 = cf.b2, c2 = cf.c2, bc1 = cf.bc1, bc2 = cf.bc2;
    const float eps = cf.eps, lr = cf.lr, wd = cf.wd;
    for (int64_t j = 0; j < len; ++j) {
        const float g = acc[j] * inv;
        const float m = b1 * m_in[j] + c1 * g;
        const float v = b2 * v_in[j] + c2 * (g * g);
        const float mh = m / bc1;
        const float vh = v / bc2;
        const float u = mh / (std::sqrt(vh) + eps);
        const float th = th_in[j];
        const float th_new = th - lr * (u + wd * th);
        m_out[j] = m;
        v_out[j] = v;
        th_out[j] = th_new;
    }
    // the fp16 cast in a loop of its own (the tile is still in L1), so the
    // update loop above vectorizes even where fp16 has no vector type
    cast_tile(th_out, params, len);
}

// Steps [lo, hi) of the shard; returns 1 if a reduced gradient was not finite.
int step_chunk(const zs_shard& s, int n_d, const CpuCoef& c, int cur, int64_t lo, int64_t hi) {
    std::unique_ptr<float[]> accbuf(new float[(size_t)std::max<int64_t>(1, std::min(kTile, hi - lo))]);
    float* acc = accbuf.get();
    int bad = 0;
    const float* th_in = s.master[cur];
    const float* m_in = s.m[cur];
    const float* v_in = s.v[cur];
    float* th_out = s.master[cur ^ 1];
    float* m_out = s.m[cur ^ 1];
    float* v_out = s.v[cur ^ 1];
    // the two state sets are separate buffers (the usual ping-pong): the
    // update loop may assume no overlap
    const bool distinct = th_in != th_out && m_in != m_out && v_in != v_out;
    for (int64_t t0 = lo; t0 < hi; t0 += kTile) {
        const int64_t len = std::min(kTile, hi - t0);
        for (int64_t j = 0; j < len; ++j) acc[j] = 0.0f;
        for (int k = 0; k < n_d; ++k) {  // rank order
            const uint16_t* h = s.grads[k] + t0;
            for (int64_t j = 0; j < len; ++j) acc[j] = acc[j] + f16_to_f32(h[j]);
        }
        for (int64_t j = 0; j < len; ++j) bad |= nonfinite_bits(acc[j]) ? 1 : 0;
        _Float16* ph = reinterpret_cast<_Float16*>(s.params + t0);
        if (distinct)
            update_tile<true>(acc, th_in + t0, m_in + t0, v_in + t0, th_out + t0, m_out + t0, v_out + t0, ph, len, c);
        else
            update_tile<false>(acc, th_in + t0, m_in + t0, v_in + t0, th_out + t0, m_out + t0, v_out + t0, ph, len,
                               c);
    }
    return bad;
}

void restore_chunk(const zs_shard& s, int cur, int64_t lo, int64_t hi) {
    cast_tile(s.master[cur] + lo, reinterpret_cast<_Float16*>(s.params + lo), hi - lo);
}

template <typename F>
void parallel_chunks(int64_t n, int threads, F&& f) {
    if (threads <= 1 || n < 2 * kMinThreadChunk) {
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

CpuCoef cpu_coef(const zs_adam* hp, double loss_scale, int64_t step, int32_t n_d) {
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
    return c;
}

bool pinned_host(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
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
    const CpuCoef c = cpu_coef(hp, loss_scale, step, n_d);

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

// ZeRO-Offload step with its transfers: the gradient contributions leave the
// GPU, the host cores run the step on the host-resident fp32 state, the new
// fp16 parameters return to the GPU.  The shard is cut into chunks; all the
// device-to-host copies are enqueued at once on d2h_stream (one
// cudaMemcpyAsync per contribution and chunk, each chunk followed by an
// event), and the worker threads step chunk c as soon as its event has
// completed, each thread its own contiguous part of the chunk, while later
// chunks are still in flight.  The thread that finishes the last part of a
// chunk enqueues that chunk's host-to-device copy of the fp16 parameters on
// h2d_stream, so the two directions of the link and the host arithmetic
// overlap.  The arithmetic per element is step_chunk's (the same as the GPU
// kernel and zero_shard_step_cpu, bit for bit).  After an overflow the fp16
// staging buffer is rewritten from the kept master weights and copied to the
// device again, so on return the device slice matches the committed state.
ZS_API int32_t zero_shard_step_offload(const zs_offload_shard* o, int32_t n_d, const zs_adam* hp,
                                       double loss_scale, int64_t step, int32_t cur, int32_t n_threads,
                                       int64_t chunk, void* d2h_stream, void* h2d_stream,
                                       int32_t* overflow_out) {
    zs::NvtxRange nvtx_range("zero_shard_step_offload");
    if (o == nullptr || n_d < 1 || n_d > ZS_MAX_ND || !zs::valid_hp(hp) || !(loss_scale > 0.0) ||
        loss_scale > 1e300 || step < 1 || (cur != 0 && cur != 1) || overflow_out == nullptr || n_threads < 0 ||
        chunk < 0 || chunk % 16 != 0 || o->n < 0)
        return ZS_ERR_ARG;
    const int64_t n = o->n;
    if (n > 0) {
        if (o->grads_dev == nullptr || o->grads_host == nullptr || o->params_dev == nullptr ||
            o->params_host == nullptr)
            return ZS_ERR_ARG;
        for (int k = 0; k < n_d; ++k) {
            if (o->grads_dev[k] == nullptr || o->grads_host[k] == nullptr) return ZS_ERR_ARG;
            if (!zs::aligned_to(o->grads_dev[k], 2) || !zs::aligned_to(o->grads_host[k], 2)) return ZS_ERR_ALIGN;
            if (!pinned_host(o->grads_host[k]))
                return zs::fail_with(ZS_ERR_ARG, "zero_shard_step_offload: grads_host[k] is not page-locked");
        }
        if (!zs::aligned_to(o->params_dev, 2) || !zs::aligned_to(o->params_host, 2)) return ZS_ERR_ALIGN;
        if (!pinned_host(o->params_host))
            return zs::fail_with(ZS_ERR_ARG, "zero_shard_step_offload: params_host is not page-locked");
        for (int b = 0; b < 2; ++b)
            if (!o->master[b] || !o->m[b] || !o->v[b] || !zs::aligned_to(o->master[b], 4) ||
                !zs::aligned_to(o->m[b], 4) || !zs::aligned_to(o->v[b], 4))
                return ZS_ERR_ARG;
    }
    int threads = n_threads > 0 ? n_threads : (int)std::thread::hardware_concurrency();
    if (threads < 1) threads = 1;
    if (chunk == 0) chunk = (int64_t)1 << 22;
    const CpuCoef c = cpu_coef(hp, loss_scale, step, n_d);
    cudaStream_t sd = (cudaStream_t)d2h_stream, sh = (cudaStream_t)h2d_stream;
    *overflow_out = 0;
    if (n == 0) return ZS_OK;

    // the host view of the shard that step_chunk walks
    zs_shard hs;
    memset(&hs, 0, sizeof(hs));
    std::vector<const uint16_t*> hg(o->grads_host, o->grads_host + n_d);
    hs.grads = hg.data();
    for (int b = 0; b < 2; ++b) {
        hs.master[b] = o->master[b];
        hs.m[b] = o->m[b];
        hs.v[b] = o->v[b];
    }
    hs.params = o->params_host;
    hs.n = n;

    const int64_t nc = (n + chunk - 1) / chunk;
    std::vector<cudaEvent_t> ev((size_t)nc, nullptr);
    auto destroy = [&] {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);
    };
    for (int64_t ci = 0; ci < nc; ++ci) {
        cudaError_t err = cudaEventCreateWithFlags(&ev[(size_t)ci], cudaEventDisableTiming);
        if (err != cudaSuccess) {
            destroy();
            return zs::cuda_fail(err, "zero_shard_step_offload: event");
        }
    }
    // every contribution of every chunk, device -> host, in chunk order
    for (int64_t ci = 0; ci < nc; ++ci) {
        const int64_t lo = ci * chunk, len = std::min(chunk, n - lo);
        for (int k = 0; k < n_d; ++k) {
            cudaError_t err = cudaMemcpyAsync(o->grads_host[k] + lo, o->grads_dev[k] + lo, (size_t)len * 2,
                                              cudaMemcpyDeviceToHost, sd);
            if (err != cudaSuccess) {
                cudaStreamSynchronize(sd);
                destroy();
                return zs::cuda_fail(err, "zero_shard_step_offload: gradients to host");
            }
        }
        cudaError_t err = cudaEventRecord(ev[(size_t)ci], sd);
        if (err != cudaSuccess) {
            cudaStreamSynchronize(sd);
            destroy();
            return zs::cuda_fail(err, "zero_shard_step_offload: event record");
        }
    }
    std::unique_ptr<std::atomic<int>[]> done(new std::atomic<int>[(size_t)nc]);
    for (int64_t ci = 0; ci < nc; ++ci) done[(size_t)ci].store(0);
    std::atomic<int> flag{0};
    std::atomic<int> cuda_err{(int)cudaSuccess};
    auto worker = [&](int t) {
        for (int64_t ci = 0; ci < nc; ++ci) {
            const int64_t lo = ci * chunk, len = std::min(chunk, n - lo);
            // this thread's part of the chunk, starts on 16-element boundaries
            const int64_t a = lo + ((len * t / threads) & ~(int64_t)15);
            const int64_t b = t == threads - 1 ? lo + len : lo + ((len * (t + 1) / threads) & ~(int64_t)15);
            cudaError_t err = cudaEventSynchronize(ev[(size_t)ci]);
            if (err != cudaSuccess) {
                cuda_err.store((int)err);
            } else if (b > a && step_chunk(hs, n_d, c, cur, a, b)) {
                flag.store(1, std::memory_order_relaxed);
            }
            if (done[(size_t)ci].fetch_add(1) == threads - 1 && cuda_err.load() == (int)cudaSuccess) {
                err = cudaMemcpyAsync(o->params_dev + lo, o->params_host + lo, (size_t)len * 2,
                                      cudaMemcpyHostToDevice, sh);
                if (err != cudaSuccess) cuda_err.store((int)err);
            }
        }
    };
    std::vector<std::thread> pool;
    pool.reserve((size_t)threads);
    for (int t = 0; t < threads; ++t) pool.emplace_back(worker, t);
    for (auto& th : pool) th.join();
    if (cuda_err.load() != (int)cudaSuccess) {
        cudaStreamSynchronize(sd);
        cudaStreamSynchronize(sh);
        destroy();
        return zs::cuda_fail((cudaError_t)cuda_err.load(), "zero_shard_step_offload: transfers");
    }
    const int ovf = flag.load();
    if (ovf) {
        // the device slice already holds fp16 of the dropped update: rewrite
        // the staging buffer from the kept master weights and send it again
        cudaError_t err = cudaStreamSynchronize(sh);
        if (err == cudaSuccess) {
            parallel_chunks(n, threads, [&](int, int64_t lo, int64_t hi) { restore_chunk(hs, cur, lo, hi); });
            err = cudaMemcpyAsync(o->params_dev, o->params_host, (size_t)n * 2, cudaMemcpyHostToDevice, sh);
        }
        if (err != cudaSuccess) {
            cudaStreamSynchronize(sh);
            destroy();
            return zs::cuda_fail(err, "zero_shard_step_offload: restore");
        }
    }
    cudaError_t err = cudaStreamSynchronize(sh);
    destroy();
    if (err != cudaSuccess) return zs::cuda_fail(err, "zero_shard_step_offload: parameters to device");
    *overflow_out = ovf;
    return ZS_OK;
}

}  // extern "C"
