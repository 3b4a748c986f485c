// diag.cpp -- status strings, last-error text, launch counter and the
// closed-form model-state footprint of libzeroshard.so.
#include <atomic>
#include <cmath>
#include <mutex>
#include <stdio.h>
#include <string>
#include <vector>

#include "zs_internal.h"

namespace zs {

static thread_local std::string g_last_error;
static std::atomic<int64_t> g_launches{0};

int32_t cuda_fail(cudaError_t err, const char* where) {
    char buf[256];
    snprintf(buf, sizeof(buf), "%s: %s (%s)", where, cudaGetErrorString(err), cudaGetErrorName(err));
    g_last_error = buf;
    return ZS_ERR_CUDA;
}

int32_t fail_with(int32_t status, const char* message) {
    g_last_error = message;
    return status;
}

void count_launches(int64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int device_sm_count() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            sms = 1;
        cache[dev] = sms;
    }
    return cache[dev];
}

}  // namespace zs

extern "C" {

ZS_API const char* zero_status_string(int32_t status) {
    switch (status) {
    case ZS_OK: return "ok";
    case ZS_ERR_ARG: return "invalid argument";
    case ZS_ERR_ALIGN: return "misaligned pointer";
    case ZS_ERR_CUDA: return "CUDA error";
    case ZS_ERR_TIMEOUT: return "timeout";
    default: return "unknown status";
    }
}

ZS_API const char* zero_last_error(void) { return zs::g_last_error.c_str(); }

ZS_API int64_t zero_kernel_launches(void) { return zs::g_launches.load(std::memory_order_relaxed); }

ZS_API int32_t zero_debug_checks(uint64_t* first_fault) {
    if (first_fault == nullptr) return ZS_ERR_ARG;
    *first_fault = 0;
#if ZS_CHECKED
    const uint64_t faults[] = {zs::take_fault_shard_step(), zs::take_fault_clip(), zs::take_fault_sgd(),
                               zs::take_fault_adam8()};
    for (uint64_t f : faults) {
        if (f == ~0ull) return zs::fail_with(ZS_ERR_CUDA, "zero_debug_checks: the fault record could not be read");
        if (f != 0 && *first_fault == 0) *first_fault = f;
    }
    return 1;
#else
    return 0;
#endif
}

// Model-state bytes per device ("DeepSpeed ZeRO Stages", sec. 1.2 and 3):
// three categories -- fp16 parameters (2 Psi), fp16 gradients (2 Psi) and
// optimizer states (K Psi) -- and the stages partition them cumulatively,
// optimizer states from stage 1, gradients from stage 2, parameters from
// stage 3.  A partitioned category costs 1/N_d of its bytes on each device.
ZS_API double zero_state_bytes(double psi, int32_t n_d, int32_t stage, double k) {
    if (n_d < 1 || stage < 0 || stage > 3) return NAN;
    const double nd = (double)n_d;
    const double bytes[3] = {k * psi, 2.0 * psi, 2.0 * psi};  // optimizer, gradients, parameters
    double total = 0.0;
    for (int c = 0; c < 3; ++c) total += (stage > c) ? bytes[c] / nd : bytes[c];
    return total;
}

}  // extern "C"
