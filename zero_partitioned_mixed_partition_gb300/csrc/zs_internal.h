// zs_internal.h -- declarations shared by the translation units of
// libzeroshard.so (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "zero_shard.h"

namespace zs {

// Records a CUDA failure for zero_last_error() and returns ZS_ERR_CUDA.
int32_t cuda_fail(cudaError_t err, const char* where);
// Records a message for zero_last_error() and returns status.
int32_t fail_with(int32_t status, const char* message);
// Adds n to the count reported by zero_kernel_launches().
void count_launches(int64_t n);

// NVTX range around an entry point, so profiler timelines show each step
// (header-only NVTX: a no-op unless a profiling tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

inline bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Checks the launch that was just enqueued.
inline int32_t check_launch(const char* where, int64_t n = 1) {
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return cuda_fail(err, where);
    count_launches(n);
    return ZS_OK;
}

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Persistent grid for `kernel`: every SM filled at the kernel's occupancy
// (at most max_per_sm blocks per SM when > 0), no more blocks than
// work_items / threads.
int persistent_blocks(const void* kernel, int threads, int64_t work_items, int max_per_sm = 0);
// Hyper-parameters finite, betas in [0, 1), eps >= 0.
bool valid_hp(const zs_adam* hp);
// Checks one shard's pointers; *width gets the access width they allow
// (2 = 16 elements per thread, 1 = 8, 0 = scalar).
int32_t check_shard(const zs_shard& s, int32_t n_d, int* width);
int32_t check_shard_list(const zs_shard* shards, int32_t n_shards, int32_t n_d, int* width);
// Enqueues the qwZ copy of blocks [b0, b1) of one shard (re-cast from master
// first when master != nullptr).
int32_t launch_qwz(const float* master, uint16_t* params, int64_t n, int8_t* codes, float* scales, int64_t b0,
                   int64_t b1, cudaStream_t stream);
// The first index-check failure recorded by the kernels of each translation
// unit (checked build only; 0 = none, ~0 = the record could not be read),
// cleared on read.
uint64_t take_fault_shard_step();
uint64_t take_fault_clip();
uint64_t take_fault_sgd();
uint64_t take_fault_adam8();
// Enqueues the device-side commit / skip of a step over `shards`.
int32_t launch_commit(const zs_shard* shards, int32_t n_shards, const zs_adam& hp, zs_ctrl* ctrl,
                      cudaStream_t stream);
// Enqueues, with programmatic serialization, the pass that follows a step
// whose last fused launch already finished it in the control block: it
// re-casts each shard's fp16 slice from master[cur] if that step overflowed
// and otherwise leaves at once (shards without a qwZ copy; only params,
// master and n of each zs_shard are read).  early_dependents: let the next
// kernel of the stream be scheduled before this pass waits (measured faster
// ahead of the 8-bit Adam kernel, whose CTAs first copy their code tables,
// and slower ahead of the fp32 Adam and SGD kernels).
int32_t launch_restore_pass(const zs_shard* shards, int32_t n_shards, zs_ctrl* ctrl, cudaStream_t stream,
                            bool early_dependents = false);

}  // namespace zs
