/*
 * zero_shard.h -- C ABI of libzeroshard.so, the GB300 (sm_103a) ZeRO-partitioned
 * mixed-precision Adam shard step.
 *
 * What the library computes, and where it is defined:
 *   - the partition of the flat parameter index set into N_d disjoint,
 *     near-equal shards, one per data-parallel rank
 *     ("DeepSpeed ZeRO Stages", sec. 2 "What 'Partitioning' Means Here";
 *      sec. 3.2, flat contiguous gradient buffer);
 *   - the rank's share of the reduce-scatter: its shard of the N_d fp16
 *     gradient contributions, averaged ("ZeRO Stage 1 Math", "The per-step
 *     mechanics", beat 2);
 *   - the elementwise Adam update of the fp32 master weights, m and v of the
 *     shard and the cast of the shard to fp16 ("DeepSpeed ZeRO Stages",
 *     sec. 2.1 Fact 1; "ZeRO Stage 1 Math", "Where the 12 bytes come from"
 *     and "The per-step mechanics", beat 3);
 *   - the model-state memory per device of stages 0-3 ("DeepSpeed ZeRO
 *     Stages", sec. 1.2 and 3.1-3.3).
 * The pages do not describe loss scaling.  The library applies the usual
 * dynamic-loss-scale rule: the contributions carry a loss scale L that the
 * step removes, and a non-finite reduced gradient anywhere in the stepped
 * shards skips the whole step and halves L (never below 1).
 *
 * Conventions shared by every entry point:
 *   - fp16 data is passed as uint16_t bit patterns (IEEE binary16);
 *   - "DEVICE" pointers are CUDA device (or managed) memory of the current
 *     device, "HOST" pointers are ordinary host memory;
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream);
 *   - the caller owns every buffer; the library allocates no memory and keeps
 *     no pointer after a call returns;
 *   - arguments are checked on the host before anything is enqueued: a bad
 *     argument returns ZS_ERR_ARG (or ZS_ERR_ALIGN) and launches nothing; a
 *     CUDA failure returns ZS_ERR_CUDA and zero_last_error() describes it.
 */
#ifndef ZERO_SHARD_H_
#define ZERO_SHARD_H_

#include <stdint.h>

#if defined(_WIN32)
#define ZS_API
#else
#define ZS_API __attribute__((visibility("default")))
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define ZS_OK 0
#define ZS_ERR_ARG (-1)     /* invalid argument; nothing was enqueued */
#define ZS_ERR_ALIGN (-2)   /* a pointer is not aligned to its element type */
#define ZS_ERR_CUDA (-3)    /* a CUDA call failed; see zero_last_error() */
#define ZS_ERR_TIMEOUT (-4) /* reserved: no kernel of this library polls a flag */

/* Largest data-parallel degree (number of gradient contributions). */
#define ZS_MAX_ND 1024
/* Largest number of shards one step may update together. */
#define ZS_MAX_SHARDS 256
/* Parameters per block of the int8 (qwZ) copy of the fp16 shard. */
#define ZS_QWZ_BLOCK 256

/* One piece of the partition: the overlap of one tensor with one shard. */
typedef struct zs_fragment {
    int32_t tensor;        /* index of the tensor in the list */
    int32_t shard;         /* owning rank */
    int64_t tensor_offset; /* first element of the piece inside the tensor */
    int64_t shard_offset;  /* first element of the piece inside the shard */
    int64_t length;        /* elements, > 0 */
} zs_fragment;

/* Arithmetic of the Adam update's last division (zs_adam.math).
 *
 *   ZS_MATH_IEEE  every fp32 operation is one IEEE round-to-nearest step:
 *                 mh = m / (1 - b1^t), vh = v / (1 - b2^t),
 *                 u = mh / (sqrt(vh) + eps).  The results equal the plain
 *                 definition bit for bit (and so the oracle of the tests).
 *   ZS_MATH_FAST  permission to form u from the hardware reciprocal estimate
 *                 of sqrt(vh) + eps with one fused-multiply-add residual
 *                 correction instead of the IEEE divide.  u is then within
 *                 1 ulp of the exact quotient and equal to the IEEE one
 *                 except when the quotient lies extremely close to a rounding
 *                 midpoint; the bias corrections, the square root, m and v are
 *                 IEEE in both modes, so m and v are always bit-identical and
 *                 master/params differ, rarely, by one rounding of lr * u.
 *                 Taken by the 8-element layout and by the 16-element layout
 *                 compiled for N_d = 16, 32 or 64 (the fused step without a
 *                 qwZ copy, and the clipped step's update); the scalar layout,
 *                 the run-time-N_d 16-element layout, the fused step with a
 *                 qwZ copy and the host-core step run IEEE.
 *
 * "DeepSpeed ZeRO Stages", sec. 2.1, Fact 1 (the Adam step of each coordinate)
 * names no rounding for these operations. */
#define ZS_MATH_IEEE 0
#define ZS_MATH_FAST 1

/* Adam / AdamW hyper-parameters.  weight_decay = 0 gives plain Adam; a
 * positive value applies decoupled decay: theta -= lr * (u + wd * theta).
 * math is ZS_MATH_IEEE or ZS_MATH_FAST; reserved must be 0.  A zero-filled
 * struct tail therefore selects the IEEE mode. */
typedef struct zs_adam {
    double lr;
    double beta1;
    double beta2;
    double eps;
    double weight_decay;
    int32_t math;
    int32_t reserved;
} zs_adam;

/* SGD-with-momentum hyper-parameters (zero_shard_step_sgd_async). */
typedef struct zs_sgd {
    double lr;
    double momentum;      /* mu >= 0; 0 gives plain SGD */
    double weight_decay;  /* L2 decay folded into the gradient */
} zs_sgd;

/* One shard of the optimizer state, as one rank owns it.
 *   grads     HOST array of n_d DEVICE pointers; grads[k] is simulated rank
 *             k's fp16 gradient for the elements of this shard (scaled by the
 *             loss scale), >= n values.  The table is read during the call.
 *   master, m, v
 *             DEVICE fp32 buffers of >= n values, two sets for ping-pong: a
 *             step reads set `cur` and writes set `cur ^ 1`, so an overflow
 *             step can be dropped without a second pass.  Passing the same
 *             pointer for both sets updates in place; the caller then accepts
 *             that an overflow step cannot be rolled back.
 *   params    DEVICE fp16 slice of the full parameter buffer that this shard
 *             maps to (params_full + rank * shard_numel), >= n values.
 *   n         elements stepped: the shard's real (non-padding) parameters.
 *             Elements past n are not read or written.
 * Access width follows alignment: with every fp32 buffer 32-byte aligned and
 * every fp16 buffer 16-byte aligned the kernel moves 16 elements per thread
 * and iteration (used when n_d > 4); with 16-byte alignment, 8; any other
 * 4-byte (fp32) / 2-byte (fp16) aligned layout takes a scalar kernel.  All
 * three do the same arithmetic in the same order.
 *   qcodes, qscales
 *             optional (both NULL, or both set): the int8 copy of the fp16
 *             shard that the parameter all-gather sends instead of fp16
 *             (ZeRO++ quantized weights, "ZeRO Optimization: Stages 1, 2, and
 *             3 Explained"; "DeepSpeed ZeRO Stages" sec. 5.3 qwZ).  DEVICE
 *             int8 codes[n] and fp32 scales[ceil(n / ZS_QWZ_BLOCK)]: block b
 *             holds params [256 b, 256 b + 256) as q = rint(x / s), ties to
 *             even, s = max|x| / 127, x the fp16 values.  When set, every
 *             step (and every restore after an overflow) leaves them matching
 *             the fp16 slice; the fused kernel writes full blocks in its own
 *             pass (1 + 4/256 extra bytes per element) and the commit writes
 *             the trailing partial block.  codes 16-byte aligned for the
 *             16-element path, 8-byte for the 8-element one. */
typedef struct zs_shard {
    const uint16_t* const* grads;
    float* master[2];
    float* m[2];
    float* v[2];
    uint16_t* params;
    int64_t n;
    int8_t* qcodes;
    float* qscales;
} zs_shard;

/* Device-resident step state for the stream-ordered (no host sync) path.
 * The caller allocates sizeof(zs_ctrl) bytes of 8-byte aligned DEVICE memory
 * and sets it up with zero_ctrl_init(); the library then owns its contents
 * between calls.  It may be copied to the host at any time the stream is
 * idle (for logging or a checkpoint) and copied back to resume. */
typedef struct zs_ctrl {
    double loss_scale;     /* L applied to the next step */
    double beta1_pow;      /* beta1^t for the t committed updates */
    double beta2_pow;      /* beta2^t */
    int64_t step;          /* t: committed updates so far */
    int64_t skipped;       /* steps dropped because of an overflow */
    int32_t cur;           /* state set (0/1) that holds the committed state */
    int32_t overflow;      /* OR of the non-finite tests of the step in flight */
    int32_t last_overflow; /* overflow flag of the last finished step */
    uint32_t arrivals;     /* internal block counter of the step's end (the commit kernel, or the
                              last fused launch of zero_shard_step_async, _sgd_async,
                              _adam8_async or _clipped_async); 0 between steps */
} zs_ctrl;

/* ------------------------------------------------------------------------ */
/* Partition ("DeepSpeed ZeRO Stages", sec. 2).                              */
/* ------------------------------------------------------------------------ */

/* Pack n_tensors tensors (HOST numels[], >= 0 each) back to back into one flat
 * buffer of Psi elements, pad it to Psi_pad = the least multiple of
 * n_d * align, and cut it into n_d equal shards of S = Psi_pad / n_d
 * elements; shard i is [i S, (i+1) S).  Outputs (HOST, each may be NULL):
 *   *psi_out, *psi_padded_out, *shard_numel_out;
 *   tensor_offsets[n_tensors]  flat offset of each tensor;
 *   shard_offsets[n_d + 1]     i * S;
 *   frags[frag_cap]            the tensor/shard overlaps, in flat order
 *                              (shard-major, tensors in list order);
 *   *n_frags_out               number of fragments (always written when
 *                              non-NULL; with frags == NULL this is a count
 *                              query).  At most n_tensors + n_d - 1.
 * n_d in [1, ZS_MAX_ND]; align a power of two.  Returns ZS_ERR_ARG for a bad
 * argument, a negative numel, or frag_cap smaller than the count (in which
 * case *n_frags_out holds the count needed and frags is left partly filled).
 * Runs on the host; no CUDA call.
 * Source: "DeepSpeed ZeRO Stages", sec. 2 (disjoint near-equal partition of the index set) and sec.
 * 3.2 (flat contiguous gradient buffer). */
ZS_API int32_t zero_partition_layout(const int64_t* numels, int32_t n_tensors, int32_t n_d,
                                     int32_t align, int64_t* psi_out, int64_t* psi_padded_out,
                                     int64_t* shard_numel_out, int64_t* tensor_offsets,
                                     int64_t* shard_offsets, zs_fragment* frags, int64_t frag_cap,
                                     int64_t* n_frags_out);

/* The same partition computed on the device by one CUDA block, stream-ordered.
 *   numels_dev[n_tensors]          DEVICE input
 *   scalars_dev[5]                 DEVICE output: Psi, Psi_pad, S, number of
 *                                  fragments, status (ZS_OK, or ZS_ERR_ARG when
 *                                  a numel is negative; the other outputs are
 *                                  then unspecified)
 *   tensor_offsets_dev[n_tensors]  DEVICE output (may be NULL if n_tensors = 0)
 *   shard_offsets_dev[n_d + 1]     DEVICE output
 *   frags_dev[frag_cap]            DEVICE output or NULL; fragments past
 *                                  frag_cap are counted but not written
 *                                  (frag_cap >= n_tensors + n_d - 1 always
 *                                  suffices).
 * The results are bit-identical to zero_partition_layout.  Host-side checks
 * return ZS_ERR_ARG / ZS_ERR_ALIGN (8-byte alignment) before any launch.
 * Source: "DeepSpeed ZeRO Stages", sec. 2 and sec. 3.2 (as zero_partition_layout). */
ZS_API int32_t zero_partition_layout_device(const int64_t* numels_dev, int32_t n_tensors,
                                            int32_t n_d, int32_t align, int64_t* scalars_dev,
                                            int64_t* tensor_offsets_dev, int64_t* shard_offsets_dev,
                                            zs_fragment* frags_dev, int64_t frag_cap, void* stream);

/* ------------------------------------------------------------------------ */
/* Model-state memory ("DeepSpeed ZeRO Stages", sec. 1.2, 3.1-3.3).          */
/* ------------------------------------------------------------------------ */

/* Bytes of model state per device for psi parameters on n_d ranks with an
 * optimizer multiplier k (12 for mixed-precision Adam):
 *   stage 0: (4 + k) psi          stage 1: 4 psi + k psi / n_d
 *   stage 2: 2 psi + (2 + k) psi / n_d      stage 3: (4 + k) psi / n_d
 * Returns NaN for a stage outside 0..3 or n_d < 1.  Host only.
 * Source: "DeepSpeed ZeRO Stages", sec. 1.2 and 3.1-3.3; "DeepSpeed ZeRO: Extreme Memory
 * Efficiency", "Three stages of partitioning the redundancy away". */
ZS_API double zero_state_bytes(double psi, int32_t n_d, int32_t stage, double k);

/* ------------------------------------------------------------------------ */
/* The shard step.                                                           */
/* ------------------------------------------------------------------------ */

/* One optimizer step over n_shards shards, with a host round trip.
 * For every element j < n of every shard, in the fused kernels (consecutive
 * shards of one access width share a launch; see
 * zero_shard_reduce_adam_all_async):
 *   gs   = sum over k = 0..n_d-1, in that order, of fp32(grads[k][j])
 *   g    = gs * (float)(1 / (n_d * loss_scale))
 *   m'   = b1 m + (1 - b1) g;   v' = b2 v + (1 - b2) g^2
 *   u    = (m' / (1 - beta1^step)) / (sqrt(v' / (1 - beta2^step)) + eps)
 *   th'  = th - lr (u + weight_decay th);   params[j] = fp16_rn(th')
 * reading state set `cur`, writing set `cur ^ 1`; with ZS_MATH_IEEE every fp32
 * operation is one IEEE round-to-nearest step, no fused multiply-add (see
 * zs_adam.math for ZS_MATH_FAST).
 * The non-finite test of gs over all shards is ORed into *flag_dev (DEVICE
 * int32 scratch, cleared by this call).  The call then waits for the stream;
 * on overflow it rewrites every shard's params from master[cur] so the fp16
 * slice again matches the committed state.  *overflow_out (HOST) gets 0 or 1.
 * The caller commits: overflow == 0 -> cur ^= 1, step + 1 for the next call;
 * overflow == 1 -> keep cur and step, halve the loss scale (floor 1).
 * step >= 1 is the Adam time t of this update (committed updates + 1).
 * Source: "ZeRO Stage 1 Math", "The per-step mechanics", beats 2-3; "DeepSpeed ZeRO Stages", sec.
 * 2.1, Fact 1; skip and loss-scale halving: the dynamic loss-scale rule (not in the pages). */
ZS_API int32_t zero_shard_step(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                               const zs_adam* hp, double loss_scale, int64_t step, int32_t cur,
                               int32_t* flag_dev, void* stream, int32_t* overflow_out);

/* Largest n_shards zero_shard_step_noalloc accepts (size of its static scratch). */
#define ZS_NOALLOC_MAX_SHARDS 64

/* zero_shard_step for callers that cannot allocate device memory.  The pages
 * have no counterpart of this entry point; it exists for the host program, not
 * for the method.  Some callers only own the buffers they are handed and may
 * not call cudaMalloc: a plugin or language binding inside an application whose
 * allocator has reserved the whole device (a stray allocation would bypass or
 * fragment that pool, or fail once the pool has claimed the memory), or code
 * that must not allocate after start-up.  zero_shard_step needs a caller
 * buffer for its overflow word; this variant keeps one overflow word per shard
 * in a 256-byte array compiled into the library (each GPU that loads the
 * library holds it until the process exits) and allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library call.
 *   - arguments, arithmetic, restore-on-overflow and *overflow_out are those of
 *     zero_shard_step (without flag_dev);
 *   - n_shards above ZS_NOALLOC_MAX_SHARDS returns ZS_ERR_ARG (the text is in
 *     zero_last_error()) and launches nothing;
 *   - the first call on each device (and in each new context of it) looks up
 *     the array's device address with that device current; make that first
 *     call before any stream capture;
 *   - the kernels are those of zero_shard_step, with the same grouping of
 *     consecutive shards into one launch; each launch ORs its non-finite
 *     test into the word of its first shard;
 *   - every call shares the array, and it keeps the last call's contents; each
 *     call clears the words it uses before its kernels run.  Calls whose work
 *     overlaps on the GPU (other streams, other host threads) race on it, so
 *     order them.
 *   - the array's address is cached per device and per CUDA context (by the
 *     driver's context ID), so a context created after cudaDeviceReset looks
 *     it up again. */
ZS_API int32_t zero_shard_step_noalloc(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                       const zs_adam* hp, double loss_scale, int64_t step,
                                       int32_t cur, void* stream, int32_t* overflow_out);

/* Set up a device control block: loss scale L, t = 0, cur = 0, counters 0.
 * Stream-ordered (one tiny kernel).
 * Source: the dynamic loss-scale rule (not in the pages) and the Adam time t of "DeepSpeed ZeRO
 * Stages", sec. 2.1, Fact 1. */
ZS_API int32_t zero_ctrl_init(zs_ctrl* ctrl_dev, double loss_scale, void* stream);

/* The same step with no host synchronisation (CUDA-graph friendly): the loss
 * scale, t and the ping-pong set come from *ctrl_dev, and the commit-or-skip
 * decision runs on the device.  Enqueues the fused kernels of every shard
 * with n > 0 (as zero_shard_reduce_adam_all_async), then:
 *   - no shard with a qwZ copy: the last fused launch finishes the step
 *     itself (its last block to finish commits or skips, as
 *     zero_step_commit_async decides), and one restore kernel follows that
 *     rewrites the params from master[cur] only if the step overflowed and
 *     otherwise ends at once.  These kernels are launched with programmatic
 *     stream serialization: each may be scheduled while the previous kernel
 *     in the stream ends, and waits for it before touching memory;
 *   - otherwise one commit kernel (zero_step_commit_async), which also writes
 *     the qwZ copies' trailing blocks.
 * The results are those of the two-call form in either case.
 * Source: "ZeRO Stage 1 Math", "The per-step mechanics", beats 2-3; "DeepSpeed ZeRO Stages", sec.
 * 2.1, Fact 1. */
ZS_API int32_t zero_shard_step_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                     const zs_adam* hp, zs_ctrl* ctrl_dev, void* stream);

/* First half of zero_shard_step_async for one shard: the fused reduce +
 * non-finite test + Adam + fp16 cast kernel, with t = ctrl->step + 1, the
 * loss scale ctrl->loss_scale and set ctrl->cur; ORs its test into
 * ctrl->overflow.  Several shards of one step each get one call, then one
 * zero_step_commit_async for all of them.
 * Source: "ZeRO Stage 1 Math", "The per-step mechanics", beats 2-3; "DeepSpeed ZeRO Stages", sec.
 * 2.1, Fact 1. */
ZS_API int32_t zero_shard_reduce_adam_async(const zs_shard* shard, int32_t n_d, const zs_adam* hp,
                                            zs_ctrl* ctrl_dev, void* stream);

/* The first half of zero_shard_step_async for every listed shard: the fused
 * kernels only, without the commit (zero_step_commit_async follows).
 * Consecutive shards that share an access width and all carry (or all lack) a
 * qwZ copy, with n_d <= 64, are stepped up to 16 at a time by one launch of a
 * grouped kernel that walks their concatenated elements (one launch ramp and
 * tail instead of one per shard); the others get one launch each, as
 * zero_shard_reduce_adam_async.  The
 * arithmetic per element is the same in both.  Arguments and errors as
 * zero_shard_step_async.
 * Source: "ZeRO Stage 1 Math", "The per-step mechanics", beats 2-3; "DeepSpeed ZeRO Stages", sec.
 * 2.1, Fact 1. */
ZS_API int32_t zero_shard_reduce_adam_all_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                                const zs_adam* hp, zs_ctrl* ctrl_dev, void* stream);

/* Second half: if ctrl->overflow is set, rewrite every listed shard's params
 * from master[ctrl->cur] and halve the loss scale (floor 1), counting a skip;
 * otherwise flip ctrl->cur, advance t and beta^t.  Records last_overflow and
 * clears overflow for the next step.  The shard list must be the shards the
 * step updated (grads are not used).
 * Source: "ZeRO Stage 1 Math", "The per-step mechanics", beat 3 (the fp16 copy of the kept master);
 * skip and halving: the dynamic loss-scale rule (not in the pages). */
ZS_API int32_t zero_step_commit_async(const zs_shard* shards, int32_t n_shards, const zs_adam* hp,
                                      zs_ctrl* ctrl_dev, void* stream);

/* The whole step with the gradient contributions and the fp16 shard in HOST
 * memory, for callers whose gradients arrive in, and whose parameters leave
 * through, host memory.  shard->grads[k] and shard->params are HOST pointers
 * into page-locked memory (cudaHostAlloc / cudaMallocHost / cudaHostRegister);
 * master, m and v stay DEVICE buffers.  No copy is staged: the fused kernel
 * reads the contributions and writes the fp16 shard through the host mapping
 * (on Grace-Blackwell over the coherent NVLink-C2C link), so transfer and
 * compute overlap in one pass.  The step is then committed on the device as in
 * zero_shard_step_async, and the call waits for the stream and returns the
 * step's overflow flag in *overflow_out (HOST).  A host pointer that is not
 * page-locked and mapped for the current device returns ZS_ERR_ARG before any
 * launch.
 * Source: "ZeRO Stage 1 Math", "The per-step mechanics", beats 2-3; "DeepSpeed ZeRO Stages", sec.
 * 2.1, Fact 1; host-resident data as in ZeRO-Offload, "DeepSpeed ZeRO Stages", sec. 5.1. */
ZS_API int32_t zero_shard_step_host(const zs_shard* shard, int32_t n_d, const zs_adam* hp,
                                    zs_ctrl* ctrl_dev, void* stream, int32_t* overflow_out);

/* ------------------------------------------------------------------------ */
/* Global gradient-norm clipping ("DeepSpeed ZeRO Stages", sec. 2.1, Fact 1:   */
/* the one operation of the step that couples coordinates, through ||g||_2   */
/* over all of P, at the price of one scalar all-reduce).                    */
/* ------------------------------------------------------------------------ */
/* With clipping the step takes two passes around one scalar S = sum_j g_j^2
 * over every shard of every rank (g the reduced, unscaled gradient of
 * zero_shard_step):
 *   1. zero_shard_grad_sqnorm_async on each local shard: reduce, ORs the
 *      non-finite test into ctrl->overflow and ADDS the shard's sum of
 *      squares (double) to *sqnorm_dev (DEVICE, 8-byte aligned; the caller
 *      clears it before the step).  g_dev (DEVICE fp32, >= n values, or NULL)
 *      keeps g for pass 2.
 *   2. the ranks sum *sqnorm_dev (one-double all-reduce); shards stepped on
 *      one device are already summed.
 *   3. zero_shard_clipped_adam_async on each shard: c = min(1, max_norm /
 *      (sqrt(S) + 1e-6)) in double, rounded once to float (max_norm <= 0: no
 *      clipping), g' = g * c in fp32, then the update and fp16 cast of
 *      zero_shard_step with g'.  g is read from g_dev, or re-reduced from the
 *      contributions when g_dev is NULL (same bits).
 *   4. zero_step_commit_async for all the shards.
 * Per element: 4 n_d + 26 bytes without g_dev, 2 n_d + 34 with it; keep g
 * once n_d > 4.  Loss scale, t and the ping-pong set come from *ctrl_dev as in
 * zero_shard_step_async.
 * Source: "DeepSpeed ZeRO Stages", sec. 2.1, Fact 1 (clipping couples the coordinates through ||g||
 * over all of P), with the update of "ZeRO Stage 1 Math", "The per-step mechanics", beats 2-3. */
ZS_API int32_t zero_shard_grad_sqnorm_async(const zs_shard* shard, int32_t n_d, float* g_dev,
                                            double* sqnorm_dev, zs_ctrl* ctrl_dev, void* stream);
ZS_API int32_t zero_shard_clipped_adam_async(const zs_shard* shard, int32_t n_d, const zs_adam* hp,
                                             double max_norm, const float* g_dev,
                                             const double* sqnorm_dev, zs_ctrl* ctrl_dev, void* stream);

/* Passes 1 and 3 above for a list of shards: consecutive shards of one access
 * width go up to 16 at a time into one launch that walks their concatenated
 * elements (n_d <= 64; one shard per launch above).  g_dev: HOST array of
 * n_shards DEVICE pointers (entries may be NULL), or NULL for none.  The
 * arithmetic per element is that of the one-shard calls.
 * Source: "DeepSpeed ZeRO Stages", sec. 2.1, Fact 1 (clipping), with the update of "ZeRO Stage 1
 *   Math", "The per-step mechanics", beats 2-3. */
ZS_API int32_t zero_shard_grad_sqnorm_all_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                                float* const* g_dev, double* sqnorm_dev, zs_ctrl* ctrl_dev,
                                                void* stream);
ZS_API int32_t zero_shard_clipped_adam_all_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                                 const zs_adam* hp, double max_norm, float* const* g_dev,
                                                 const double* sqnorm_dev, zs_ctrl* ctrl_dev, void* stream);
/* Steps 1-4 for shards that all live on this device (the norm is then exact
 * over them): clears *sqnorm_dev, runs pass 1 over every shard, pass 2 over
 * every shard, and the commit: without a qwZ copy, pass 2's last launch ends
 * the step itself and one restore kernel follows (as in
 * zero_shard_step_async); with one, the commit kernel.  g_dev: HOST array of
 * n_shards DEVICE pointers (each may be NULL), or NULL to re-reduce
 * everywhere.
 * Source: "DeepSpeed ZeRO Stages", sec. 2.1, Fact 1 (clipping). */
ZS_API int32_t zero_shard_step_clipped_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                             const zs_adam* hp, double max_norm, float* const* g_dev,
                                             double* sqnorm_dev, zs_ctrl* ctrl_dev, void* stream);

/* params[j] = fp16_rn(master[j]) for j < n (DEVICE buffers): initialises the
 * fp16 parameter slice from fp32 master weights.  Stream-ordered.
 * Source: "ZeRO Stage 1 Math", "The per-step mechanics", beat 3 (fp16 parameters cast from the fp32
 * master). */
ZS_API int32_t zero_params_from_master(const float* master_dev, uint16_t* params_dev, int64_t n,
                                       void* stream);

/* ------------------------------------------------------------------------ */
/* Mixed-precision SGD with momentum (the other optimizer of the state        */
/* multiplier K, "DeepSpeed ZeRO Stages", sec. 1.2).                         */
/* ------------------------------------------------------------------------ */

/* The step of zero_shard_step_async with SGD with momentum in place of Adam:
 *   g as for Adam,  d = g + weight_decay theta,  b' = momentum b + d,
 *   theta' = theta - lr b',  params = fp16_rn(theta')
 * The momentum b lives in zs_shard.m (both sets; b starts at 0), zs_shard.v
 * is unused (may be NULL) and qcodes must be NULL.  Loss scale and the
 * ping-pong set come from *ctrl_dev; consecutive shards of one access width
 * are stepped up to 16 per launch; the step's last launch ends it in the
 * control block (its last block to finish commits or skips, as
 * zero_step_commit_async decides, with beta1 = beta2 = 0 for the unused
 * beta^t products) and one restore kernel follows that re-casts the fp16
 * slices only after an overflow, both with programmatic serialization (a call
 * with only empty shards ends in the commit kernel instead).  Per element
 * 2 n_d + 18 bytes.
 * Source: "DeepSpeed ZeRO Stages", sec. 1.2 (mixed-precision SGD with momentum, K = 4). */
ZS_API int32_t zero_shard_step_sgd_async(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                         const zs_sgd* hp, zs_ctrl* ctrl_dev, void* stream);

/* ------------------------------------------------------------------------ */
/* 8-bit Adam (the optimizer of state multiplier K = 6, "DeepSpeed ZeRO       */
/* Stages", sec. 1.2; block-wise quantization after Dettmers et al., "8-bit  */
/* Optimizers via Block-wise Quantization").                                 */
/* ------------------------------------------------------------------------ */

/* Elements per quantization block of the 8-bit states. */
#define ZS_ADAM8_BLOCK 2048

/* One shard of 8-bit Adam state.  As zs_shard, with m and v kept as one byte
 * per element and one fp32 scale per block of ZS_ADAM8_BLOCK elements (block b
 * = elements [2048 b, 2048 b + 2048), the last one possibly shorter):
 *   grads, master, params, n   as in zs_shard;
 *   m_codes, v_codes           DEVICE uint8[n], two sets (ping-pong with
 *                              master): bit 7 of an m code is the sign, bits
 *                              0-6 index the 128 magnitudes of the signed map;
 *                              a v code indexes the 256 values of the unsigned
 *                              map (zero_adam8_maps);
 *   m_scale, v_scale           DEVICE fp32[ceil(n / 2048)], two sets: the
 *                              block's largest |m| (largest v).
 * The state value is map[code] * scale; codes and scales all 0 are m = v = 0
 * (the state before the first step).  With grads and params 16-byte aligned,
 * master 16-byte and the codes 8-byte aligned a thread moves 8 elements per
 * access (16 with n_d > 16 and master 32-byte, codes 16-byte aligned); other
 * naturally aligned buffers take element-wise accesses, same arithmetic. */
typedef struct zs_adam8_shard {
    const uint16_t* const* grads;
    float* master[2];
    uint8_t* m_codes[2];
    uint8_t* v_codes[2];
    float* m_scale[2];
    float* v_scale[2];
    uint16_t* params;
    int64_t n;
} zs_adam8_shard;

/* The step of zero_shard_step_async with 8-bit states: g, the non-finite
 * test, the loss scale, t and the ping-pong set as there; then for every
 * block, reading set cur and writing set cur ^ 1:
 *   m = +-mag7[m_code & 127] * m_scale,   v = mag8[v_code] * v_scale
 *   m', v', theta' and params = fp16_rn(theta') as in zero_shard_step
 *   m_scale' = max |m'| and v_scale' = max v' over the block
 *   m_code' = the code of the map value nearest to x = m' / m_scale' (the
 *   quotient rounded once to fp32, as an IEEE division rounds it; x = 0 when
 *   the scale is 0), ties to the smaller magnitude, sign bit for a negative x
 *   with a non-zero magnitude code; v alike.
 * hp->math applies to u as in zero_shard_step; the codes do not depend on it.
 * Consecutive shards of one access width (empty shards join any group) are
 * stepped up to 16 per launch with n_d <= 64, one per launch above.  The
 * step's last launch ends it in the control block and one restore kernel
 * follows, as in zero_shard_step_sgd_async (a skipped step leaves set cur, so
 * codes and scales too, untouched).  Per element 2 n_d + 14 bytes (+ 16 per
 * block).
 * Source: "DeepSpeed ZeRO Stages", sec. 1.2 (8-bit Adam, K = 6), with the update of "ZeRO Stage 1
 * Math", "The per-step mechanics", beats 2-3. */
ZS_API int32_t zero_shard_step_adam8_async(const zs_adam8_shard* shards, int32_t n_shards, int32_t n_d,
                                           const zs_adam* hp, zs_ctrl* ctrl_dev, void* stream);

/* The library's two code maps (HOST outputs): mag7[128], the magnitudes of the
 * signed map for m, and mag8[256], the unsigned map for v.  Code 0 is 0;
 * code k > 0 has decimal exponent E = (number of leading zero bits of k in a
 * 7- or 8-bit field) and fraction bits j below its leading one bit (f of
 * them): value 10^-E (0.1 + 0.9 (j + 1) / 2^f), formed in double, rounded once
 * to float.  Returns ZS_ERR_ARG for a NULL output.  No CUDA call.
 * Source: the dynamic map of Dettmers et al., "8-bit Optimizers via Block-wise Quantization", for
 * the 8-bit Adam of "DeepSpeed ZeRO Stages", sec. 1.2. */
ZS_API int32_t zero_adam8_maps(float* mag7, float* mag8);

/* ------------------------------------------------------------------------ */
/* The step on the host CPU cores (ZeRO-Offload, "DeepSpeed ZeRO Stages",     */
/* sec. 5.1: optimizer state and update on the CPU, with SIMD and threads).  */
/* ------------------------------------------------------------------------ */

/* zero_shard_step with every buffer in HOST memory (grads[k], master, m, v,
 * params; no qwZ copy), run on n_threads host threads (0 = all cores).  Same
 * arithmetic, ping-pong, overflow test and restore as zero_shard_step, bit for
 * bit; synchronous; *overflow_out (HOST) gets 0 or 1 and the caller commits as
 * for zero_shard_step.  No CUDA call.
 * Source: "DeepSpeed ZeRO Stages", sec. 5.1 (ZeRO-Offload: the optimizer step on the CPU). */
ZS_API int32_t zero_shard_step_cpu(const zs_shard* shards, int32_t n_shards, int32_t n_d,
                                   const zs_adam* hp, double loss_scale, int64_t step, int32_t cur,
                                   int32_t n_threads, int32_t* overflow_out);

/* One rank's shard for the ZeRO-Offload step with its transfers.
 *   grads_dev    HOST array of n_d DEVICE pointers: the rank's n-element
 *                slices of the n_d fp16 gradient contributions (rank order)
 *   params_dev   DEVICE fp16 slice of the full parameter buffer (n elements)
 *                that receives the updated parameters
 *   grads_host   HOST array of n_d page-locked HOST staging buffers of n fp16
 *                elements each (cudaHostAlloc / cudaHostRegister)
 *   params_host  page-locked HOST staging buffer of n fp16 elements
 *   master, m, v two sets of HOST fp32 state (n elements each), set cur read,
 *                set cur ^ 1 written, as for zero_shard_step_cpu
 *   n            elements of the shard (>= 0)
 * The caller owns every buffer; the library allocates no memory (it creates
 * and destroys one CUDA event per chunk within the call). */
typedef struct zs_offload_shard {
    const uint16_t* const* grads_dev;
    uint16_t* params_dev;
    uint16_t* const* grads_host;
    uint16_t* params_host;
    float* master[2];
    float* m[2];
    float* v[2];
    int64_t n;
} zs_offload_shard;

/* ZeRO-Offload's step of one rank: the gradients cross the link to the host,
 * the host cores run the Adam step on the host-resident fp32 state, and the
 * new fp16 parameters cross back.  The shard is cut into chunks of `chunk`
 * elements (0: 4,194,304; else a multiple of 16): every contribution of every
 * chunk is copied device -> host on d2h_stream (one cudaMemcpyAsync per
 * contribution and chunk), n_threads host threads (0 = all cores) step each
 * chunk as soon as its copies have landed, and each finished chunk's fp16
 * parameters are copied host -> device on h2d_stream while later chunks are
 * still crossing or being stepped.  Pass two different streams so both link
 * directions run at once.  Arithmetic, ping-pong, overflow test and restore as
 * zero_shard_step_cpu, bit for bit; after an overflow the fp16 slice is sent
 * again from the kept master weights.  Synchronous: on return the device slice
 * holds the step's (or, after an overflow, the kept) parameters, and
 * *overflow_out (HOST) gets 0 or 1; the caller commits as for zero_shard_step.
 * Link bytes per step: 2 n_d n device -> host and 2 n host -> device (2 n more
 * after an overflow).  ZS_ERR_ARG for a bad argument or staging memory that is
 * not page-locked (text in zero_last_error()); ZS_ERR_CUDA for a failed copy
 * or event.
 * Source: "DeepSpeed ZeRO Stages", sec. 5.1 (ZeRO-Offload: optimizer state and
 * step on the CPU, transfers overlapped); "DeepSpeed ZeRO: Extreme Memory
 * Efficiency", "Offloading the optimizer entirely: ZeRO-Offload" (fp16
 * gradients down and fp16 parameters up each step, 4 Psi bytes at N_d = 1). */
ZS_API int32_t zero_shard_step_offload(const zs_offload_shard* shard, int32_t n_d, const zs_adam* hp,
                                       double loss_scale, int64_t step, int32_t cur, int32_t n_threads,
                                       int64_t chunk, void* d2h_stream, void* h2d_stream,
                                       int32_t* overflow_out);

/* ------------------------------------------------------------------------ */
/* Quantized weights (qwZ) on their own.                                     */
/* ------------------------------------------------------------------------ */

/* codes / scales (DEVICE) of n fp16 params (DEVICE), by the rule of
 * zs_shard.qcodes.  Stream-ordered.
 * Source: "ZeRO Optimization: Stages 1, 2, and 3 Explained" (ZeRO++ quantized weights); "DeepSpeed
 * ZeRO Stages", sec. 5.3. */
ZS_API int32_t zero_qwz_quantize(const uint16_t* params_dev, int64_t n, int8_t* codes_dev,
                                 float* scales_dev, void* stream);
/* The all-gather receiver's side: params[j] = fp16_rn(codes[j] * scales[j / 256])
 * (DEVICE buffers).  Stream-ordered.
 * Source: "ZeRO Optimization: Stages 1, 2, and 3 Explained" (ZeRO++ quantized weights); "DeepSpeed
 * ZeRO Stages", sec. 5.3. */
ZS_API int32_t zero_qwz_dequantize(const int8_t* codes_dev, const float* scales_dev, int64_t n,
                                   uint16_t* params_dev, void* stream);

/* ------------------------------------------------------------------------ */
/* Diagnostics.                                                              */
/* ------------------------------------------------------------------------ */

/* Static description of a status code.
 * Source: no counterpart in the pages (a property of this library). */
ZS_API const char* zero_status_string(int32_t status);
/* Text of the last ZS_ERR_CUDA failure on the calling host thread ("" if none).
 * Source: no counterpart in the pages (a property of this library). */
ZS_API const char* zero_last_error(void);
/* Number of kernels this library has enqueued in this process.
 * Source: no counterpart in the pages (a property of this library). */
ZS_API int64_t zero_kernel_launches(void);

/* Index checks of the debug build.  The same sources compiled with
 * ZS_CHECKED=1 give libzeroshard_checked.so, whose kernels test every element
 * range they are about to touch against the extent the call was given (the
 * shard's n, or its qwZ block count); a failed test records the first failure
 * -- (site << 48) | first element, site 1-9 naming the kernel and access --
 * and skips the access instead of trapping.  This call synchronises the
 * device, writes that record (0: none) to *first_fault, clears it, and
 * returns 1 in the checked build; the ordinary build has no checks and
 * returns 0 with *first_fault = 0.  ZS_ERR_ARG if first_fault is NULL,
 * ZS_ERR_CUDA if the record cannot be read.
 * Source: no counterpart in the pages (a property of this library). */
ZS_API int32_t zero_debug_checks(uint64_t* first_fault);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_SHARD_H_ */
