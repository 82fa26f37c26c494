/*
 * moe.h — C ABI of the GB300 small-batch MXFP8 MoE step.
 *
 * One decode MoE step of a DeepSeek-V4.1-Flash-style layer, on one GPU:
 *   router top-k + softmax weights
 *   -> sort-free placement of (token, expert) pairs into 8-row tiles
 *   -> MXFP8 quantisation of the token rows
 *   -> SwiGLU gate/up projection, bf16 intermediate, MXFP8 quantisation of h
 *   -> down projection
 *   -> weighted combine (+ an optional always-active shared expert).
 *
 * Passages that define the operation (page title, section):
 *  - "SGLang's Low-Latency Mode Boosts DeepSeek-V4.1-Flash Speed by 1.56x on
 *    AMD", "NVIDIA overlaps the dependency chain", bullet "Routing without
 *    sorting". Each expert's rows fit 8-row tiles, and a bitmap plus population
 *    counts place them with no scan or sort, keeping the top-k choices.
 *  - Same page, "Four stages keep megakernels outside core". The plugin
 *    contract is Register / Guard / Build / Runtime, and unsupported shapes
 *    fall back. Here:
 *      Register = loading this library and checking moe_abi_version();
 *      Guard + Build = moe_plan();
 *      Runtime = moe_forward();
 *      teardown = moe_destroy().
 *    The fallback is the caller's business: moe_plan and moe_forward return
 *    MOE_ERR_UNSUPPORTED, and this library has no CPU fallback.
 *  - "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", section 2.1:
 *      - group-32 FP8 weights and scales reorganised for Blackwell MXFP8;
 *      - MXFP8 activation quantisation fused into the producer;
 *      - the router emits the downstream layout;
 *      - the weighted reduction of expert outputs is fused with the
 *        shared-expert addition;
 *      - scratch buffers are reused across calls.
 *  - Same page, section 3.1. The MoE kernels fuse the clipped SwiGLU and keep
 *    the original intermediate rounding. Here g and u are rounded to bf16,
 *    and h = bf16(silu(g) * u) is then quantised to MXFP8. The clip limit is
 *    a config value (moe_config_t.swiglu_limit; 0 = no clip).
 *  - "FlyDSL Mono Kernels for High-Interactivity LLM Serving in ATOM",
 *    "MiniMax-M3: Connecting Attention and Experts". Each expert does an
 *    up/gate and a down projection, for the shared and the routed experts.
 *
 * Formats (OCP Microscaling Formats v1.0):
 *   E4M3 has bias 7, a largest finite value of 448 and NaN codes 0x7F/0xFF.
 *   A UE8M0 scale code c has value 2^(c - 127).
 *   The shared scale of a 32-group is 2^(floor(log2 amax) - 8), with the code
 *   clamped to [0, 254]; amax = 0 gives code 0. Elements are rounded to
 *   nearest-even and saturate at +-448.
 *
 * Conventions shared by every entry point:
 *  - Every call returns a moe_status_t. None aborts, exits or traps. An
 *    out-parameter is written only on MOE_OK.
 *  - Device pointers are CUDA device memory on the plan's device, owned by the
 *    caller, 16-byte aligned unless stated otherwise. Rows are contiguous
 *    (row stride = row length).
 *  - `cuda_stream` is a cudaStream_t (NULL = the legacy default stream).
 *    Work is enqueued on it. Only moe_plan, moe_destroy, moe_forward_host and
 *    moe_kernel_times synchronise.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 3

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* NULL or misaligned pointer, a size out of range, T > max_rows */
  MOE_ERR_UNSUPPORTED = 2,   /* Guard: shape or device this library does not handle */
  MOE_ERR_CUDA = 3,          /* a CUDA runtime call failed */
  MOE_ERR_OOM = 4,           /* device memory for the plan could not be allocated */
  MOE_ERR_TIMEOUT = 5,       /* device side: a bounded wait gave up (reported through d_status) */
  MOE_ERR_DEVICE_BOUNDS = 6  /* device side: an index check failed; the access was skipped */
} moe_status_t;

/* moe_config_t.flags */
#define MOE_FLAG_TIMING (1u << 0)
/* Record CUDA events around the expert kernel of every moe_forward. Read the
 * times back with moe_kernel_times. Events are recorded on the launch stream. */

#define MOE_FLAG_PATH_GEMV (1u << 1)
#define MOE_FLAG_PATH_MMA (1u << 2)
/* Expert kernel selection. By default every step runs the tensor-core expert
 * kernel: block-scaled MXFP8 tcgen05 MMA, one MMA covering up to 16, 32, 64 or
 * 96 token rows of an expert (above 128 rows, and for MXFP4 weights at every
 * row count, each unit covers two 128-row weight blocks on one token tile), so
 * each expert's weights stream from HBM about once per step.
 * PATH_GEMV selects the CUDA-core GEMV expert kernel instead (8-row tiles;
 * an expert's weights stream once per tile). PATH_MMA pins the default.
 * Setting both is MOE_ERR_INVALID_ARG. Both kernels compute the same result
 * within the fp32 summation-order tolerance; routing, placement and every
 * MXFP8 quantisation of a given input are identical. */

#define MOE_FLAG_TEST_SKIP_READY (1u << 8)
/* Host-side fault injection for tests. The gate/up units of the first placed
 * tile (on the tensor-core kernel: chunk) never publish their ready count.
 * The down units of that tile then give
 * up after wait_timeout_ns, and MOE_ERR_TIMEOUT appears in *d_status; y is
 * undefined for that step. The GPU does not fault or hang, and the next
 * moe_forward on a plan without this flag is unaffected. */

#define MOE_FLAG_TEST_BOUNDS (1u << 9)
/* Test hook of the bounds-checked build (libmoe_debug.so, compiled with
 * -DMOE_DEBUG_BOUNDS): the expert kernel's checks see only half of the
 * combine counters the step uses (T rows x the kernel's blocks per row), so a
 * check trips at an index that is still inside the buffer, and the step
 * reports MOE_ERR_DEVICE_BOUNDS (site 6 in the
 * diagnostics). It shows the checks are live without any access out of
 * bounds; y is undefined for that step. No effect in the normal build. */

/* moe_config_t.weight_format */
#define MOE_WEIGHTS_MXFP8 0u  /* E4M3 elements, UE8M0 scale per 32 along K */
#define MOE_WEIGHTS_MXFP4 1u  /* E2M1 elements (two per byte, element 2i in the low nibble), UE8M0 per 32 */

typedef struct moe_config {
  int32_t hidden;        /* H: token width, the K of gate/up. A multiple of 128, 128..16384
                          * (the GEMV kernel and the static-scratch step: 512, 1024 or 4096). */
  int32_t intermediate;  /* I: expert width, the K of down. A multiple of 128, 128..16384
                          * (GEMV kernel: 256, 512 or 2048, paired with H as 512/256, 1024/512, 4096/2048). */
  int32_t num_experts;   /* E: routed experts, 1..1024 */
  int32_t top_k;         /* k: experts per token, 1..min(E, 32) */
  int32_t num_shared;    /* 0 or 1 always-active shared expert (weight 1.0 in the combine) */
  int32_t max_rows;      /* largest T a moe_forward on this plan may pass, 1..4096 */
  uint32_t flags;        /* MOE_FLAG_* */
  int64_t wait_timeout_ns; /* bound on every device-side wait; <= 0 selects 200 ms */
  uint32_t weight_format;  /* MOE_WEIGHTS_MXFP8 (0) or MOE_WEIGHTS_MXFP4 (tensor-core kernel only) */
  float swiglu_limit;      /* clipped SwiGLU: with L > 0, h = silu(min(g, L)) * clamp(u, -L, L),
                            * g and u taken after their bf16 rounding; <= 0: no clip.
                            * "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", 3.1
                            * (the pages do not give the limit). */
} moe_config_t;

/* Expert weights in the canonical layout: group-32 scales along K, K contiguous.
 * MXFP8:
 *   w_gate, w_up: E4M3 [E][I][H]     s_gate, s_up: UE8M0 [E][I][H/32]
 *   w_down:       E4M3 [E][H][I]     s_down:       UE8M0 [E][H][I/32]
 * MXFP4: the same with w_gate, w_up packed E2M1 [E][I][H/2] and w_down packed
 * E2M1 [E][H][I/2] (two codes per byte, element 2i in the low nibble); the
 * w_* pointers must then be 32-byte aligned.
 * The sh_* pointers are the same for one shared expert, without the E axis. They
 * must be NULL when num_shared == 0.
 * Ownership: the plan keeps these pointers. It does not copy the weights. They
 * must stay valid and unchanged until moe_destroy. */
typedef struct moe_weights {
  const uint8_t *w_gate, *s_gate, *w_up, *s_up, *w_down, *s_down;
  const uint8_t *sh_w_gate, *sh_s_gate, *sh_w_up, *sh_s_up, *sh_w_down, *sh_s_down;
} moe_weights_t;

/* Optional debug taps: device buffers that moe_forward fills with intermediate
 * results after the step (device-to-device copies on the same stream). Any
 * member may be NULL. A "pair" p is a (token t, slot j) choice, p = t*k + j;
 * the shared expert's pairs are p = T*k + t. P = T*k + T*num_shared.
 *   topk_ids int32 [T][k]  expert ids in rank order (descending logit, ties -> lower id)
 *   topk_w   fp32  [T][k]  softmax over the selected logits
 *   bitmap   uint32 [E][ceil(T/32)]  bit t of row e set iff token t chose expert e
 *   counts   int32 [E]     rows placed on each expert
 *   slot     int32 [T][k]  (e << 16) | rank, rank = tile*8 + row
 *   xq, xs   uint8 [T][H], [T][H/32]  MXFP8 token rows
 *   h_bf16   uint16 [P][I] SwiGLU output before quantisation (bf16 bits)
 *   hq, hs   uint8 [P][I], [P][I/32]  MXFP8 h
 *   o        fp32  [P][H]  expert outputs before the combine */
typedef struct moe_taps {
  int32_t *topk_ids;
  float *topk_w;
  uint32_t *bitmap;
  int32_t *counts;
  int32_t *slot;
  uint8_t *xq, *xs;
  uint16_t *h_bf16;
  uint8_t *hq, *hs;
  float *o;
} moe_taps_t;

/* Register: the ABI version this library implements (MOE_ABI_VERSION). */
int32_t moe_abi_version(void);

/* Human-readable name of a status code (a static string). */
const char *moe_status_string(moe_status_t status);

/* Guard + Build.
 * The Guard checks the config and the device and returns MOE_ERR_UNSUPPORTED
 * or MOE_ERR_INVALID_ARG before touching the device when a check fails. The
 * device must be compute capability 10.3 (sm_103).
 * The Build step allocates every scratch buffer for max_rows. moe_forward
 * allocates nothing. It also records the weight pointers.
 * Weight ownership: the plan does NOT copy or re-lay-out the weights. A plugin
 * Build that reorganises the weights would own a copy and let the caller free
 * its own; this one reads the caller's canonical K-major MXFP8/MXFP4 arrays in
 * place (the tensor-core kernel's TMA tensor maps are encoded over them here),
 * which saves a second copy of every expert (6.5 GB at E = 256, H = 4096,
 * I = 2048). So the caller must keep the weight buffers allocated and
 * unchanged until moe_destroy; changing them changes the next step's result,
 * and freeing them first is undefined.
 * On success *plan_out receives an opaque handle; on failure it is set to NULL.
 * The plan belongs to the device that is current at this call. */
moe_status_t moe_plan(const moe_config_t *config, const moe_weights_t *weights,
                      void *cuda_stream, void **plan_out);

/* Runtime: one MoE step over T token rows, enqueued on cuda_stream.
 *   x      device bf16 [T][H]   token rows (not aliased with y)
 *   logits device fp32 [T][E]   router logits (finite)
 *   y      device bf16 [T][H]   output: sum_j w[t][j] * expert_{ids[t][j]}(x[t]) (+ shared(x[t]))
 *   taps   optional debug outputs (NULL for none)
 *   d_status optional device int32. It is set to MOE_OK at the start of the
 *            step and to the first device-side error (MOE_ERR_TIMEOUT,
 *            MOE_ERR_DEVICE_BOUNDS) if one occurs. Read it after the stream
 *            has synchronised. NULL: errors go to a plan-owned word instead.
 * T = 0 is valid and enqueues nothing. T > max_rows returns MOE_ERR_INVALID_ARG.
 * The call allocates nothing and never synchronises. A plan serves one stream
 * at a time: calls on one plan must not overlap on the GPU. */
moe_status_t moe_forward(void *plan, const void *x, const float *logits, int32_t T,
                         void *y, const moe_taps_t *taps, int32_t *d_status,
                         void *cuda_stream);

/* Runtime with a device-side row count, for CUDA-graph capture and replay.
 * Same as moe_forward, except that the kernels read the step's T from
 * *d_T (device int32, 4-byte aligned) when they run, so one captured graph
 * serves any T in [0, max_rows]. x, logits and y are sized for max_rows
 * rows; rows at or past T are neither read nor written. A value outside
 * [0, max_rows] is clamped and MOE_ERR_DEVICE_BOUNDS is written to the
 * status word; T = 0 is an empty step. Always runs the tensor-core expert
 * kernel (MOE_ERR_UNSUPPORTED on a plan built with MOE_FLAG_PATH_GEMV) with
 * the chunk size for max_rows. No taps. Allocates nothing, does not
 * synchronise. Source: "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in
 * SGLang", section 3.1: lengths are read from GPU memory, so a replayed
 * CUDA graph uses the current length, and the work follows the actual
 * length rather than the capacity. */
moe_status_t moe_forward_dev(void *plan, const void *x, const float *logits, const int32_t *d_T, void *y,
                             int32_t *d_status, void *cuda_stream);

/* The steps on either side of the MoE step: the router projection fused into
 * the route kernel, and the residual-stream epilogue as one kernel launched
 * right behind the expert kernel with programmatic dependent launch (PDL).
 * Source: "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", section 2.1:
 *  - MoE bullet: the router produces the downstream layout directly; the
 *    kernels also fuse the mHC output combination, the next layer's input
 *    combination or normalisation, to cut intermediate writes;
 *  - mHC bullet: the weighted combination of the four residual streams is
 *    fused with RMSNorm in one kernel, with quantisation on supported paths;
 *  - small-operator bullet: RMSNorm is fused with MXFP8 quantisation;
 *  - communication bullet: PDL overlaps portions of adjacent kernels.
 *
 * In front (w_router set): the route kernel computes the router logits
 *   logits[t][e] = sum_h x[t][h] * w_router[e][h]
 * (bf16 operands, binary32 accumulation in a fixed order, no bias) before its
 * top-k. The top-k, the softmax weights and the placement then read these
 * logits.
 *
 * Behind (num_streams = S > 0): each token row carries S residual streams.
 * Once y is complete (bf16), the epilogue kernel computes, per row:
 *   new_s[t] = sum_s' mix_res[t][s][s'] * resid_in[t][s'] + mix_post[t][s] * y[t]
 *              (binary32, stored as bf16 in resid_out)
 *   u[t]     = sum_s mix_pre[t][s] * new_s[t]                  (binary32)
 *   z[t]     = bf16( u[t] * norm_weight / sqrt(mean_h(u[t]^2) + rms_eps) )
 *   zq, zs   = MXFP8 of z[t] along H (the rule used for x)
 * S = 1 with NULL coefficients is the plain residual add followed by RMSNorm.
 * The mixing coefficients are inputs; they are computed elsewhere.
 * y is still written. Fused steps run the tensor-core expert kernel only. */
typedef struct moe_fused_io {
  const void *w_router;     /* bf16 [E][H] router weight, or NULL: logits are given */
  const float *logits;      /* fp32 [T][E]. With w_router == NULL: the router logits (input,
                             * finite). With w_router set: NULL, or a buffer that receives
                             * the computed logits. */
  int32_t num_streams;      /* S: 0 (no epilogue; the members below are ignored) or 1..4 */
  const void *resid_in;     /* bf16 [T][S][H] residual streams before this layer's output */
  void *resid_out;          /* bf16 [T][S][H] new streams; may be resid_in (updated in place) */
  const float *mix_res;     /* fp32 [T][S][S] stream mixing, or NULL (identity); 4-byte aligned */
  const float *mix_post;    /* fp32 [T][S] weight of y in each stream, or NULL (all 1) */
  const float *mix_pre;     /* fp32 [T][S] next layer's input combination, or NULL (all 1) */
  const void *norm_weight;  /* bf16 [H] RMSNorm weight */
  float rms_eps;            /* RMSNorm epsilon, finite and >= 0 */
  uint8_t *zq;              /* E4M3 [T][H]: the next layer's quantised input */
  uint8_t *zs;              /* UE8M0 [T][H/32]; any alignment */
  void *z;                  /* optional bf16 [T][H]: z before quantisation (a tap), or NULL */
} moe_fused_io_t;

/* Runtime with the fused steps around the MoE step: as moe_forward, with the
 * router logits computed from w_router (or read from io->logits) and, with
 * io->num_streams > 0, the residual-stream epilogue above. Pointers follow
 * the conventions at the top of this file (16-byte aligned device memory)
 * unless stated in moe_fused_io_t. Returns MOE_ERR_UNSUPPORTED on a plan
 * built with MOE_FLAG_PATH_GEMV. Taps as for moe_forward. Allocates nothing,
 * does not synchronise. */
moe_status_t moe_forward_fused(void *plan, const void *x, int32_t T, const moe_fused_io_t *io, void *y,
                               const moe_taps_t *taps, int32_t *d_status, void *cuda_stream);

/* Runtime with host buffers: runs moe_forward on x and logits in host memory
 * and leaves y in host memory. It then synchronises cuda_stream and returns
 * the device-side status of the step. A buffer in pinned (page-locked) host
 * memory, 16-byte aligned, is read or written by the kernels in place over
 * the host link; any other buffer is copied through plan-owned device memory
 * (pageable memory works, with synchronous copies). The caller must not touch
 * the buffers until the call returns.
 * x_host: bf16 [T][H]; logits_host: fp32 [T][E]; y_host: bf16 [T][H]. */
moe_status_t moe_forward_host(void *plan, const void *x_host, const float *logits_host,
                              int32_t T, void *y_host, void *cuda_stream);

/* MXFP8 quantisation of bf16 rows along their last axis, groups of 32. This is
 * the same device routine moe_forward applies to x.
 *   x bf16 [rows][cols] (device), cols a multiple of 32
 *   q E4M3 [rows][cols] (device), s UE8M0 [rows][cols/32] (device)
 * This also prepares canonical MXFP8 weights from bf16 checkpoints: W_gate[e]
 * is [I][H], quantised along H. The pages' checkpoints are already group-32 FP8. */
moe_status_t moe_quantize_mxfp8(const void *x, int64_t rows, int32_t cols,
                                uint8_t *q, uint8_t *s, void *cuda_stream);

/* MXFP4 quantisation of bf16 rows along their last axis, groups of 32 (OCP MX
 * v1.0: scale 2^(floor(log2 amax) - 2), elements E2M1 rounded to nearest
 * even and clamped to +-6). Prepares MXFP4 expert weights from bf16.
 *   x bf16 [rows][cols] (device), cols a multiple of 32
 *   q packed E2M1 [rows][cols/2] (device), s UE8M0 [rows][cols/32] (device) */
moe_status_t moe_quantize_mxfp4(const void *x, int64_t rows, int32_t cols,
                                uint8_t *q, uint8_t *s, void *cuda_stream);

/* Timing read-back for plans built with MOE_FLAG_TIMING. Synchronises with
 * the recorded events. Returns the summed expert-kernel time in ms over the
 * moe_forward calls since the last reset, and the number of such calls; then
 * resets both. At most 4096 calls are recorded between two reads; later ones
 * are not timed. */
moe_status_t moe_kernel_times(void *plan, double *expert_ms_out, int32_t *launches_out);

/* Device-side status word of a plan (used when moe_forward got d_status ==
 * NULL). Synchronises the plan's device and then reads it. */
moe_status_t moe_plan_status(void *plan, int32_t *status_out);

/* Diagnostics of the last device-side error on this plan: 8 int64 words
 *   [0] site: 1 ready-counter wait, 2 pipeline full wait, 3 pipeline empty wait, 4 router,
 *       5 unit-queue wait (tensor-core expert kernel), 6 bounds check (only in the
 *       bounds-checked build, libmoe_debug.so)
 *   [1] work unit (site 6: the id of the check), [2] tile (or ring stage),
 *   [3] value observed (site 6: the index), [4] value expected (site 6: the limit),
 *   [5] ns waited, [6] SM cycles waited, [7] block index.
 * All zero when the last step had no device-side error. Synchronises the device. */
moe_status_t moe_plan_diagnostics(void *plan, int64_t *out8);

/* Size of the fixed device array used by moe_forward_static_scratch. */
#define MOE_STATIC_SCRATCH_BYTES (8u << 20)

/* A MoE step that allocates nothing, for callers that cannot call cudaMalloc
 * where they run the step. Examples:
 *  - a server whose allocator has already reserved nearly all device memory;
 *  - code that must avoid the synchronisation and latency of cudaMalloc/cudaFree;
 *  - a plugin that is only handed its input and output buffers.
 * It runs the same kernels as moe_forward (always the CUDA-core GEMV expert
 * kernel; the path flags are ignored), with every intermediate kept in a
 * fixed device array of MOE_STATIC_SCRATCH_BYTES compiled into this library.
 * Every GPU that loads the library holds that array until the process exits.
 * There is no plan: the config and weights are passed on every call, as for
 * moe_plan (max_rows is ignored; T bounds the step).
 *   x, logits, y, d_status: as moe_forward (device memory, caller-owned).
 * Returns MOE_ERR_UNSUPPORTED, before any device work, when the step's
 * scratch (about T * (k*(4H + 1.03 I) + 1.03 H + 4(E+1)) bytes) exceeds
 * MOE_STATIC_SCRATCH_BYTES. At H = 4096, I = 2048, E = 256, k = 8 that is
 * about 50 rows. It also returns the Guard's errors, as moe_plan does.
 * Every call uses the same array. Calls that overlap on the GPU (two streams,
 * or two host threads) race and corrupt each other's results. Everything that
 * must start at zero is cleared by the step itself, except one counter at the
 * start of the array that every completed step leaves at zero.
 * The first call on a device checks the device (with that device current)
 * and may load this library's device code: make it before any stream capture.
 * Every call looks up the array's device address (cudaGetSymbolAddress) and
 * sets the two kernels' shared-memory limits (cudaFuncSetAttribute), with the
 * device current; both are host-side and allocate nothing, so a
 * cudaDeviceReset leaves no stale address behind.
 * d_status NULL: the step's status is written into the array, and no call
 * reads it back, so device-side errors (MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_BOUNDS)
 * are then lost. Pass d_status to see them.
 * The pages have no counterpart to this entry point. */
moe_status_t moe_forward_static_scratch(const moe_config_t *config, const moe_weights_t *weights, const void *x,
                                        const float *logits, int32_t T, void *y, int32_t *d_status,
                                        void *cuda_stream);

/* Teardown: frees the plan's device memory and events, after a device-wide
 * synchronise. NULL is a no-op. */
moe_status_t moe_destroy(void *plan);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
