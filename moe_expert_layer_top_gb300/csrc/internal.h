// internal.h — plan layout and kernel launchers shared by the .cu files of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kTileRows = 8;            // rows per expert tile
constexpr int kGroup = 32;              // MXFP8 group along K
constexpr int kConsumerWarps = 16;      // expert kernel: compute warps
constexpr int kExpertThreads = (kConsumerWarps + 2) * 32;  // + one producer warp + one reducer warp
constexpr int kStageBytes = 32768;      // weight bytes per pipeline stage
constexpr int kStages = 5;              // pipeline depth
constexpr int kRouteThreads = 1024;     // route kernel: block 0 (router + placement)
constexpr int kQuantThreads = 256;      // route kernel: x-quantisation blocks (one group per thread)
constexpr int kMaxTimedCalls = 4096;
constexpr int kChunkRowsMax = 96;       // tensor-core expert kernel: most token rows per chunk (MMA N)
constexpr int kMmaDownRows = 128;       // tensor-core expert kernel: W_down rows per down unit
constexpr int kMmaMinRowsDefault = 1;   // steps with at least this many rows take the tensor-core kernel
constexpr int kRouterExperts = 8;       // route kernel: experts per router-projection block
constexpr size_t kRouteSmemMax = 200 * 1024;  // Guard: the route kernel's largest dynamic shared memory
constexpr int kMaxStreams = 4;          // residual streams per token row in the fused epilogue

// Device scratch and schedule of one plan (all sized for max_rows).
struct Scratch {
  int32_t *topk_ids;    // [Tmax][k]
  float *topk_w;        // [Tmax][k]
  uint32_t *bitmap;     // [E][words]
  int32_t *counts;      // [E + 1]    (index E: shared expert)
  int32_t *slot;        // [Tmax][k]
  int32_t *rows_of;     // [E + 1][Tmax] pair ids in rank order
  int32_t *tile_list;   // [n_tiles_max] (expert << 16) | tile
  int32_t *n_tiles;     // [1]
  int32_t *chunk_list;  // [n_tiles_max] (expert << 16) | chunk, chunks of <= mma_chunk_rows(T, H) rows
  int32_t *n_chunks;    // [1]
  uint32_t *ready;      // [n_tiles_max] gate/up units finished per tile (per chunk on the tensor-core path)
  uint32_t *comb_cnt;   // [Tmax][down blocks] down blocks of a token row finished (fused combine)
  uint32_t *work;       // [4] expert-kernel unit counter, abort flag, route-kernel ticket, (unused)
  int32_t *status;      // [1] plan-owned status word
  int64_t *diag;        // [8] first device-side error of the last step (site, unit, tile, ...)
  uint8_t *xq, *xs;     // [Tmax][H], [Tmax][H/32]
  uint8_t *hq, *hs;     // [P][I], [P][I/32]
  uint16_t *h_bf16;     // [P][I]
  float *o;             // [P][H]
  // fused steps (moe_forward_fused)
  float *logits_proj;   // [Tmax][E] router logits computed by the route kernel
  uint32_t *rg_cnt;     // [ceil(Tmax/32)] projection blocks finished per row group (zero between steps)
  // staging for moe_forward_host
  void *x_dev;
  float *logits_dev;
  void *y_dev;
};

// TMA tensor maps over the caller's weights (canonical layout, 128-byte swizzle),
// for the tensor-core expert kernel. Boxes: 128 bytes of K x 64 rows (gate, up)
// or x 128 rows (down, and gate/up of the two-block units).
struct MmaMaps {
  CUtensorMap gate, up, down;           // rows: E*I, E*I, E*H (boxes of 64, 64, 128 rows)
  CUtensorMap sh_gate, sh_up, sh_down;  // shared expert (zero when absent)
  CUtensorMap gate2, up2, sh_gate2, sh_up2;  // the same gate/up rows in boxes of 128 (two-block units)
};

struct Plan {
  moe_config_t cfg;
  moe_weights_t w;
  int device;
  int num_sms;
  int words;             // ceil(max_rows / 32)
  int n_tiles_max;       // upper bound on tiles in a step
  int64_t pairs_max;     // P for T = max_rows
  int comb_per_row_max;  // combine counters per token row (the larger of the two expert kernels' block counts)
  int64_t timeout_ns;
  int mma_min_rows;      // steps with T >= this take the tensor-core expert kernel
  MmaMaps maps;
  Scratch s;
  void *arena;           // single device allocation backing Scratch
  size_t arena_bytes;
  int32_t *status_host;  // pinned host word: the status of moe_forward_host's steps
  int32_t *status_mapped;  // the same word's device address (the kernels write it over the host link)
  // timing
  cudaEvent_t ev_start[kMaxTimedCalls];
  cudaEvent_t ev_stop[kMaxTimedCalls];
  int timed_calls;
  bool events_created;
};

struct RouteArgs {
  const float *logits;  // read by the top-k; with w_router set, the buffer the projection writes
  const uint16_t *x;
  const uint16_t *w_router;  // bf16 [E][H] router weight, or NULL (logits are an input)
  uint32_t *rg_cnt;          // per row group: projection blocks finished (w_router set)
  int n_eblk;                // projection blocks per row group: ceil(E / kRouterExperts)
  int T, H, E, k, shared, words, Tmax;  // T: the step's rows, or the grid's bound when d_T is set
  const int32_t *d_T;   // device-side row count (clamped to Tmax), or NULL
  int32_t *topk_ids;
  float *topk_w;
  uint32_t *bitmap;
  int32_t *counts;
  int32_t *slot;
  int32_t *rows_of;
  int32_t *tile_list;
  int32_t *n_tiles;
  int32_t *chunk_list;  // NULL: no chunk list (the GEMV expert kernel only)
  int32_t *n_chunks;
  int chunk_rows;       // rows per chunk (16, 32, 64 or 96)
  uint32_t *ready;
  int n_tiles_max;
  uint32_t *comb_cnt;
  int comb_per_row;     // combine counters per token row
  uint32_t *work;
  uint32_t *ticket;     // phase-2 ticket of the route grid (zero between steps)
  int32_t *status;
  int64_t *diag;
  uint8_t *xq, *xs;
};

struct ExpertArgs {
  const uint8_t *w_gate, *s_gate, *w_up, *s_up, *w_down, *s_down;
  const uint8_t *sh_w_gate, *sh_s_gate, *sh_w_up, *sh_s_up, *sh_w_down, *sh_s_down;
  int T, H, I, E, k, Tmax;
  const int32_t *d_T;   // device-side row count (tensor-core kernel only), or NULL
  const int32_t *counts;
  const int32_t *rows_of;
  const int32_t *tile_list;
  const int32_t *n_tiles;
  const int32_t *chunk_list;  // tensor-core kernel: chunks of <= mma_chunk_rows(T, H) rows per expert
  const int32_t *n_chunks;
  const uint8_t *xq, *xs;
  uint8_t *hq, *hs;
  uint16_t *h_bf16;  // NULL unless the h tap is requested
  float *o;
  uint32_t *ready;
  uint32_t *comb_cnt;       // per (token row, down block): arrivals of the row's k (+ shared) pairs
  const float *topk_w;      // combine weights [T][k]
  uint16_t *y;              // bf16 [T][H] output
  int shared;
  uint32_t *work;
  int32_t *status;
  int64_t *diag;
  int64_t timeout_ns;
  int skip_ready_tile;  // fault injection: tile index whose ready count is never published, or -1
  int fp4;              // weights are MXFP4 (E2M1) rather than MXFP8 (tensor-core kernel only)
  float swiglu_limit;   // clipped SwiGLU limit; <= 0: no clip
  // Capacities for the bounds checks of a -DMOE_DEBUG_BOUNDS build (unused otherwise):
  int n_tiles_max;      // entries of tile_list, chunk_list and ready
  int64_t pairs_cap;    // rows of hq, hs, h_bf16 and o
  int64_t comb_cap;     // entries of comb_cnt
};

// The residual-stream + RMSNorm + MXFP8 epilogue (residual_norm.cu), one block per token row.
struct ResidArgs {
  const uint16_t *y;         // bf16 [T][H], the step's output
  const uint16_t *resid_in;  // bf16 [T][S][H]
  uint16_t *resid_out;       // bf16 [T][S][H] (may equal resid_in)
  const float *mix_res, *mix_post, *mix_pre;  // [T][S][S], [T][S], [T][S] or NULL
  const uint16_t *norm_w;    // bf16 [H]
  float rms_eps;
  uint8_t *zq, *zs;          // [T][H], [T][H/32]
  uint16_t *z_bf16;          // [T][H] or NULL
  int T, H, S;
};

size_t route_smem_bytes(int E, int words);
cudaError_t prepare_residual_norm(int H);
cudaError_t launch_residual_norm(const ResidArgs &a, cudaStream_t st);
// Sets the route kernel's dynamic shared-memory limit to kRouteSmemMax. The
// limit is one per-function setting for the whole process, so it is never
// set lower: every plan and the static-scratch step work under it.
cudaError_t prepare_route();
cudaError_t prepare_experts(int H, int I);
cudaError_t launch_route(const RouteArgs &a, cudaStream_t st);
cudaError_t launch_quantize(const uint16_t *x, int64_t rows, int cols, uint8_t *q, uint8_t *s, cudaStream_t st);
cudaError_t launch_quantize_fp4(const uint16_t *x, int64_t rows, int cols, uint8_t *q, uint8_t *s, cudaStream_t st);
cudaError_t launch_experts(const ExpertArgs &a, int grid, cudaStream_t st);
int experts_down_blocks(int H, int I);  // H / DB: down units per tile
bool experts_shape_supported(int H, int I);
moe_status_t guard_host(const moe_config_t &c, const moe_weights_t &w);
// Tensor-core expert kernel (tcgen05 block-scaled MXFP8 MMA).
bool experts_mma_shape_supported(int H, int I);
bool encode_mma_maps(const moe_config_t &c, const moe_weights_t &w, MmaMaps *maps);
int mma_chunk_rows(int T, int H);
cudaError_t prepare_experts_mma();
cudaError_t launch_experts_mma(const MmaMaps &maps, const ExpertArgs &a, int grid, int chunk_rows, cudaStream_t st);

}  // namespace moe
