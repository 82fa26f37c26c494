// combine.cuh — the weighted combine of one token row over one block of H, run
// by one warp inside an expert kernel.
//
// y[t][h] = bf16( ((w_0*o_0 + w_1*o_1) + ... + w_{k-1}*o_{k-1}) + o_shared )
// in binary32, rank order, each product and sum rounded once (no FMA
// contraction), then round to nearest even to bf16.
// Source: "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", 2.1. The
// weighted reduction of expert outputs is fused with the shared-expert addition.
//
// o rows are pair-indexed: routed pair t*k + j, shared pair T*k + t. The o
// values were written by other blocks of the same grid, so every load goes
// through L2 (the caller has already ordered them with a counter and fences).
#pragma once

#include <stdint.h>

#include "device.cuh"

namespace moe {

// Q outputs per lane: h = h0 + lane + 32 q, q < Q (a block of 32 Q rows of H).
// yb receives the lane's bf16 results as well.
template <int Q>
__device__ __forceinline__ void combine_row_block(const float *__restrict__ o, const float *__restrict__ topk_w,
                                                  uint16_t *__restrict__ y, int T, int k, int shared, int H, int t,
                                                  int64_t h0, int lane, uint16_t (&yb)[Q]) {
  const int64_t hl = h0 + lane;
  float acc[Q], sv[Q];
#pragma unroll
  for (int q = 0; q < Q; ++q) acc[q] = 0.0f;
  // the shared expert's row and the routed pairs in chunks of 8: all loads of
  // a chunk (and the shared row) are in flight together
  if (shared) {
    const float *src = o + (int64_t(T) * k + t) * H + hl;
#pragma unroll
    for (int q = 0; q < Q; ++q) sv[q] = __ldcg(src + 32 * q);
  }
  for (int j0 = 0; j0 < k; j0 += 8) {
    float w[8], v[8][Q];
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int j = j0 + jj < k ? j0 + jj : k - 1;
      w[jj] = __ldcg(topk_w + int64_t(t) * k + j);
      const float *src = o + (int64_t(t) * k + j) * H + hl;
#pragma unroll
      for (int q = 0; q < Q; ++q) v[jj][q] = __ldcg(src + 32 * q);
    }
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      if (j0 + jj >= k) break;
#pragma unroll
      for (int q = 0; q < Q; ++q)
        acc[q] = (j0 + jj == 0) ? __fmul_rn(w[jj], v[jj][q]) : __fadd_rn(acc[q], __fmul_rn(w[jj], v[jj][q]));
    }
  }
  if (shared) {
#pragma unroll
    for (int q = 0; q < Q; ++q) acc[q] = __fadd_rn(acc[q], sv[q]);
  }
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    yb[q] = float_to_bf16_bits(acc[q]);
    y[int64_t(t) * H + hl + 32 * q] = yb[q];
  }
}

}  // namespace moe
