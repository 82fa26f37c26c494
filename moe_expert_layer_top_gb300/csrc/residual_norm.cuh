// residual_norm.cuh — the epilogue behind the MoE step, fused into the
// tensor-core expert kernel's combine.
//
// For each token row t with S residual streams (S <= 4):
//   new_s = sum_s' res[s][s'] * stream_s' + post[s] * y     binary32, stored as bf16
//   u     = sum_s pre[s] * new_s                            binary32
//   z     = bf16( (u * r) * gamma ),  r = 1 / sqrt(mean_h(u^2) + eps)
//   zq, zs = MXFP8 of z along H (groups of 32)
// Source: "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", section
// 2.1. The MoE kernels fuse the mHC output combination, the next layer's input
// combination and normalisation; the four-stream combination is fused with
// RMSNorm and quantisation; RMSNorm is fused with MXFP8 quantisation.
//
// Two parts:
//  1. residual_block: run by the warp that has just combined y for one
//     128-column block of row t. It writes the new streams and u for those
//     columns, plus the block's sum of u^2.
//  2. norm_row: the warp that completes the row's last block (a counter per
//     row) sums the blocks' partial sums in block order, then normalises and
//     quantises the whole row, one 32-group per lane.
// No warp waits for another: the counter decides which warp finishes the row.
// Every sum has a fixed order, so the results are the same on every run.
#pragma once

#include <stdint.h>

#include "device.cuh"
#include "internal.h"

namespace moe {

// Part 2: normalise and quantise row t (H columns, nblk blocks of partial sums).
__device__ __noinline__ void norm_row(const ExpertArgs &a, int t, int H, int nblk, int lane) {
  // sum of u^2 over the row: lane-strided block sums, then a butterfly
  float ss = 0.0f;
  for (int b = lane; b < nblk; b += 32) ss = __fadd_rn(ss, __ldcg(a.ss_part + int64_t(t) * nblk + b));
#pragma unroll
  for (int off = 16; off; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, off));
  const float ms = __fdiv_rn(ss, float(H));
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.rms_eps)));
  const int groups = H / kGroup;
  for (int g = lane; g < groups; g += 32) {
    const float4 *u4 = reinterpret_cast<const float4 *>(a.u_buf + int64_t(t) * H + int64_t(g) * kGroup);
    const uint4 *g4 = reinterpret_cast<const uint4 *>(a.norm_w + int64_t(g) * kGroup);
    float z[32];
    uint32_t zb[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 gw = __ldg(g4 + i);
      const float4 ua = __ldcg(u4 + 2 * i), ub = __ldcg(u4 + 2 * i + 1);
      const float uu[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
      const uint32_t gg[4] = {gw.x, gw.y, gw.z, gw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float g0 = __uint_as_float(gg[j] << 16), g1 = __uint_as_float(gg[j] & 0xFFFF0000u);
        const uint16_t b0 = float_to_bf16_bits(__fmul_rn(__fmul_rn(uu[2 * j], r), g0));
        const uint16_t b1 = float_to_bf16_bits(__fmul_rn(__fmul_rn(uu[2 * j + 1], r), g1));
        zb[4 * i + j] = uint32_t(b0) | (uint32_t(b1) << 16);
        z[8 * i + 2 * j] = bf16_bits_to_float(b0);
        z[8 * i + 2 * j + 1] = bf16_bits_to_float(b1);
        amax = fmaxf(amax, fmaxf(fabsf(z[8 * i + 2 * j]), fabsf(z[8 * i + 2 * j + 1])));
      }
    }
    const uint32_t code = mx_scale_code(amax);
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      q[i] = uint32_t(float_to_e4m3(mx_unscale(z[4 * i + 0], code))) |
             (uint32_t(float_to_e4m3(mx_unscale(z[4 * i + 1], code))) << 8) |
             (uint32_t(float_to_e4m3(mx_unscale(z[4 * i + 2], code))) << 16) |
             (uint32_t(float_to_e4m3(mx_unscale(z[4 * i + 3], code))) << 24);
    }
    uint4 *zq4 = reinterpret_cast<uint4 *>(a.zq + int64_t(t) * H + int64_t(g) * kGroup);
    zq4[0] = make_uint4(q[0], q[1], q[2], q[3]);
    zq4[1] = make_uint4(q[4], q[5], q[6], q[7]);
    a.zs[int64_t(t) * groups + g] = uint8_t(code);
    if (a.z_bf16) {
      uint4 *z4 = reinterpret_cast<uint4 *>(a.z_bf16 + int64_t(t) * H + int64_t(g) * kGroup);
#pragma unroll
      for (int i = 0; i < 4; ++i) z4[i] = make_uint4(zb[4 * i], zb[4 * i + 1], zb[4 * i + 2], zb[4 * i + 3]);
    }
  }
}

// Part 1, for the Q columns h0 + lane + 32 q of row t, whose combined y (bf16)
// the calling warp holds in yb. blk / nblk: this block and the row's block count.
template <int Q>
__device__ __forceinline__ void residual_block(const ExpertArgs &a, int t, int64_t h0, int blk, int nblk, int lane,
                                               const uint16_t (&yb)[Q]) {
  const int S = a.n_streams, H = a.H;
  float res[kMaxStreams][kMaxStreams], post[kMaxStreams], pre[kMaxStreams];
#pragma unroll
  for (int s = 0; s < kMaxStreams; ++s) {
    post[s] = (s < S && a.mix_post) ? __ldg(a.mix_post + int64_t(t) * S + s) : 1.0f;
    pre[s] = (s < S && a.mix_pre) ? __ldg(a.mix_pre + int64_t(t) * S + s) : 1.0f;
#pragma unroll
    for (int s2 = 0; s2 < kMaxStreams; ++s2)
      res[s][s2] = (s < S && s2 < S && a.mix_res) ? __ldg(a.mix_res + (int64_t(t) * S + s) * S + s2)
                                                  : (s == s2 ? 1.0f : 0.0f);
  }
  float ss = 0.0f;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int64_t h = h0 + lane + 32 * q;
    const float y = bf16_bits_to_float(yb[q]);
    float old[kMaxStreams];
#pragma unroll
    for (int s = 0; s < kMaxStreams; ++s)
      old[s] = s < S ? bf16_bits_to_float(a.resid_in[(int64_t(t) * S + s) * H + h]) : 0.0f;
    float u = 0.0f;
#pragma unroll
    for (int s = 0; s < kMaxStreams; ++s) {
      if (s >= S) break;
      // post * y, then the mixed streams in stream order (one rounding each)
      float v = __fmul_rn(post[s], y);
#pragma unroll
      for (int s2 = 0; s2 < kMaxStreams; ++s2)
        if (s2 < S) v = __fmaf_rn(res[s][s2], old[s2], v);
      const uint16_t nb = float_to_bf16_bits(v);
      a.resid_out[(int64_t(t) * S + s) * H + h] = nb;
      const float nf = bf16_bits_to_float(nb);
      u = (s == 0) ? __fmul_rn(pre[0], nf) : __fmaf_rn(pre[s], nf, u);
    }
    a.u_buf[int64_t(t) * H + h] = u;
    ss = __fmaf_rn(u, u, ss);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, off));
  if (lane == 0) a.ss_part[int64_t(t) * nblk + blk] = ss;
  // Count the block in: every lane fences its own stores, then one lane counts.
  __threadfence();
  __syncwarp();
  uint32_t before = 0;
  if (lane == 0) before = atomicAdd(a.row_cnt + t, 1u);
  before = __shfl_sync(0xFFFFFFFFu, before, 0);
  if (before == uint32_t(nblk - 1)) {
    __threadfence();  // the other blocks' u and partial sums, before they are read
    norm_row(a, t, H, nblk, lane);
  }
}

}  // namespace moe
