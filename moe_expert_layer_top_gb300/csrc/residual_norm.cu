// residual_norm.cu — the epilogue behind the MoE step, one kernel launched
// with programmatic dependent launch (PDL) right after the expert kernel.
//
// For each token row t with S residual streams (S <= 4):
//   new_s = sum_s' res[s][s'] * stream_s' + post[s] * y     binary32, stored as bf16
//   u     = sum_s pre[s] * new_s                            binary32
//   z     = bf16( (u * r) * gamma ),  r = 1 / sqrt(mean_h(u^2) + eps)
//   zq, zs = MXFP8 of z along H (groups of 32)
// Source: "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", section 2.1:
//  - mHC bullet: the weighted combination of the four residual streams and
//    RMSNorm run in one kernel, with quantisation on supported paths;
//  - small-operator bullet: RMSNorm is fused with MXFP8 quantisation;
//  - communication bullet: PDL overlaps portions of adjacent kernels.
//
// One block per token row and one 32-group per thread (looping when H/32
// exceeds the block). The output combination and u need no other thread.
// The row's sum of u^2 is a fixed-order block reduction: each thread in
// element order, then a butterfly in each warp, then the warps in order.
// u waits in shared memory for the reduction, stored transposed (element i of
// group g at i * groups + g) so a warp's accesses hit 32 banks. The block
// starts before the expert kernel ends (PDL), loads its coefficients and old
// streams, and waits for the expert kernel before reading y.
#include <stdint.h>

#include "device.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kNormThreadsMax = 256;

__global__ void __launch_bounds__(kNormThreadsMax) residual_norm_kernel(const ResidArgs a) {
  extern __shared__ float u_s[];  // [32][groups], transposed
  __shared__ float warp_ss[kNormThreadsMax / 32];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = a.S, H = a.H, groups = H / kGroup;
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

  // The old streams of this thread's first group do not depend on the expert
  // kernel: they are loaded before the wait.
  uint4 ov[kMaxStreams][4];
  const auto load_streams = [&](int g) {
#pragma unroll
    for (int s = 0; s < kMaxStreams; ++s) {
      if (s < S) {
        const uint4 *o4 = reinterpret_cast<const uint4 *>(a.resid_in + (int64_t(t) * S + s) * H + int64_t(g) * kGroup);
#pragma unroll
        for (int i = 0; i < 4; ++i) ov[s][i] = __ldcg(o4 + i);
      }
    }
  };
  if (tid < groups) load_streams(tid);
  pdl_wait_primary();  // the expert kernel's y is complete and visible

  float ss = 0.0f;
  for (int g = tid; g < groups; g += blockDim.x) {
    const int64_t c0 = int64_t(g) * kGroup;
    if (g != tid) load_streams(g);
    // y of this group (written by the previous kernel: read through L2)
    uint4 yv[4];
    const uint4 *y4 = reinterpret_cast<const uint4 *>(a.y + int64_t(t) * H + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) yv[i] = __ldcg(y4 + i);
    // 8 columns at a time: the new streams of those columns are stored as one vector each
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
      uint32_t nw[kMaxStreams][4];  // new streams, bf16 pairs
#pragma unroll
      for (int iw = 0; iw < 4; ++iw) {
        const int i = 4 * i4 + iw;
        const uint32_t yw = reinterpret_cast<const uint32_t *>(yv)[i];
        float u2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float y = h ? __uint_as_float(yw & 0xFFFF0000u) : __uint_as_float(yw << 16);
          float old[kMaxStreams];
#pragma unroll
          for (int s = 0; s < kMaxStreams; ++s) {
            const uint32_t w = s < S ? reinterpret_cast<const uint32_t *>(ov[s])[i] : 0u;
            old[s] = h ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
          }
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
            nw[s][iw] = h ? (nw[s][iw] | (uint32_t(nb) << 16)) : uint32_t(nb);
            const float nf = bf16_bits_to_float(nb);
            u = (s == 0) ? __fmul_rn(pre[0], nf) : __fmaf_rn(pre[s], nf, u);
          }
          u2[h] = u;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          u_s[(2 * i + h) * groups + g] = u2[h];
          ss = __fmaf_rn(u2[h], u2[h], ss);
        }
      }
#pragma unroll
      for (int s = 0; s < kMaxStreams; ++s)
        if (s < S)
          reinterpret_cast<uint4 *>(a.resid_out + (int64_t(t) * S + s) * H + c0)[i4] =
              make_uint4(nw[s][0], nw[s][1], nw[s][2], nw[s][3]);
    }
  }
  // sum of u^2 over the row, in a fixed order
#pragma unroll
  for (int off = 16; off; off >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, off));
  if (lane == 0) warp_ss[warp] = ss;
  __syncthreads();
  float tot = warp_ss[0];
  for (int w = 1; w < int(blockDim.x) / 32; ++w) tot = __fadd_rn(tot, warp_ss[w]);
  const float ms = __fdiv_rn(tot, float(H));
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, a.rms_eps)));

  for (int g = tid; g < groups; g += blockDim.x) {
    const int64_t c0 = int64_t(g) * kGroup;
    const uint4 *g4 = reinterpret_cast<const uint4 *>(a.norm_w + c0);
    float z[32];
    uint32_t zb[16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 gw = __ldg(g4 + i);
      const uint32_t gg[4] = {gw.x, gw.y, gw.z, gw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 8 * i + 2 * j;
        const uint16_t b0 = float_to_bf16_bits(__fmul_rn(__fmul_rn(u_s[e * groups + g], r), __uint_as_float(gg[j] << 16)));
        const uint16_t b1 =
            float_to_bf16_bits(__fmul_rn(__fmul_rn(u_s[(e + 1) * groups + g], r), __uint_as_float(gg[j] & 0xFFFF0000u)));
        zb[4 * i + j] = uint32_t(b0) | (uint32_t(b1) << 16);
        z[e] = bf16_bits_to_float(b0);
        z[e + 1] = bf16_bits_to_float(b1);
        amax = fmaxf(amax, fmaxf(fabsf(z[e]), fabsf(z[e + 1])));
      }
    }
    const uint32_t code = mx_scale_code(amax);
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      q[i] = uint32_t(float_to_e4m3(mx_unscale(z[4 * i + 0], code))) |
             (uint32_t(float_to_e4m3(mx_unscale(z[4 * i + 1], code))) << 8) |
             (uint32_t(float_to_e4m3(mx_unscale(z[4 * i + 2], code))) << 16) |
             (uint32_t(float_to_e4m3(mx_unscale(z[4 * i + 3], code))) << 24);
    uint4 *zq4 = reinterpret_cast<uint4 *>(a.zq + int64_t(t) * H + c0);
    zq4[0] = make_uint4(q[0], q[1], q[2], q[3]);
    zq4[1] = make_uint4(q[4], q[5], q[6], q[7]);
    a.zs[int64_t(t) * groups + g] = uint8_t(code);
    if (a.z_bf16) {
      uint4 *z4 = reinterpret_cast<uint4 *>(a.z_bf16 + int64_t(t) * H + c0);
#pragma unroll
      for (int i = 0; i < 4; ++i) z4[i] = make_uint4(zb[4 * i], zb[4 * i + 1], zb[4 * i + 2], zb[4 * i + 3]);
    }
  }
}

int norm_threads(int H) {
  const int groups = H / kGroup;
  const int t = (groups + 31) / 32 * 32;
  return t < kNormThreadsMax ? t : kNormThreadsMax;
}

}  // namespace

cudaError_t prepare_residual_norm(int H) {
  return cudaFuncSetAttribute(residual_norm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, H * 4);
}

cudaError_t launch_residual_norm(const ResidArgs &a, cudaStream_t st) {
  if (a.T <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(a.T));
  cfg.blockDim = dim3(unsigned(norm_threads(a.H)));
  cfg.dynamicSmemBytes = size_t(a.H) * 4;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, residual_norm_kernel, a);
}

}  // namespace moe
