// combine.cu — weighted combine of the expert outputs, plus the shared expert.
//
// y[t][h] = bf16_rne( ((w[t][0]*o[t*k][h] + w[t][1]*o[t*k+1][h]) + ...) + o_shared[t][h] )
// in binary32, in rank order, with no contraction into FMA. Given the same o
// and w, the result is the same bits on every run.
// Source: "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", section
// 2.1. The weighted reduction of expert outputs is fused with the
// shared-expert addition. The cross-GPU all-reduce that follows it there has
// no counterpart on one GPU.
#include <stdint.h>

#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

// One thread per 8 consecutive outputs of a row (two float4 loads per expert slot).
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  pdl_wait_primary();
  const int per_row = a.H / 8;
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= int64_t(a.T) * per_row) return;
  const int t = int(idx / per_row);
  const int h0 = int(idx % per_row) * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  for (int j = 0; j < a.k; ++j) {
    const float w = __ldcg(a.topk_w + int64_t(t) * a.k + j);
    const float4 *src = reinterpret_cast<const float4 *>(a.o + (int64_t(t) * a.k + j) * a.H + h0);
    const float4 v0 = __ldcs(src), v1 = __ldcs(src + 1);
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = j == 0 ? __fmul_rn(w, v[i]) : __fadd_rn(acc[i], __fmul_rn(w, v[i]));
  }
  if (a.shared) {
    const float4 *src = reinterpret_cast<const float4 *>(a.o + (int64_t(a.T) * a.k + t) * a.H + h0);
    const float4 v0 = __ldcs(src), v1 = __ldcs(src + 1);
    const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], v[i]);
  }
  uint32_t packed[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    packed[i] = uint32_t(float_to_bf16_bits(acc[2 * i])) | (uint32_t(float_to_bf16_bits(acc[2 * i + 1])) << 16);
  *reinterpret_cast<uint4 *>(a.y + int64_t(t) * a.H + h0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t st) {
  const int64_t threads = int64_t(a.T) * (a.H / 8);
  if (threads == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((threads + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

}  // namespace moe
