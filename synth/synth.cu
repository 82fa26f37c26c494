// synth.cu — device implementation of the seeded input generator in synth/__init__.py.
//
// Same counter-based SplitMix64 (Steele, Lea, Flood 2014; Vigna's
// splitmix64.c) and the same approximately normal bf16 draw:
//   out_i = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
//   S     = sum of the four 16-bit fields of out_i
//   v     = float32(S - 131070) * c      (one binary32 multiply)
//   bf16  = v rounded to nearest-even
// The host passes key = mix64(seed * 0x9E3779B97F4A7C15 + stream) and c. This
// file draws numbers only; it holds none of the MoE method's arithmetic.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

__global__ void normal_bf16_kernel(uint64_t key, uint64_t start, uint64_t count, float c, uint16_t *out) {
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t i = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < count; i += stride) {
    const uint64_t h = mix64(key + (start + i + 1) * 0x9E3779B97F4A7C15ull);
    const int64_t s = int64_t(h & 0xFFFF) + int64_t((h >> 16) & 0xFFFF) + int64_t((h >> 32) & 0xFFFF) + int64_t(h >> 48);
    const float v = __fmul_rn(float(s - 131070), c);  // the int -> float conversion is exact (|.| < 2^24)
    const uint32_t u = __float_as_uint(v);
    out[i] = uint16_t((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
  }
}

}  // namespace

extern "C" {

// Draws count values, starting at counter index start, into out (device, bf16 bits).
// Returns 0 on success, else the cudaError_t of the launch.
int synth_normal_bf16(uint64_t key, uint64_t start, uint64_t count, float c_sigma, uint16_t *out, void *stream) {
  if (count == 0) return 0;
  uint64_t blocks = (count + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  normal_bf16_kernel<<<unsigned(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(key, start, count, c_sigma, out);
  return int(cudaGetLastError());
}

}  // extern "C"
