// device.cuh — device-side building blocks of the MoE step (sm_103a).
//
// mbarrier / bulk-copy (TMA) wrappers, bounded waits, the global timer, and
// the number formats of the step: bf16, FP8 E4M3, UE8M0 scales, MXFP8 group-32
// quantisation, and the binary32 exponential used for the combine weights.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ------------------------------------------------------------------ timers

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint64_t sm_cycles() { return clock64(); }

// First device-side error wins; later ones are dropped. Returns true for the winner.
__device__ __forceinline__ bool report_error(int32_t *status, int32_t code) {
  return atomicCAS(status, (int32_t)MOE_OK, code) == (int32_t)MOE_OK;
}

// A bounded wait gives up only when both the global timer and the SM cycle
// counter say the limit has passed. The cycle test assumes at least 1 GHz, so
// a forward jump of the global timer alone cannot end a wait early. A stalled
// global timer cannot stretch a wait past 4x the limit in cycles.
struct WaitClock {
  uint64_t t0, c0;
  __device__ __forceinline__ WaitClock() : t0(global_ns()), c0(sm_cycles()) {}
  __device__ __forceinline__ bool expired(int64_t limit_ns) const {
    const int64_t dc = (int64_t)(sm_cycles() - c0);
    const int64_t dt = (int64_t)(global_ns() - t0);
    return (dt > limit_ns && dc > limit_ns) || dc > 4 * limit_ns;
  }
  __device__ __forceinline__ int64_t ns() const { return (int64_t)(global_ns() - t0); }
  __device__ __forceinline__ int64_t cycles() const { return (int64_t)(sm_cycles() - c0); }
};

// Diagnostic record of the first device-side error of a step (plan-owned, 8 words):
// site, unit, tile, observed, expected, elapsed ns, elapsed cycles, block.
enum DiagSite : int64_t { kDiagReadyWait = 1, kDiagFullWait = 2, kDiagEmptyWait = 3, kDiagRoute = 4, kDiagQueueWait = 5,
                          kDiagBounds = 6 };

__device__ __forceinline__ void report_diag(int32_t *status, int64_t *diag, int32_t code, int64_t site, int64_t unit,
                                            int64_t tile, int64_t observed, int64_t expected, int64_t ns,
                                            int64_t cycles) {
  if (report_error(status, code) && diag) {
    diag[0] = site;
    diag[1] = unit;
    diag[2] = tile;
    diag[3] = observed;
    diag[4] = expected;
    diag[5] = ns;
    diag[6] = cycles;
    diag[7] = blockIdx.x;
  }
}

// ------------------------------------------------------------------ bounds checks
// Built with -DMOE_DEBUG_BOUNDS (libmoe_debug.so), every global and shared
// index the kernels compute is checked before its access: in_bounds(i, n)
// is true when 0 <= i < n; otherwise it records MOE_ERR_DEVICE_BOUNDS with a
// diagnostics record (site kDiagBounds, the check's id, the index, the limit)
// and returns false, and the caller skips the access. No check traps. In the
// normal build in_bounds is the constant true and adds no code.
#ifdef MOE_DEBUG_BOUNDS
constexpr bool kBoundsChecked = true;
#else
constexpr bool kBoundsChecked = false;
#endif

__device__ __forceinline__ bool in_bounds(int32_t *status, int64_t *diag, int check, int64_t i, int64_t n) {
  if constexpr (kBoundsChecked) {
    if (i < 0 || i >= n) {
      report_diag(status, diag, MOE_ERR_DEVICE_BOUNDS, kDiagBounds, check, -1, i, n, 0, 0);
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// One try_wait. The thread sleeps in hardware until the phase completes or
// about suspend_ns have passed, so waiting warps do not take issue slots
// from working ones.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity, uint32_t suspend_ns = 20000) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Gives up after
// timeout_ns (see WaitClock) and returns false; the caller reports MOE_ERR_TIMEOUT.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int64_t timeout_ns,
                                         int64_t *waited_ns = nullptr) {
  // try_wait suspends the thread on its own; poll it a few times before
  // reading the clocks.
#pragma unroll 1
  for (int i = 0; i < 4; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const WaitClock wc;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (wc.expired(timeout_ns)) {
      if (waited_ns) *waited_ns = wc.ns();
      return false;
    }
  }
}

// ------------------------------------------------------------------ bulk copy (TMA, no tensor map)

// L2 policy for weights that are read once per step: evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// L2 policy for weights that later blocks read again (multi-tile experts).
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// global -> shared bulk copy; completion is counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------------ acquire / release on global counters

// Moves `bytes` (a multiple of 16, from a 16-byte aligned address) of global
// memory into L2 without waiting (an untiled bulk prefetch; no completion to track).
__device__ __forceinline__ void l2_prefetch_bulk(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile(const uint32_t *p) {
  return *reinterpret_cast<const volatile uint32_t *>(p);
}

// ------------------------------------------------------------------ Programmatic Dependent Launch

__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ formats

// 2^(code - 127) as a binary32. Code 0 is the subnormal 2^-127.
__device__ __forceinline__ float ue8m0_to_float(uint32_t code) {
  return code ? __uint_as_float(code << 23) : __uint_as_float(0x00400000u);
}

// Two E4M3 codes (low byte first) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2 *>(&h));
}

// Two E4M3 codes (low byte first) -> f16x2 bits (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  return *reinterpret_cast<uint32_t *>(&h);
}

// c + a.lo * b.lo + a.hi * b.hi with f16 operands and an fp32 accumulator, two
// fma.rn.f32.f16: each product is exact in fp32 and each step rounds once.
__device__ __forceinline__ float fma_f16x2_f32(uint32_t a2, uint32_t b2, float c) {
  asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\t"
      "mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(c)
      : "r"(a2), "r"(b2));
  return c;
}

// float -> E4M3, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint8_t float_to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t *>(&b);
}

// OCP MX v1.0 shared-scale rule for E4M3 elements:
//   code = clamp(floor(log2 amax) - 8 + 127, 0, 254), amax = 0 -> 0.
// floor(log2 amax) is read from the binary32 exponent field (or, for a
// subnormal amax, from the position of its leading mantissa bit).
__device__ __forceinline__ uint32_t mx_scale_code(float amax) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (b == 0) return 0;
  const int ef = int(b >> 23);
  const int fl = ef ? ef - 127 : (31 - __clz(int(b & 0x7FFFFFu))) - 149;
  int c = fl - 8 + 127;
  c = c < 0 ? 0 : (c > 254 ? 254 : c);
  return uint32_t(c);
}

// The same rule for an element type whose largest normal has exponent emax
// (2 for E2M1): code = clamp(floor(log2 amax) - emax + 127, 0, 254).
__device__ __forceinline__ uint32_t mx_scale_code_emax(float amax, int emax) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (b == 0) return 0;
  const int ef = int(b >> 23);
  const int fl = ef ? ef - 127 : (31 - __clz(int(b & 0x7FFFFFu))) - 149;
  int c = fl - emax + 127;
  c = c < 0 ? 0 : (c > 254 ? 254 : c);
  return uint32_t(c);
}

// Two floats -> two E2M1 codes in one byte (a in the low nibble), round to
// nearest even, saturating at +-6.
__device__ __forceinline__ uint8_t float2_to_e2m1x2(float a, float b) {
  return static_cast<uint8_t>(__nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest));
}

// v * 2^(127 - code). The product is exact whenever it lies in the binary32
// normal range. Anything smaller rounds to zero in E4M3 anyway.
__device__ __forceinline__ float mx_unscale(float v, uint32_t code) {
  const int s = 127 - int(code);
  if (s >= -126) return __fmul_rn(v, __uint_as_float(uint32_t(s + 127) << 23));
  return __fmul_rn(__fmul_rn(v, 0x1p-64f), 0x1p-63f);
}

// ------------------------------------------------------------------ binary32 exponential
// Cody-Waite argument reduction with ln2 split into a 16-bit hi part (n*hi is
// exact for |n| < 2^8) and a lo part; a degree-8 Taylor polynomial by Horner;
// scaling by 2^n. Every step is one correctly rounded binary32 operation (no
// contraction into FMA). The constants are the correctly rounded binary32
// values of log2(e), ln2 - hi and 1/i!.
__device__ __forceinline__ float exp_rn(float x) {
  const float kLog2e = __uint_as_float(0x3fb8aa3bu);
  const float kLn2Hi = __uint_as_float(0x3f317200u);  // 45426 / 65536
  const float kLn2Lo = __uint_as_float(0x35bfbe8eu);
  const float kInvFact[9] = {
      __uint_as_float(0x3f800000u), __uint_as_float(0x3f800000u), __uint_as_float(0x3f000000u),
      __uint_as_float(0x3e2aaaabu), __uint_as_float(0x3d2aaaabu), __uint_as_float(0x3c088889u),
      __uint_as_float(0x3ab60b61u), __uint_as_float(0x39500d01u), __uint_as_float(0x37d00d01u)};
  const float n = rintf(__fmul_rn(x, kLog2e));
  float r = __fsub_rn(x, __fmul_rn(n, kLn2Hi));
  r = __fsub_rn(r, __fmul_rn(n, kLn2Lo));
  float p = kInvFact[8];
#pragma unroll
  for (int i = 7; i >= 0; --i) p = __fadd_rn(kInvFact[i], __fmul_rn(r, p));
  const int ni = int(n);
  if (ni >= -126) return __fmul_rn(p, __uint_as_float(uint32_t(ni + 127) << 23));
  if (ni >= -150) return __fmul_rn(__fmul_rn(p, __uint_as_float(uint32_t(ni + 64 + 127) << 23)), 0x1p-64f);
  return 0.0f;
}

}  // namespace moe
