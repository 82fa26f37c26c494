// route.cu — router top-k + combine weights, sort-free tile placement, and
// MXFP8 quantisation of the token rows, in one launch.
//
// Two phases in one grid:
//  1. ceil(T/32) routing blocks route their 32 token rows each, while the
//     other blocks quantise x.
//     - With a router weight W_r [E][H] (bf16), the logits are computed here
//       first: each row group has ceil(E/8) projection blocks, each for 8
//       experts. The last projection block of a row group to finish (a
//       ticket per row group) routes the group's rows. "Beyond Day-0:
//       Optimizing DeepSeek-V4.1 Flash in SGLang" 2.1: the router produces
//       the layout the downstream kernels need.
//     - Top-k per token row uses one warp per row, in k rounds of warp argmax.
//     - The combine weights are a softmax over the selected logits in
//       binary32, using exp_rn.
//  2. The last routing block to finish phase 1 places the pairs (it takes a
//     ticket after a fence; no block waits for another).
//     - Token bitmaps are built per expert in shared memory.
//     - Placement uses population counts: rank(t, e) = popc(bits of expert e
//       below t). Tile = rank / 8 and row = rank % 8.
// This follows "SGLang's Low-Latency Mode Boosts DeepSeek-V4.1-Flash Speed by
// 1.56x on AMD", "NVIDIA overlaps the dependency chain", bullet "Routing
// without sorting". A bitmap and population counts place the 8-row tiles with
// no scan or sort, keeping the top-k choices. It also follows "Beyond Day-0:
// Optimizing DeepSeek-V4.1 Flash in SGLang" 2.1: the router writes the layout
// the expert kernel consumes. That layout is:
//   rows_of[e][rank]   pair ids (t*k + j), in token order;
//   tile_list[]        (expert, tile) work items for the expert kernel;
//   chunk_list[]       (expert, chunk) items of <= 16..128 rows for the
//                      tensor-core expert kernel.
// The lists' per-expert offsets come from block-wide prefixes over the E+1
// tile (chunk) counts, the shared expert first, then the routed experts by id.
// That is work enumeration, not row placement.
//
// x is quantised to MXFP8 one 32-group per thread. "Beyond Day-0" 2.1 fuses
// activation quantisation into the producer, and here it shares the launch
// with the router.
#include <stdint.h>

#include "device.cuh"
#include "internal.h"

namespace moe {

// ------------------------------------------------------------------ MXFP8 group quantiser (shared by x and moe_quantize_mxfp8)

__device__ __forceinline__ void quantize_group32(const uint16_t *__restrict__ src, uint8_t *__restrict__ dst,
                                                 uint8_t *__restrict__ scale) {
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 r = __ldg(s4 + i);
    w[4 * i + 0] = r.x;
    w[4 * i + 1] = r.y;
    w[4 * i + 2] = r.z;
    w[4 * i + 3] = r.w;
  }
  float v[32];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
  }
  const uint32_t code = mx_scale_code(amax);
  uint32_t q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t b0 = float_to_e4m3(mx_unscale(v[4 * i + 0], code));
    uint32_t b1 = float_to_e4m3(mx_unscale(v[4 * i + 1], code));
    uint32_t b2 = float_to_e4m3(mx_unscale(v[4 * i + 2], code));
    uint32_t b3 = float_to_e4m3(mx_unscale(v[4 * i + 3], code));
    q[i] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
  }
  uint4 *d4 = reinterpret_cast<uint4 *>(dst);
  d4[0] = make_uint4(q[0], q[1], q[2], q[3]);
  d4[1] = make_uint4(q[4], q[5], q[6], q[7]);
  *scale = static_cast<uint8_t>(code);
}

// MXFP4 group quantiser (OCP MX v1.0): code = clamp(floor(log2 amax) - 2 + 127,
// 0, 254); elements E2M1, round to nearest even, saturating at +-6, two per
// byte with element 2i in the low nibble.
__device__ __forceinline__ void quantize_group32_fp4(const uint16_t *__restrict__ src, uint8_t *__restrict__ dst,
                                                     uint8_t *__restrict__ scale) {
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 r = __ldg(s4 + i);
    w[4 * i + 0] = r.x;
    w[4 * i + 1] = r.y;
    w[4 * i + 2] = r.z;
    w[4 * i + 3] = r.w;
  }
  float v[32];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
  }
  const uint32_t code = mx_scale_code_emax(amax, 2);
  uint32_t q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      word |= uint32_t(float2_to_e2m1x2(mx_unscale(v[8 * i + 2 * j], code), mx_unscale(v[8 * i + 2 * j + 1], code)))
              << (8 * j);
    q[i] = word;
  }
  *reinterpret_cast<uint4 *>(dst) = make_uint4(q[0], q[1], q[2], q[3]);
  *scale = static_cast<uint8_t>(code);
}

__global__ void __launch_bounds__(kQuantThreads) quantize_fp4_kernel(const uint16_t *__restrict__ x, int64_t groups,
                                                                     uint8_t *__restrict__ q, uint8_t *__restrict__ s) {
  for (int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; g < groups; g += int64_t(gridDim.x) * blockDim.x)
    quantize_group32_fp4(x + g * kGroup, q + g * (kGroup / 2), s + g);
}

__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(const uint16_t *__restrict__ x, int64_t groups,
                                                                 uint8_t *__restrict__ q, uint8_t *__restrict__ s) {
  for (int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; g < groups; g += int64_t(gridDim.x) * blockDim.x)
    quantize_group32(x + g * kGroup, q + g * kGroup, s + g);
}

// ------------------------------------------------------------------ router + placement (block 0)

struct RouteSmem {
  // followed in dynamic shared memory by uint32_t bitmap[E][words]
  int32_t sel_i[kRouteThreads / 32][32];
  float sel_v[kRouteThreads / 32][32];
  int32_t tiles[kRouteThreads];
  int32_t offs[kRouteThreads];
  int32_t warp_sums[kRouteThreads / 32];
  float part[4][kRouterExperts][32];  // router projection, <= 8 rows: [H quarter][expert][row] partial sums
  float part_mma[16][32][kRouterExperts];  // router projection, > 8 rows: [K slice][row][expert]
  int32_t last;  // this block finished phase 1 last
};

// One warp-level tensor-core product D[16x8] += A[16x16] * B[16x8]: bf16
// operands, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Router projection for a row group of more than 8 rows (up to 32: two
// 16-row tiles) and experts 8 eb .. 8 eb + 7, on the tensor cores.
// Warp w takes the row tile w % 2 and the K slice w / 2: 32-column blocks
// kb = slice, slice + 16, ... Within a 32-column block, lane (g, t) loads 8
// contiguous columns 8t .. 8t+7 of its two rows (g, g + 8) and of expert g.
// The two MMAs of the block take columns {8t .. 8t+3} and {8t+4 .. 8t+7} in
// the k positions (2t, 2t+1, 2t+8, 2t+9) of A and B alike. A permutation of k
// applied to both operands leaves the sum unchanged, and every load is one
// 16-byte vector. The 16 slices' partial sums are then added in slice order.
__device__ void router_block_mma(const RouteArgs &a, int T, int rg, int eb, RouteSmem &sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int mt = warp & 1, ks = warp >> 1;
  const int H = a.H, nkb = H / 32;
  const int t0 = rg * (kRouteThreads / 32);
  const int nrows = min(kRouteThreads / 32, T - t0);
  const int ra = mt * 16 + g, rb = ra + 8;  // this lane's two rows within the group
  const int e = eb * kRouterExperts + g;
  const bool va = ra < nrows, vb = rb < nrows, ve = e < a.E;
  const uint16_t *xa = a.x + int64_t(t0 + (va ? ra : 0)) * H + 8 * t4;
  const uint16_t *xb = a.x + int64_t(t0 + (vb ? rb : 0)) * H + 8 * t4;
  const uint16_t *wr = a.w_router + int64_t(ve ? e : 0) * H + 8 * t4;
  float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
  for (int kb = ks; kb < nkb; kb += 32) {
    // two 32-column blocks in flight: kb and kb + 16
    uint4 A0[2], B0[2], W0[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int k = kb + 16 * u;
      const bool in = k < nkb;
      A0[u] = (in && va) ? __ldg(reinterpret_cast<const uint4 *>(xa + 32 * k)) : z4;
      B0[u] = (in && vb) ? __ldg(reinterpret_cast<const uint4 *>(xb + 32 * k)) : z4;
      W0[u] = (in && ve) ? __ldg(reinterpret_cast<const uint4 *>(wr + 32 * k)) : z4;
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      mma_bf16_16816(d, A0[u].x, B0[u].x, A0[u].y, B0[u].y, W0[u].x, W0[u].y);
      mma_bf16_16816(d, A0[u].z, B0[u].z, A0[u].w, B0[u].w, W0[u].z, W0[u].w);
    }
  }
  // D: lane (g, t) holds rows (g, g + 8) of its tile, experts (2t, 2t + 1)
  sm.part_mma[ks][mt * 16 + g][2 * t4] = d[0];
  sm.part_mma[ks][mt * 16 + g][2 * t4 + 1] = d[1];
  sm.part_mma[ks][mt * 16 + g + 8][2 * t4] = d[2];
  sm.part_mma[ks][mt * 16 + g + 8][2 * t4 + 1] = d[3];
  __syncthreads();
  if (threadIdx.x < 32 * kRouterExperts) {
    const int r = threadIdx.x / kRouterExperts, es = threadIdx.x % kRouterExperts;
    const int e2 = eb * kRouterExperts + es;
    if (r < nrows && e2 < a.E) {
      float l = sm.part_mma[0][r][es];
#pragma unroll
      for (int s = 1; s < 16; ++s) l = __fadd_rn(l, sm.part_mma[s][r][es]);
      const_cast<float *>(a.logits)[int64_t(t0 + r) * a.E + e2] = l;
    }
  }
}

// Router projection for row group rg (rows 32 rg ..) and experts 8 eb .. 8 eb + 7:
// logits[t][e] = sum_h x[t][h] * W_r[e][h], bf16 operands, binary32 sums.
// Warp w takes expert 8 eb + w / 4 and the quarter w % 4 of H. Each lane
// accumulates 8 rows at a time over its 8-column vectors (one fused
// multiply-add per product, in column order); the warp then sums its lanes by
// a butterfly, and the four quarters are added in order. The order is fixed,
// so the logits are the same on every run.
__device__ void router_block(const RouteArgs &a, int T, int rg, int eb, RouteSmem &sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int es = warp >> 2, qq = warp & 3;
  const int e = eb * kRouterExperts + es;
  const int H = a.H, HQ = H / 4;
  const int t0 = rg * (kRouteThreads / 32);
  const int nrows = min(kRouteThreads / 32, T - t0);
  const uint16_t *wrow = a.w_router + int64_t(e < a.E ? e : 0) * H + qq * HQ;
  const uint16_t *xrow = a.x + int64_t(t0) * H + qq * HQ;
  for (int rb = 0; rb < nrows; rb += 8) {
    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.0f;
    // four W_r vectors in flight at a time, then their products with the rows
    for (int c0 = lane * 8; c0 < HQ; c0 += 256 * 4) {
      uint4 wv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + 256 * j;
        wv[j] = c < HQ ? __ldg(reinterpret_cast<const uint4 *>(wrow + c)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + 256 * j;
        if (c >= HQ) break;
        const uint32_t ww[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (rb + r < nrows) {
            const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(xrow + int64_t(rb + r) * H + c));
            const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc[r] = __fmaf_rn(__uint_as_float(xx[i] << 16), __uint_as_float(ww[i] << 16), acc[r]);
              acc[r] = __fmaf_rn(__uint_as_float(xx[i] & 0xFFFF0000u), __uint_as_float(ww[i] & 0xFFFF0000u), acc[r]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float v = acc[r];
#pragma unroll
      for (int off = 16; off; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
      if (lane == 0 && rb + r < 32) sm.part[qq][es][rb + r] = v;
    }
  }
  __syncthreads();
  if (threadIdx.x < kRouterExperts * 32) {
    const int es2 = threadIdx.x >> 5, r = threadIdx.x & 31;
    const int e2 = eb * kRouterExperts + es2;
    if (r < nrows && e2 < a.E) {
      const float l = __fadd_rn(__fadd_rn(__fadd_rn(sm.part[0][es2][r], sm.part[1][es2][r]), sm.part[2][es2][r]),
                                sm.part[3][es2][r]);
      const_cast<float *>(a.logits)[int64_t(t0 + r) * a.E + e2] = l;
    }
  }
}

// Top-k and combine weights, one warp per token row. Each lane keeps its NC
// candidates (lane, lane + 32, ...) in registers as the order-preserving bits
// of the logit, with a mask of the candidates not taken yet. A round takes the
// largest key in the warp (redux.sync max), then the lowest expert id that
// holds it (redux.sync min): the largest logit and, among equal logits, the
// lower id.
// bm: the block's bitmap in shared memory when one block routes every row
// (the bits are set here); NULL when the last block builds it in phase 2.
// rg: the row group (rows 32 rg .. 32 rg + 31, one per warp). The logits are
// read through L2: with a router weight they were written by other blocks of
// this grid.
template <int NC>
__device__ __forceinline__ void route_topk(const RouteArgs &a, int T, int rg, RouteSmem &sm, uint32_t *bm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, k = a.k, W = a.words;
  constexpr int kWarps = kRouteThreads / 32;
  {
    const int t = rg * kWarps + warp;
    if (t >= T) return;
    const float *row = a.logits + int64_t(t) * E;
    uint32_t ord[NC];
    uint32_t live = 0;  // bit j: candidate j (expert 32 j + lane) not taken yet
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const int i = j * 32 + lane;
      ord[j] = 0;
      if (i < E) {
        uint32_t b = __float_as_uint(__ldcg(row + i));
        // -0.0 and +0.0 compare equal: one key for both, so they tie to the lower id
        if (b == 0x80000000u) b = 0u;
        ord[j] = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
        live |= 1u << j;
      }
    }
    for (int r = 0; r < k; ++r) {
      uint32_t lmax = 0;
#pragma unroll
      for (int j = 0; j < NC; ++j)
        if ((live >> j) & 1u) lmax = ord[j] > lmax ? ord[j] : lmax;
      const uint32_t best = __reduce_max_sync(0xFFFFFFFFu, lmax);
      uint32_t lid = 0xFFFFFFFFu;  // this lane's lowest live id holding the best key
#pragma unroll
      for (int j = NC - 1; j >= 0; --j)
        if (((live >> j) & 1u) && ord[j] == best) lid = uint32_t(j * 32 + lane);
      const uint32_t uid = __reduce_min_sync(0xFFFFFFFFu, lid);
      const int id = int(uid);
      if (uid >= uint32_t(E)) report_error(a.status, MOE_ERR_DEVICE_BOUNDS);  // cannot happen for k <= E
      if (lid == uid) live &= ~(1u << (uid >> 5));  // taken (only the owning lane matches)
      if (lane == 0) {
        const uint32_t bits = (best & 0x80000000u) ? (best & 0x7FFFFFFFu) : ~best;
        sm.sel_i[warp][r] = uid < uint32_t(E) ? id : 0;
        sm.sel_v[warp][r] = __uint_as_float(bits);
      }
    }
    __syncwarp();
    // weights: e_j = exp_rn(l_j - l_0); s = ((e_0 + e_1) + ...) ; w_j = e_j / s
    float e = 0.0f;
    if (lane < k) e = exp_rn(__fsub_rn(sm.sel_v[warp][lane], sm.sel_v[warp][0]));
    float s = 0.0f;
    for (int j = 0; j < k; ++j) {
      const float ej = __shfl_sync(0xFFFFFFFFu, e, j);
      s = (j == 0) ? ej : __fadd_rn(s, ej);
    }
    if (lane < k) {
      const int id = sm.sel_i[warp][lane];
      a.topk_ids[int64_t(t) * k + lane] = id;
      a.topk_w[int64_t(t) * k + lane] = __fdiv_rn(e, s);
      if (bm && in_bounds(a.status, a.diag, 1, int64_t(id) * W + (t >> 5), int64_t(E) * W))
        atomicOr(&bm[id * W + (t >> 5)], 1u << (t & 31));
    }
    __syncwarp();
  }
}

// Exclusive prefix of v over the block's kRouteThreads threads, in thread
// order; *total gets the sum. Every thread of the block must call it.
__device__ __forceinline__ int block_exclusive_scan(RouteSmem &sm, int v, int &total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += u;
  }
  __syncthreads();  // an earlier scan's readers are done with warp_sums
  if (lane == 31) sm.warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int ws = sm.warp_sums[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xFFFFFFFFu, ws, off);
      if (lane >= off) ws += u;
    }
    sm.warp_sums[lane] = ws;  // inclusive
  }
  __syncthreads();
  total = sm.warp_sums[kRouteThreads / 32 - 1];
  return x - v + (warp ? sm.warp_sums[warp - 1] : 0);
}

// Phase 2 (one block): bitmaps, counts, work lists and placement of every pair.
// have_bitmap: phase 1 already set the bits in this block's shared memory.
__device__ void route_place(const RouteArgs &a, int T, RouteSmem &sm, uint32_t *bm, bool have_bitmap) {
  const int tid = threadIdx.x;
  const int E = a.E, k = a.k, W = a.words;

  if (!have_bitmap) {
    for (int i = tid; i < E * W; i += blockDim.x) bm[i] = 0;
    __syncthreads();
    // the selected experts were written by every block of phase 1: read through L2
    for (int p = tid; p < T * k; p += blockDim.x) {
      const int t = p / k;
      const int id = __ldcg(a.topk_ids + p);
      if (in_bounds(a.status, a.diag, 2, id, E) && in_bounds(a.status, a.diag, 3, t >> 5, W))
        atomicOr(&bm[id * W + (t >> 5)], 1u << (t & 31));
    }
  }
  __syncthreads();

  // --- counts and tiles per expert (index E: the shared expert, every row).
  // Thread p enumerates expert ex: the shared expert first, then the routed
  // experts by id. The expert kernels take units in this order, so the shared
  // expert, which completes the combine of every row it is the last
  // contribution to, runs first and not in the last wave of units.
  const int nexp = E + a.shared;
  const int ex = a.shared ? (tid == 0 ? E : tid - 1) : tid;
  int cnt = 0;
  if (tid < nexp) {
    if (ex < E) {
      cnt = 0;
      for (int w = 0; w < W; ++w) cnt += __popc(bm[ex * W + w]);
    } else {
      cnt = T;
    }
    a.counts[ex] = cnt;
    sm.tiles[tid] = (cnt + kTileRows - 1) / kTileRows;
  } else {
    sm.tiles[tid] = 0;
  }
  // Block-wide exclusive prefixes of the tile and chunk counts (work
  // enumeration for the expert kernels), in one scan of packed counts: each
  // total is at most T (k + 1) / 8 + E + 1 < 2^15 (T <= 4096, k <= 32,
  // E <= 1024), so the low half never carries into the high half.
  const int nch = (a.chunk_list && tid < nexp) ? (cnt + a.chunk_rows - 1) / a.chunk_rows : 0;
  int packed_total = 0;
  const int packed_excl = block_exclusive_scan(sm, sm.tiles[tid] | (nch << 16), packed_total);
  const int excl = packed_excl & 0xFFFF, total = packed_total & 0xFFFF;
  if (tid < nexp) {
    for (int j = 0; j < sm.tiles[tid]; ++j) {
      const int idx = excl + j;
      if (idx < a.n_tiles_max) a.tile_list[idx] = (ex << 16) | j;
      else report_error(a.status, MOE_ERR_DEVICE_BOUNDS);
    }
  }
  if (tid == 0) *a.n_tiles = min(total, a.n_tiles_max);

  // chunks of <= chunk_rows rows per expert, for the tensor-core expert kernel
  if (a.chunk_list) {
    const int cexcl = packed_excl >> 16, nch_total = packed_total >> 16;
    for (int j = 0; j < nch; ++j) {
      const int idx = cexcl + j;
      if (idx < a.n_tiles_max) a.chunk_list[idx] = (ex << 16) | j;
      else report_error(a.status, MOE_ERR_DEVICE_BOUNDS);
    }
    if (tid == 0) *a.n_chunks = min(nch_total, a.n_tiles_max);
  }

  // --- placement: rank by population count of lower token bits
  for (int p = tid; p < T * k; p += blockDim.x) {
    const int t = p / k;
    const int e = __ldcg(a.topk_ids + p);
    if (!in_bounds(a.status, a.diag, 2, e, E) || !in_bounds(a.status, a.diag, 3, t >> 5, W)) continue;
    const uint32_t *b = bm + e * W;
    int rank = __popc(b[t >> 5] & ((1u << (t & 31)) - 1u));
    for (int w = 0; w < (t >> 5); ++w) rank += __popc(b[w]);
    a.slot[p] = (e << 16) | rank;
    if (in_bounds(a.status, a.diag, 4, rank, a.Tmax)) a.rows_of[int64_t(e) * a.Tmax + rank] = p;
  }
  if (a.shared)
    for (int t = tid; t < T; t += blockDim.x) a.rows_of[int64_t(E) * a.Tmax + t] = T * k + t;
  for (int i = tid; i < E * W; i += blockDim.x) a.bitmap[i] = bm[i];
}

// Blocks [0, R) route R*32 token rows (R = ceil(T/32)); the blocks after them
// quantise x, one 32-group per thread.
__device__ __host__ __forceinline__ int route_blocks(int T) { return (T + kRouteThreads / 32 - 1) / (kRouteThreads / 32); }

__global__ void __launch_bounds__(kRouteThreads) route_kernel(const RouteArgs a) {
  extern __shared__ __align__(16) unsigned char route_smem[];
  // Let the expert kernel's blocks get scheduled early; it waits for this grid
  // before reading. Every block of this grid is running when it triggers, so
  // the expert kernel's blocks cannot take the SMs this grid still needs.
  pdl_launch_dependents();
  // This grid is itself launched behind the previous kernel on the stream
  // (programmatic dependent launch): its blocks get scheduled while that
  // kernel finishes. The router weight is a constant, so a projection block
  // moves its 8 rows of W_r towards L2 first; everything else waits here
  // for the previous kernel (x, the logits, and this plan's scratch that the
  // previous step's expert kernel may still read).
  if (a.w_router && !a.d_T && int(blockIdx.x) < route_blocks(a.T) * a.n_eblk) {
    const int e = (int(blockIdx.x) % a.n_eblk) * kRouterExperts + int(threadIdx.x);  // one W_r row per thread
    if (threadIdx.x < kRouterExperts && e < a.E) l2_prefetch_bulk(a.w_router + int64_t(e) * a.H, uint32_t(a.H) * 2u);
  }
  pdl_wait_primary();
  RouteSmem &sm = *reinterpret_cast<RouteSmem *>(route_smem);
  uint32_t *bm = reinterpret_cast<uint32_t *>(route_smem + sizeof(RouteSmem));
  const int tid = threadIdx.x;
  // The step's row count: a.T, or the value at a.d_T (clamped to the plan's
  // max_rows) when the step was enqueued with a device-side row count. The
  // grid is sized for a.T either way.
  int T = a.T;
  bool bad_T = false;
  if (a.d_T) {
    const int td = *reinterpret_cast<const volatile int32_t *>(a.d_T);
    bad_T = td < 0 || td > a.Tmax;
    T = td < 0 ? 0 : (td > a.Tmax ? a.Tmax : td);
  }
  const int Rg = route_blocks(a.T);  // row groups of the grid
  const int R = route_blocks(T);     // row groups with rows
  const bool proj = a.w_router != nullptr;
  const int nrb = proj ? Rg * a.n_eblk : Rg;  // routing (projection) blocks of the grid
  // the step's counters (the expert kernel reads them after this grid completes)
  const int64_t gtid = int64_t(blockIdx.x) * blockDim.x + tid, gstride = int64_t(gridDim.x) * blockDim.x;
  const int64_t n_comb = int64_t(T) * a.comb_per_row;
  for (int64_t i = gtid; i < a.n_tiles_max; i += gstride) a.ready[i] = 0;
  for (int64_t i = gtid; i < n_comb; i += gstride) a.comb_cnt[i] = 0;

  if (int(blockIdx.x) >= nrb) {  // x quantisation
    const int64_t groups = int64_t(T) * (a.H / kGroup);
    const int64_t qstride = int64_t(gridDim.x - nrb) * blockDim.x;
    for (int64_t g = int64_t(blockIdx.x - nrb) * blockDim.x + tid; g < groups; g += qstride)
      quantize_group32(a.x + g * kGroup, a.xq + g * kGroup, a.xs + g);
    return;
  }
  if (blockIdx.x == 0) {
    if (tid < 8) a.diag[tid] = 0;
    if (tid == 0) {
      *a.status = MOE_OK;  // start of the step
      a.work[0] = 0;       // unit counter of the tensor-core expert kernel
      a.work[1] = 0;       // abort flag
      if (bad_T) report_error(a.status, MOE_ERR_DEVICE_BOUNDS);
      if (T == 0) {        // an empty step: empty work lists
        *a.n_tiles = 0;
        if (a.chunk_list) *a.n_chunks = 0;
      }
    }
  }
  int rg = int(blockIdx.x);  // this block's row group
  if (proj) {
    rg = int(blockIdx.x) / a.n_eblk;
    if (rg >= R) return;  // no rows for this row group
    // up to 8 rows: CUDA-core sums (latency-bound); more: tensor cores
    if (T - rg * (kRouteThreads / 32) > 8) router_block_mma(a, T, rg, int(blockIdx.x) % a.n_eblk, sm);
    else router_block(a, T, rg, int(blockIdx.x) % a.n_eblk, sm);
    // The last projection block of the row group routes its rows (ticket
    // after a fence; the counter wraps back to zero on the last ticket).
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.last = atomicInc(a.rg_cnt + rg, uint32_t(a.n_eblk - 1)) == uint32_t(a.n_eblk - 1);
    __syncthreads();
    if (!sm.last) return;
    __threadfence();  // the other projection blocks' logits, before they are read
  } else if (rg >= R) {
    return;  // no rows for this routing block
  }
  // One routing block keeps the bitmap in shared memory from the start and
  // needs no ticket.
  const bool single = R == 1;
  if (single) {
    for (int i = tid; i < a.E * a.words; i += blockDim.x) bm[i] = 0;
    __syncthreads();
  }

  // --- phase 1: top-k + combine weights, one warp per row
  uint32_t *bits = single ? bm : nullptr;
  const int nc = (a.E + 31) / 32;
  if (nc <= 1) route_topk<1>(a, T, rg, sm, bits);
  else if (nc <= 2) route_topk<2>(a, T, rg, sm, bits);
  else if (nc <= 4) route_topk<4>(a, T, rg, sm, bits);
  else if (nc <= 8) route_topk<8>(a, T, rg, sm, bits);
  else if (nc <= 16) route_topk<16>(a, T, rg, sm, bits);
  else route_topk<32>(a, T, rg, sm, bits);

  // --- phase 2 in the last routing block to finish phase 1 (ticket after a
  // fence; the ticket counter wraps back to zero on the last ticket)
  if (!single) {
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.last = atomicInc(a.ticket, uint32_t(R - 1)) == uint32_t(R - 1);
    __syncthreads();
    if (!sm.last) return;
    __threadfence();  // the other blocks' results, before they are read
  }
  route_place(a, T, sm, bm, single);
}

size_t route_smem_bytes(int E, int words) { return sizeof(RouteSmem) + size_t(E) * words * sizeof(uint32_t); }

cudaError_t prepare_route() {
  return cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kRouteSmemMax));
}

// R routing blocks (R * ceil(E/8) projection blocks with a router weight),
// then one block per 1024 32-groups of x.
int route_grid(int T, int H, int nproj) {
  const int64_t groups = int64_t(T) * (H / kGroup);
  return route_blocks(T) * nproj + int((groups + kRouteThreads - 1) / kRouteThreads);
}

cudaError_t launch_route(const RouteArgs &a, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(route_grid(a.T, a.H, a.w_router ? a.n_eblk : 1));
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = route_smem_bytes(a.E, a.words);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_kernel, a);
}

cudaError_t launch_quantize_fp4(const uint16_t *x, int64_t rows, int cols, uint8_t *q, uint8_t *s, cudaStream_t st) {
  const int64_t groups = rows * (cols / kGroup);
  if (groups == 0) return cudaSuccess;
  int64_t blocks = (groups + kQuantThreads - 1) / kQuantThreads;
  if (blocks > 65535 * 16) blocks = 65535 * 16;
  quantize_fp4_kernel<<<unsigned(blocks), kQuantThreads, 0, st>>>(x, groups, q, s);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const uint16_t *x, int64_t rows, int cols, uint8_t *q, uint8_t *s, cudaStream_t st) {
  const int64_t groups = rows * (cols / kGroup);
  if (groups == 0) return cudaSuccess;
  int64_t blocks = (groups + kQuantThreads - 1) / kQuantThreads;
  if (blocks > 65535 * 16) blocks = 65535 * 16;
  quantize_kernel<<<unsigned(blocks), kQuantThreads, 0, st>>>(x, groups, q, s);
  return cudaGetLastError();
}

}  // namespace moe
