// experts.cu — persistent expert kernel: gate/up GEMV + SwiGLU + MXFP8(h), then down GEMV.
//
// Work units, claimed in order from one global counter:
//   gate/up unit (tile g, block b): 32 gate rows + 32 up rows, i in [32b, 32b+32),
//       for the <= 8 token rows of tile g. Output: h for those rows, quantised
//       to MXFP8 along I (one 32-group per unit). Then ready[g] is bumped.
//   down unit (tile g, block b): DB rows of W_down, h in [b*DB, (b+1)*DB), for the
//       rows of tile g. It waits (bounded) until ready[g] counts every gate/up
//       unit of g, then writes o[pair][h] in fp32.
// All gate/up units come before all down units in the claim order. So a down
// unit waits only on units that running blocks have already claimed, and those
// never wait. The schedule cannot deadlock, and every wait is bounded anyway.
//
// Pages followed:
// - "FlyDSL Mono Kernels for High-Interactivity LLM Serving in ATOM",
//   "MiniMax-M3: Connecting Attention and Experts":
//     - blocks take on the next task (persistent blocks);
//     - a later stage's weight loads start before its input is ready (the
//       down-projection weights are fetched before the wait on h);
//     - tagged buffers signal ready data (the per-tile ready counters).
// - "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", 2.1: GEMV at
//   small batch, with the reduction fused with MXFP8 quantisation of its
//   output (h is quantised in the epilogue of the gate/up unit).
// - Same page, 3.1: SwiGLU with the original intermediate rounding. g and u are
//   rounded to bf16, and h = bf16(silu(g) * u) is then quantised.
//
// Block layout: 16 compute warps + 1 producer warp + 1 reducer warp. The producer's elected
// lane streams the unit's weight rows with bulk copies (TMA, no tensor map, no
// multicast) into a 5-stage ring of 32 KB + scales.
//
// Each compute thread owns 16 consecutive K columns of 4 rows of every stage:
//  - K/16 threads cover a row, and 512/(K/16) row groups split the stage's rows;
//  - per row it reads 16 weight bytes (one 16-byte shared load) and the
//    group's scale, decodes E4M3 to fp32, and accumulates with packed FFMA2
//    against its 16 columns of the token rows (fp32 registers, 2 tokens per
//    pass).
// A transposing butterfly reduces 4 rows x NP tokens across the lanes. Each
// compute warp then posts its partial sums to shared memory and arrives on the
// stage's reduction barrier. The reducer warp sums the partials across warps in
// a fixed order, writes the outputs, runs the gate/up epilogue and frees the
// stage. Compute warps never wait for each other or for the reducer except
// through the depth of the ring. No block-wide barrier runs in steady state. Every output goes through the same addition tree
// whatever the tile's row count, so results do not depend on tile-mates.
#include <stdint.h>

#include "combine.cuh"
#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr uint32_t kDone = 0xFFFFFFFFu;
constexpr int kConsumers = kConsumerWarps * 32;   // 512
constexpr int kStageScaleBytes = kStageBytes / kGroup;
constexpr int kStageStride = kStageBytes + kStageScaleBytes;
constexpr int kMaxSlots = kConsumers / 16;        // reduction slots (K = 256 uses half-warps)
constexpr int kRedValues = 32;                    // per slot: passes x 4 rows x NP tokens
constexpr int kUnitSlots = 8;                     // gate/up units in flight per block
constexpr int kCombineQueue = 256;                // combine jobs a block can defer to its end

// A work unit as the producer publishes it (decoded once, read by every consumer warp).
struct UnitMeta {
  int32_t valid;     // 0: past the end of this block's schedule
  int32_t down;      // 0: gate/up, 1: down
  int32_t tile;      // index into tile_list
  int32_t block;     // b
  int32_t expert;    // e (E = shared)
  int32_t n;         // rows in this tile (1..8)
  int32_t cnt;       // rows of the expert (all tiles)
  int32_t pairs[kTileRows];
};

struct __align__(16) ExpertSmem {
  unsigned char stage[kStages][kStageStride];
  float red[kStages][kMaxSlots][kRedValues];      // per-warp partial sums of a stage
  float gu[kTileRows][2][32];                     // gate/up results of the reducer's unit, [token][gate|up][i]
  UnitMeta meta[kUnitSlots];                      // unit i of this block lives in slot i % kUnitSlots
  uint64_t full[kStages];                         // weights landed (producer arrive + tx bytes)
  uint64_t empty[kStages];                        // stage free again (the reducer warp)
  uint64_t red_full[kStages];                     // partial sums posted (16 compute warps)
  uint32_t meta_unit[kStages];                    // unit sequence number of the stage, or kDone
  uint32_t meta_step[kStages];                    // stage index within the unit
  uint4 pf_q[2][kConsumers];                      // per-thread prefetch of the next unit's columns
  uint32_t cq[kCombineQueue];                     // deferred combine jobs (token row << 16 | down block)
  uint32_t cq_head;                               // jobs queued by the reducer
  uint32_t cq_tail;                               // jobs taken by compute warps at the end
  uint32_t cq_done;                               // the reducer has finished
};
static_assert(sizeof(ExpertSmem) <= 227 * 1024, "shared memory budget");

template <int KG, int KD>
struct Shape {
  static constexpr int H = KG, I = KD;
  static constexpr int RS_G = kStageBytes / KG;    // rows per stage (gate/up)
  static constexpr int RS_D = kStageBytes / KD;    // rows per stage (down)
  static constexpr int SPU_G = 64 / RS_G;          // stages per gate/up unit (64 rows)
  static constexpr int SPU_D = (H / RS_D) < 8 ? (H / RS_D) : 8;
  static constexpr int DB = SPU_D * RS_D;          // rows of W_down per down unit
  static constexpr int NBG = I / 32;               // gate/up units per tile
  static constexpr int NBD = H / DB;               // down units per tile
  static_assert(KG >= 512 && KG <= 4096 && (KG & (KG - 1)) == 0, "H: power of two in [512, 4096]");
  static_assert(KD >= 256 && KD <= 4096 && (KD & (KD - 1)) == 0, "I: power of two in [256, 4096]");
  static_assert(SPU_G >= 1 && 64 % RS_G == 0, "gate/up unit spans whole stages");
  static_assert(H % DB == 0, "down units tile H");
};

// Row geometry of a stage for a K-wide weight matrix and 512 compute threads.
template <int K>
struct Rows {
  static constexpr int TPR = K / 16;                 // threads per row
  static constexpr int RG = kConsumers / TPR;        // row groups
  static constexpr int RS = kStageBytes / K;         // rows per stage
  static constexpr int PER_THREAD = RS / RG;         // rows per thread per stage (4)
  static constexpr int LANES = TPR < 32 ? TPR : 32;  // lanes of a row group inside one warp
  static constexpr int SPG = TPR / LANES;            // reduction slots per row group
  static_assert(PER_THREAD == 4, "4 rows per thread per stage");
};

// ------------------------------------------------------------------ per-thread math

struct XRegs {
  uint32_t h[2][8];         // the pass's tokens: 16 E4M3 values as 8 f16x2 (exact, unscaled)
  float sc[2];              // their group scales 2^(code - 127)
};

// 16 E4M3 codes -> 8 f16x2 (exact: every E4M3 value is an f16 normal or zero).
__device__ __forceinline__ void decode16_h2(const uint4 v, uint32_t (&o)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = e4m3x2_to_f16x2(uint16_t(w[i] & 0xFFFFu));
    o[2 * i + 1] = e4m3x2_to_f16x2(uint16_t(w[i] >> 16));
  }
}

// Tokens [NP*pass, NP*pass + NP) of the tile into registers (f16x2 codes + scale).
// row_q(tok) / row_s(tok) give the thread's 16 E4M3 codes and the group's scale
// code of a tile row. They are read through L2: an earlier grid or block wrote them.
template <int NP, class FQ, class FS>
__device__ __forceinline__ void load_pass(XRegs &x, int pass, int n, FQ &&row_q, FS &&row_s) {
#pragma unroll
  for (int t = 0; t < NP; ++t) {
    const int tok = NP * pass + t;
    if (tok < n) {
      decode16_h2(__ldcg(reinterpret_cast<const uint4 *>(row_q(tok))), x.h[t]);
      x.sc[t] = ue8m0_to_float(__ldcg(row_s(tok)));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x.h[t][i] = 0u;
      x.sc[t] = 0.f;
    }
  }
}

// This thread's partial dot products for its 4 rows of the stage and NP tokens.
// Products of two E4M3 values are exact in fp32; fma.rn.f32.f16 accumulates
// them in fp32 directly from the f16 operands (no separate widening).
template <int K, int NP>
__device__ __forceinline__ void stage_dot(const unsigned char *st, int g, int c, const XRegs &x,
                                          float (&acc)[4 * NP]) {
  using R = Rows<K>;
  const unsigned char *sw = st;
  const unsigned char *ss = st + kStageBytes;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = g + R::RG * j;
    const uint4 wv = *reinterpret_cast<const uint4 *>(sw + r * K + 16 * c);
    const float ws = ue8m0_to_float(ss[r * (K / kGroup) + (c >> 1)]);
    uint32_t w[8];
    decode16_h2(wv, w);
#pragma unroll
    for (int t = 0; t < NP; ++t) {
      float c0 = 0.f, c1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        c0 = fma_f16x2_f32(w[i], x.h[t][i], c0);
        c1 = fma_f16x2_f32(w[i + 1], x.h[t][i + 1], c1);
      }
      acc[j * NP + t] = (c0 + c1) * (ws * x.sc[t]);
    }
  }
}

// Transposing butterfly over LANES lanes. On return, lane l holds CNT values;
// value i has original index i + sum over halving steps s of
// (l & (LANES >> (s+1))) ? (V >> (s+1)) : 0. Each is the full LANES-lane sum.
// The additions follow the same tree (offsets LANES/2 ... 1) for every V.
template <int V, int LANES>
struct Butterfly {
  static constexpr int LOGV = V == 4 ? 2 : V == 8 ? 3 : V == 16 ? 4 : 5;
  static constexpr int LOGL = LANES == 32 ? 5 : 4;
  static constexpr int HSTEPS = LOGV < LOGL ? LOGV : LOGL;
  static constexpr int CNT = V >> HSTEPS;
  static constexpr int TAILMASK = (LANES >> HSTEPS) - 1;

  __device__ __forceinline__ static void run(float (&a)[V], int l) {
#pragma unroll
    for (int s = 0; s < HSTEPS; ++s) {
      const int off = LANES >> (s + 1);
      const int half = (V >> s) / 2;
      const bool upper = (l & off) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = upper ? a[i] : a[i + half];
        const float keep = upper ? a[i + half] : a[i];
        a[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
      }
    }
#pragma unroll
    for (int off = (LANES >> HSTEPS) / 2; off >= 1; off >>= 1)
#pragma unroll
      for (int i = 0; i < CNT; ++i) a[i] += __shfl_xor_sync(0xFFFFFFFFu, a[i], off);
  }

  __device__ __forceinline__ static int index(int l, int i) {
    int idx = i;
#pragma unroll
    for (int s = 0; s < HSTEPS; ++s)
      if (l & (LANES >> (s + 1))) idx += V >> (s + 1);
    return idx;
  }
};


// ------------------------------------------------------------------ unit schedule
// Static round-robin: block b runs units b, b + G, b + 2G, ... (G = grid size) in
// increasing order. Every gate/up unit precedes every down unit in that order,
// so a down unit only ever waits on lower-numbered units. Each block runs its
// units in increasing order, so the waits cannot form a cycle.

template <class S>
__device__ __forceinline__ void unit_coords(uint32_t u, int n_tiles, int &down, int &tile, int &block) {
  const uint32_t ngu = uint32_t(n_tiles) * S::NBG;
  if (u < ngu) {
    down = 0;
    tile = int(u / S::NBG);
    block = int(u % S::NBG);
  } else {
    const uint32_t v = u - ngu;
    down = 1;
    tile = int(v / S::NBD);
    block = int(v % S::NBD);
  }
}

// ------------------------------------------------------------------ producer (one warp)
// A three-step fetch pipeline keeps the decode loads off the critical path.
// Iteration i:
//   1. lane 0 loads the tile_list entry of unit i+3;
//   2. using unit i+2's tile_list entry (loaded one iteration earlier), load
//      its expert row count (lane 0) and its <= 8 pair ids (lanes 0..7);
//   3. issue the weight stages of unit i;
//   4. publish unit i+2's metadata. The loads of step 2 have landed during step 3.
// Units i and i+1 were published before unit i's first stage, so consumers can
// prefetch unit i+1's token rows while they work on unit i.

template <class S>
__device__ void producer(const ExpertArgs &a, ExpertSmem &sm, int n_tiles) {
  const int lane = threadIdx.x & 31;
  const uint64_t pol = l2_evict_first_policy();
  const uint64_t pol_reuse = l2_evict_normal_policy();
  const uint32_t total = uint32_t(n_tiles) * (S::NBG + S::NBD);
  const uint32_t G = gridDim.x;
  // The producer's waits outlast the consumers' bounded ready wait, so a
  // consumer that gives up on a tile always drains the ring first.
  const int64_t wait_ns = 4 * a.timeout_ns;
  auto unit_of = [&](uint32_t i) -> uint32_t { return blockIdx.x + i * G; };
  auto load_te = [&](uint32_t i) -> int32_t {
    const uint32_t u = unit_of(i);
    if (u >= total) return -1;
    int down, tile, block;
    unit_coords<S>(u, n_tiles, down, tile, block);
    if (!in_bounds(a.status, a.diag, 30, tile, a.n_tiles_max)) return -1;
    return __ldcg(a.tile_list + tile);
  };
  struct Fetch {
    int32_t te, cnt, pair;
  };
  // step 2: counts and pair ids (one pair per lane 0..7) of the unit whose tile entry is te
  auto load_rows = [&](int32_t te) -> Fetch {
    Fetch f{te, 0, 0};
    if (te < 0) return f;
    const int expert = te >> 16, tile_in = te & 0xFFFF;
    if (!in_bounds(a.status, a.diag, 31, expert, a.E + 1)) {
      f.te = -1;
      return f;
    }
    f.cnt = __ldcg(a.counts + expert);
    const int row = min(kTileRows * tile_in + (lane & 7), a.Tmax - 1);
    f.pair = __ldcg(a.rows_of + int64_t(expert) * a.Tmax + row);
    if constexpr (kBoundsChecked) {  // a pair id outside [0, P) becomes 0 (reported for the tile's own rows)
      if (f.pair < 0 || f.pair >= a.pairs_cap) {
        if ((lane & 7) < f.cnt - kTileRows * tile_in) in_bounds(a.status, a.diag, 32, f.pair, a.pairs_cap);
        f.pair = 0;
      }
    }
    return f;
  };
  auto publish = [&](uint32_t i, const Fetch &f) {
    UnitMeta &m = sm.meta[i & (kUnitSlots - 1)];
    const uint32_t u = unit_of(i);
    if (lane < kTileRows) m.pairs[lane] = f.pair;
    if (lane == 0) {
      m.valid = u < total && f.te >= 0;
      int down = 0, tile = 0, block = 0;
      if (m.valid) unit_coords<S>(u, n_tiles, down, tile, block);
      m.down = down;
      m.tile = tile;
      m.block = block;
      m.expert = f.te >> 16;
      const int n = f.cnt - kTileRows * (f.te & 0xFFFF);
      m.n = n < kTileRows ? n : kTileRows;
      m.cnt = f.cnt;
    }
    __syncwarp();
  };

  // prologue: units 0 and 1 published, unit 2's rows in flight, unit 3's tile entry in flight
  publish(0, load_rows(__shfl_sync(0xFFFFFFFFu, load_te(0), 0)));
  publish(1, load_rows(__shfl_sync(0xFFFFFFFFu, load_te(1), 0)));
  int32_t te_next = __shfl_sync(0xFFFFFFFFu, load_te(2), 0);  // unit i+2's entry at iteration i

  int stage = 0;
  uint32_t phase = 0;  // flips each time the ring wraps; empty-barrier parity is phase ^ 1
  for (uint32_t i = 0;; ++i) {
    const UnitMeta &m = sm.meta[i & (kUnitSlots - 1)];
    // end of schedule, or abort: lane 0 decides for the warp
    const int stop = __shfl_sync(0xFFFFFFFFu, (!m.valid || ld_volatile(a.work + 1) != 0) ? 1 : 0, 0);
    if (stop) {
      int64_t waited = 0;
      const int ok = __shfl_sync(0xFFFFFFFFu, mbar_wait(&sm.empty[stage], phase ^ 1u, wait_ns, &waited) ? 1 : 0, 0);
      if (!ok) {
        if (lane == 0) report_diag(a.status, a.diag, MOE_ERR_TIMEOUT, kDiagEmptyWait, i, stage, phase, -1, waited, 0);
        return;
      }
      if (lane == 0) {
        sm.meta_unit[stage] = kDone;
        sm.meta_step[stage] = 0;
        mbar_arrive(&sm.full[stage]);
      }
      return;
    }
    // steps 1 and 2 (loads in flight while the stages are issued)
    const int32_t te_far = load_te(i + 3);
    const Fetch f2 = load_rows(te_next);
    const bool sh = m.expert == a.E;
    const int e = sh ? 0 : m.expert;
    const int down = m.down, block = m.block;
    // Weights of a single-tile expert are read once per step: evict first.
    // A multi-tile expert's weights are read once per tile: keep them in L2.
    const uint64_t pol_u = m.cnt > kTileRows ? pol_reuse : pol;
    const int steps = down ? S::SPU_D : S::SPU_G;
    for (int s = 0; s < steps; ++s) {
      int64_t waited = 0;
      const int ok = __shfl_sync(0xFFFFFFFFu, mbar_wait(&sm.empty[stage], phase ^ 1u, wait_ns, &waited) ? 1 : 0, 0);
      if (!ok) {
        if (lane == 0) {
          report_diag(a.status, a.diag, MOE_ERR_TIMEOUT, kDiagEmptyWait, i, stage, phase, s, waited, 0);
          atomicExch(a.work + 1, 1u);
        }
        return;
      }
      if (lane == 0) {
        sm.meta_unit[stage] = i;
        sm.meta_step[stage] = uint32_t(s);
        unsigned char *dst = sm.stage[stage];
        mbar_arrive_expect_tx(&sm.full[stage], uint32_t(kStageStride));
        if (!down) {
          // gate rows i0 .. i0 + RS/2, then up rows i0 .. i0 + RS/2
          constexpr int HALF = S::RS_G / 2;
          const int64_t i0 = int64_t(block) * 32 + int64_t(s) * HALF;
          const uint8_t *wg = sh ? a.sh_w_gate : a.w_gate + int64_t(e) * S::I * S::H;
          const uint8_t *wu = sh ? a.sh_w_up : a.w_up + int64_t(e) * S::I * S::H;
          const uint8_t *sg = sh ? a.sh_s_gate : a.s_gate + int64_t(e) * S::I * (S::H / kGroup);
          const uint8_t *su = sh ? a.sh_s_up : a.s_up + int64_t(e) * S::I * (S::H / kGroup);
          bulk_g2s(dst, wg + i0 * S::H, HALF * S::H, &sm.full[stage], pol_u);
          bulk_g2s(dst + kStageBytes / 2, wu + i0 * S::H, HALF * S::H, &sm.full[stage], pol_u);
          bulk_g2s(dst + kStageBytes, sg + i0 * (S::H / kGroup), HALF * (S::H / kGroup), &sm.full[stage], pol_u);
          bulk_g2s(dst + kStageBytes + kStageScaleBytes / 2, su + i0 * (S::H / kGroup), HALF * (S::H / kGroup),
                   &sm.full[stage], pol_u);
        } else {
          const int64_t r0 = int64_t(block) * S::DB + int64_t(s) * S::RS_D;
          const uint8_t *wd = sh ? a.sh_w_down : a.w_down + int64_t(e) * S::H * S::I;
          const uint8_t *sd = sh ? a.sh_s_down : a.s_down + int64_t(e) * S::H * (S::I / kGroup);
          bulk_g2s(dst, wd + r0 * S::I, kStageBytes, &sm.full[stage], pol_u);
          bulk_g2s(dst + kStageBytes, sd + r0 * (S::I / kGroup), kStageScaleBytes, &sm.full[stage], pol_u);
        }
      }
      __syncwarp();
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // step 4: publish unit i+2 (its slot last held unit i-6, long finished)
    publish(i + 2, f2);
    te_next = __shfl_sync(0xFFFFFFFFu, te_far, 0);
  }
}

// ------------------------------------------------------------------ consumers

// One pass (NP tokens) over this thread's 4 rows of the stage: dot products,
// warp reduction, and the per-slot partial sums into red[stage].
template <int K, int NP>
__device__ __forceinline__ void stage_pass(ExpertSmem &sm, const unsigned char *st, int stage, int pass,
                                           const XRegs &x) {
  using R = Rows<K>;
  constexpr int V = 4 * NP;
  using BF = Butterfly<V, R::LANES>;
  const int tid = threadIdx.x;
  const int g = tid / R::TPR, c = tid % R::TPR;
  const int l = tid & (R::LANES - 1);
  const int slot = tid / R::LANES;
  float acc[V];
  stage_dot<K, NP>(st, g, c, x, acc);
  BF::run(acc, l);
  if ((l & BF::TAILMASK) == 0) {
#pragma unroll
    for (int i = 0; i < BF::CNT; ++i) sm.red[stage][slot][pass * V + BF::index(l, i)] = acc[i];
  }
}

// The stage's last warp to post: sums one stage's partials across the warps of each
// row group, in slot order. Calls out(row_in_stage, token, value).
template <int K, class F>
__device__ __forceinline__ void reduce_stage(const ExpertSmem &sm, int stage, int passes, int np, int n, int lane,
                                             F &&out) {
  using R = Rows<K>;
  const int V = 4 * np;
  const int per_pass = R::RG * V;
  for (int o = lane; o < passes * per_pass; o += 32) {
    const int pass = o / per_pass;
    const int q = o % per_pass;
    const int g = q / V;
    const int v = q % V;
    const int j = v / np, t = v % np;
    const int tok = np * pass + t;
    if (tok >= n) continue;
    const int idx = pass * V + v;
    float s = sm.red[stage][g * R::SPG][idx];
#pragma unroll
    for (int k = 1; k < R::SPG; ++k) s += sm.red[stage][g * R::SPG + k][idx];
    out(g + R::RG * j, tok, s);
  }
}

// gate/up epilogue, one warp: h = bf16(silu(bf16 g) * bf16 u), MXFP8 along I; then publish.
template <class S>
__device__ __forceinline__ void gate_up_epilogue(const ExpertArgs &a, ExpertSmem &sm, const UnitMeta &m, int lane) {
  for (int t = 0; t < m.n; ++t) {
    float gb = bf16_bits_to_float(float_to_bf16_bits(sm.gu[t][0][lane]));
    float ub = bf16_bits_to_float(float_to_bf16_bits(sm.gu[t][1][lane]));
    if (a.swiglu_limit > 0.0f) {  // clipped SwiGLU
      gb = fminf(gb, a.swiglu_limit);
      ub = fminf(fmaxf(ub, -a.swiglu_limit), a.swiglu_limit);
    }
    const float silu = gb / (1.0f + expf(-gb));
    const uint16_t hb = float_to_bf16_bits(silu * ub);
    const float hv = bf16_bits_to_float(hb);
    float amax = fabsf(hv);
#pragma unroll
    for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const uint32_t code = mx_scale_code(amax);
    const int64_t p = m.pairs[t];
    a.hq[p * S::I + int64_t(m.block) * 32 + lane] = float_to_e4m3(mx_unscale(hv, code));
    if (lane == 0) a.hs[p * (S::I / kGroup) + m.block] = uint8_t(code);
    if (a.h_bf16) a.h_bf16[p * S::I + int64_t(m.block) * 32 + lane] = hb;
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) {
    if (m.tile != a.skip_ready_tile) red_release_gpu_add(a.ready + m.tile, 1u);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ activation prefetch
// Each compute thread owns 16 columns of a tile row. For units with <= 2 rows
// it copies its columns of the next unit's rows (and the group scales) into its
// own shared-memory slot with cp.async while it works on the current unit.
// Only that thread reads the slot, so the copy needs no block synchronisation
// (cp.async.wait_group covers it). A down unit's h is prefetched only after its
// tile's ready count has been observed complete.

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// This thread's 16 columns (codes) and scale byte address of tile row `tok` of unit m.
template <class S>
__device__ __forceinline__ const uint8_t *row_codes(const ExpertArgs &a, const UnitMeta &m, int tok, int tid) {
  const int64_t p = m.pairs[tok];
  if (m.down) return a.hq + p * S::I + 16 * (tid % (S::I / 16));
  const int64_t t = m.expert == a.E ? p - int64_t(a.T) * a.k : p / a.k;
  return a.xq + t * S::H + 16 * (tid % (S::H / 16));
}
template <class S>
__device__ __forceinline__ const uint8_t *row_scale(const ExpertArgs &a, const UnitMeta &m, int tok, int tid) {
  const int64_t p = m.pairs[tok];
  if (m.down) return a.hs + p * (S::I / kGroup) + ((tid % (S::I / 16)) >> 1);
  const int64_t t = m.expert == a.E ? p - int64_t(a.T) * a.k : p / a.k;
  return a.xs + t * (S::H / kGroup) + ((tid % (S::H / 16)) >> 1);
}

// The 16 code bytes go to shared memory by cp.async (L2 path). The scale byte
// goes to a register with an L2 load; neither is waited for until the unit starts.
template <class S>
__device__ __forceinline__ void prefetch_rows(const ExpertArgs &a, ExpertSmem &sm, const UnitMeta &m, int tid,
                                              uint32_t (&pf_sc)[2]) {
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    if (t < m.n) {
      cp_async16(&sm.pf_q[t][tid], row_codes<S>(a, m, t, tid));
      pf_sc[t] = __ldcg(row_scale<S>(a, m, t, tid));
    }
  }
  cp_async_commit();
}

// Tokens 0..n-1 (n <= 2) of the unit from this thread's prefetch slot.
__device__ __forceinline__ void load_prefetched(XRegs &x, const ExpertSmem &sm, const UnitMeta &m, int tid,
                                                const uint32_t (&pf_sc)[2]) {
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    if (t < m.n) {
      decode16_h2(sm.pf_q[t][tid], x.h[t]);
      x.sc[t] = ue8m0_to_float(pf_sc[t]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x.h[t][i] = 0u;
      x.sc[t] = 0.f;
    }
  }
}

// Bounded wait until every gate/up unit of `tile` has published (lane 0 polls,
// the warp agrees). Returns false after a timeout.
template <class S>
__device__ __forceinline__ bool wait_tile_ready(const ExpertArgs &a, int tile, uint32_t i, int lane) {
  int ok = 1;
  if (lane == 0) {
    const WaitClock wc;
    uint32_t seen;
    while ((seen = ld_acquire_gpu(a.ready + tile)) < uint32_t(S::NBG)) {
      if (wc.expired(a.timeout_ns)) {
        report_diag(a.status, a.diag, MOE_ERR_TIMEOUT, kDiagReadyWait, i, tile, seen, S::NBG, wc.ns(), wc.cycles());
        atomicExch(a.work + 1, 1u);
        ok = 0;
        break;
      }
      __nanosleep(64);
    }
  }
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;  // the shuffle also orders lane 0's acquire before the warp's loads
}

template <class S>
__device__ __forceinline__ void run_deferred_combines(const ExpertArgs &a, ExpertSmem &sm, int lane);

template <class S>
__device__ void consumers(const ExpertArgs &a, ExpertSmem &sm, int n_tiles) {
  (void)n_tiles;
  const int tid = threadIdx.x, lane = tid & 31;
  int stage = 0;
  uint32_t phase = 0;   // barrier parity of the current ring pass
  uint32_t unit = 0;    // this block's unit sequence number of the current unit
  int uslot = 0;
  XRegs x;
  int np = 1, passes = 1;
  bool skip = false;
  bool pf_ready_now = false;   // the prefetch slot holds the current unit's rows
  bool pf_pending = false;     // the next unit's rows are being prefetched into the slot
  bool pf_down_next = false;   // the next unit is a down unit whose rows may be prefetched late
  uint32_t ready_seen = 0;     // lane 0: the next down unit's ready count, loaded early
  uint32_t pf_sc[2] = {0, 0};  // scale codes of the prefetched rows
  while (true) {
    int64_t waited = 0;
    if (!mbar_wait(&sm.full[stage], phase, 16 * a.timeout_ns, &waited)) {
      if (lane == 0) {
        report_diag(a.status, a.diag, MOE_ERR_TIMEOUT, kDiagFullWait, -1, stage, phase, -1, waited, 0);
        atomicExch(a.work + 1, 1u);
      }
      return;
    }
    const uint32_t u = sm.meta_unit[stage];
    const int s = int(sm.meta_step[stage]);
    if (u == kDone) {
      cp_async_wait_all();
      run_deferred_combines<S>(a, sm, lane);
      return;
    }
    const unsigned char *st = sm.stage[stage];
    if (s == 0) {
      // ---- unit start. The producer published this unit and the next one.
      unit = u;
      uslot = int(unit & (kUnitSlots - 1));
      const UnitMeta &m = sm.meta[uslot];
      cp_async_wait_all();
      pf_ready_now = pf_pending;
      pf_pending = false;
      skip = false;
      np = m.n <= 1 ? 1 : 2;
      passes = (m.n + np - 1) / np;
      if (pf_ready_now) {
        load_prefetched(x, sm, m, tid, pf_sc);
      } else {
        if (m.down) skip = !wait_tile_ready<S>(a, m.tile, unit, lane);
        if (passes == 1 && !skip) {
          auto rq = [&](int tok) { return row_codes<S>(a, m, tok, tid); };
          auto rs = [&](int tok) { return row_scale<S>(a, m, tok, tid); };
          if (np == 1) load_pass<1>(x, 0, m.n, rq, rs);
          else load_pass<2>(x, 0, m.n, rq, rs);
        }
      }
      // prefetch the next unit's rows (gate/up now; down once its tile is seen ready)
      const UnitMeta &mn = sm.meta[(unit + 1) & (kUnitSlots - 1)];
      pf_down_next = false;
      if (mn.valid && mn.n <= 2) {
        if (!mn.down) {
          prefetch_rows<S>(a, sm, mn, tid, pf_sc);
          pf_pending = true;
        } else {
          // a relaxed look now (no ordering stall); upgraded by a fence when used
          pf_down_next = true;
          if (lane == 0) ready_seen = ld_relaxed_gpu(a.ready + mn.tile);
        }
      }
    }
    const UnitMeta &m = sm.meta[uslot];
    // ---- this stage: dot products and warp reductions, posted to red[stage]
    if (!skip) {
      for (int p = 0; p < passes; ++p) {
        if (np == 1) {
          if (m.down) stage_pass<S::I, 1>(sm, st, stage, p, x);
          else stage_pass<S::H, 1>(sm, st, stage, p, x);
        } else {
          if (passes > 1) {
            auto rq = [&](int tok) { return row_codes<S>(a, m, tok, tid); };
            auto rs = [&](int tok) { return row_scale<S>(a, m, tok, tid); };
            load_pass<2>(x, p, m.n, rq, rs);
          }
          if (m.down) stage_pass<S::I, 2>(sm, st, stage, p, x);
          else stage_pass<S::H, 2>(sm, st, stage, p, x);
        }
      }
    }
    const int spu = m.down ? S::SPU_D : S::SPU_G;
    if (s == spu - 1 && pf_down_next) {
      // the next unit is a down unit: prefetch its h if its tile was already complete
      const int ok = __shfl_sync(0xFFFFFFFFu, ready_seen >= uint32_t(S::NBG) ? 1 : 0, 0);
      if (ok) {
        // relaxed load that saw the count complete + fence = acquire; the
        // warp's copies below are ordered after it by the shuffle
        if (lane == 0) __threadfence();
        __syncwarp();
        prefetch_rows<S>(a, sm, sm.meta[(unit + 1) & (kUnitSlots - 1)], tid, pf_sc);
        pf_pending = true;
      }
      pf_down_next = false;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.red_full[stage]);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

// ------------------------------------------------------------------ fused combine
// y[t][h] for h in down block b, one warp: the warp whose down unit was the
// last of token row t's k (+ shared) pairs to finish block b (combine.cuh).
template <class S>
__device__ __forceinline__ void fused_combine(const ExpertArgs &a, int t, int b, int lane) {
  uint16_t yb[S::DB / 32];
  combine_row_block<S::DB / 32>(a.o, a.topk_w, a.y, a.T, a.k, a.shared, S::H, t, int64_t(b) * S::DB, lane, yb);
}

// After a down unit's last stage: count each of its pairs in for (token row,
// block). For each row this unit completes, a combine job is queued. The 16
// compute warps run the queue in parallel once their stream of stages ends, so
// the combine stays off the reducer's path. If the queue is full, the reducer
// combines the row itself.
template <class S>
__device__ __forceinline__ void down_unit_done(const ExpertArgs &a, ExpertSmem &sm, const UnitMeta &m, int lane) {
  __threadfence();  // this unit's o stores, before the counts
  __syncwarp();
  const uint32_t target = uint32_t(a.k + a.shared);
  for (int r = 0; r < m.n; ++r) {
    const int64_t p = m.pairs[r];
    const int t = p < int64_t(a.T) * a.k ? int(p / a.k) : int(p - int64_t(a.T) * a.k);
    if (!in_bounds(a.status, a.diag, 33, t, a.T) ||
        !in_bounds(a.status, a.diag, 34, int64_t(t) * S::NBD + m.block, a.comb_cap))
      continue;
    uint32_t before = 0;
    if (lane == 0) before = atomicAdd(a.comb_cnt + int64_t(t) * S::NBD + m.block, 1u);
    before = __shfl_sync(0xFFFFFFFFu, before, 0);
    if (before != target - 1) continue;
    __threadfence();  // the other pairs' o stores, before anyone reads them
    const uint32_t head = sm.cq_head;  // only this warp writes it
    if (head < uint32_t(kCombineQueue)) {
      if (lane == 0) {
        sm.cq[head] = (uint32_t(t) << 16) | uint32_t(m.block);
        sm.cq_head = head + 1;
      }
      __syncwarp();
    } else {
      fused_combine<S>(a, t, m.block, lane);
    }
  }
  __syncwarp();
}

// Compute warps, after their last stage: wait (bounded) for the reducer to
// finish, then take the queued combine jobs one by one.
template <class S>
__device__ __forceinline__ void run_deferred_combines(const ExpertArgs &a, ExpertSmem &sm, int lane) {
  int done = 0;
  if (lane == 0) {
    const WaitClock wc;
    while (!(done = *reinterpret_cast<volatile uint32_t *>(&sm.cq_done) != 0)) {
      if (wc.expired(16 * a.timeout_ns)) {
        report_error(a.status, MOE_ERR_TIMEOUT);
        break;
      }
      __nanosleep(128);
    }
  }
  if (!__shfl_sync(0xFFFFFFFFu, done, 0)) return;
  __threadfence_block();
  const uint32_t head = *reinterpret_cast<volatile uint32_t *>(&sm.cq_head);
  while (true) {
    uint32_t j = 0;
    if (lane == 0) j = atomicAdd(&sm.cq_tail, 1u);
    j = __shfl_sync(0xFFFFFFFFu, j, 0);
    if (j >= head) return;
    const uint32_t job = sm.cq[j];
    fused_combine<S>(a, int(job >> 16), int(job & 0xFFFFu), lane);
  }
}

// ------------------------------------------------------------------ reducer (one warp)
// For every stage: waits until the 16 compute warps have posted their partial
// sums, sums them across warps in a fixed order, writes the outputs and frees
// the stage. At the end of a gate/up unit it runs the SwiGLU + MXFP8 epilogue
// and publishes the tile's ready count. The compute warps never wait for it
// except through the depth of the ring.
template <class S>
__device__ void reducer(const ExpertArgs &a, ExpertSmem &sm) {
  const int lane = threadIdx.x & 31;
  int stage = 0;
  uint32_t phase = 0;
  while (true) {
    int64_t waited = 0;
    if (!__shfl_sync(0xFFFFFFFFu, mbar_wait(&sm.full[stage], phase, 16 * a.timeout_ns, &waited) ? 1 : 0, 0)) {
      if (lane == 0) {
        report_diag(a.status, a.diag, MOE_ERR_TIMEOUT, kDiagFullWait, -1, stage, phase, -3, waited, 0);
        atomicExch(a.work + 1, 1u);
        *reinterpret_cast<volatile uint32_t *>(&sm.cq_done) = 1u;
      }
      return;
    }
    const uint32_t u = sm.meta_unit[stage];
    const int s = int(sm.meta_step[stage]);
    if (u == kDone) {
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        *reinterpret_cast<volatile uint32_t *>(&sm.cq_done) = 1u;
      }
      return;
    }
    if (!__shfl_sync(0xFFFFFFFFu, mbar_wait(&sm.red_full[stage], phase, 16 * a.timeout_ns, &waited) ? 1 : 0, 0)) {
      if (lane == 0) {
        report_diag(a.status, a.diag, MOE_ERR_TIMEOUT, kDiagFullWait, u, stage, phase, -2, waited, 0);
        atomicExch(a.work + 1, 1u);
        *reinterpret_cast<volatile uint32_t *>(&sm.cq_done) = 1u;
      }
      return;
    }
    const int uslot = int(u & (kUnitSlots - 1));
    const UnitMeta &m = sm.meta[uslot];
    const int np = m.n <= 1 ? 1 : 2;
    const int passes = (m.n + np - 1) / np;
    if (m.down) {
      const int64_t hrow0 = int64_t(m.block) * S::DB + int64_t(s) * S::RS_D;
      reduce_stage<S::I>(sm, stage, passes, np, m.n, lane, [&](int r, int tok, float v) {
        a.o[int64_t(m.pairs[tok]) * S::H + hrow0 + r] = v;
      });
      __syncwarp();
      if (s == S::SPU_D - 1) down_unit_done<S>(a, sm, m, lane);
    } else {
      constexpr int HALF = S::RS_G / 2;
      reduce_stage<S::H>(sm, stage, passes, np, m.n, lane, [&](int r, int tok, float v) {
        const int which = r < HALF ? 0 : 1;
        const int i = s * HALF + (r < HALF ? r : r - HALF);
        sm.gu[tok][which][i] = v;
      });
      __syncwarp();
      if (s == S::SPU_G - 1) gate_up_epilogue<S>(a, sm, m, lane);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

template <int KG, int KD>
__global__ void __launch_bounds__(kExpertThreads, 1) experts_kernel(const ExpertArgs a) {
  using S = Shape<KG, KD>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ExpertSmem &sm = *reinterpret_cast<ExpertSmem *>(smem_raw);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
      mbar_init(&sm.red_full[i], kConsumerWarps);
    }
    sm.cq_head = sm.cq_tail = sm.cq_done = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Everything below reads the router's outputs.
  pdl_wait_primary();
  const int n_tiles = __ldcg(a.n_tiles);
  if (warp == kConsumerWarps) {
    producer<S>(a, sm, n_tiles);  // the whole warp: lanes 0..7 fetch pair ids, lane 0 issues copies
    return;
  }
  if (warp == kConsumerWarps + 1) {
    reducer<S>(a, sm);
    return;
  }

  consumers<S>(a, sm, n_tiles);
}

template <int KG, int KD>
cudaError_t prepare_shape() {
  return cudaFuncSetAttribute(experts_kernel<KG, KD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(sizeof(ExpertSmem)));
}

template <int KG, int KD>
cudaError_t launch_shape(const ExpertArgs &a, int grid, cudaStream_t st) {
  const size_t smem = sizeof(ExpertSmem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kExpertThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, experts_kernel<KG, KD>, a);
}

}  // namespace


int experts_down_blocks(int H, int I) {
  if (H == 4096 && I == 2048) return Shape<4096, 2048>::NBD;
  if (H == 1024 && I == 512) return Shape<1024, 512>::NBD;
  if (H == 512 && I == 256) return Shape<512, 256>::NBD;
  return 0;
}

// Shapes compiled into the library: (H, I) = (4096, 2048), (1024, 512), (512, 256).
bool experts_shape_supported(int H, int I) {
  return (H == 4096 && I == 2048) || (H == 1024 && I == 512) || (H == 512 && I == 256);
}

cudaError_t prepare_experts(int H, int I) {
  if (H == 4096 && I == 2048) return prepare_shape<4096, 2048>();
  if (H == 1024 && I == 512) return prepare_shape<1024, 512>();
  if (H == 512 && I == 256) return prepare_shape<512, 256>();
  return cudaErrorInvalidValue;
}

cudaError_t launch_experts(const ExpertArgs &a, int grid, cudaStream_t st) {
  if (a.H == 4096 && a.I == 2048) return launch_shape<4096, 2048>(a, grid, st);
  if (a.H == 1024 && a.I == 512) return launch_shape<1024, 512>(a, grid, st);
  if (a.H == 512 && a.I == 256) return launch_shape<512, 256>(a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace moe
