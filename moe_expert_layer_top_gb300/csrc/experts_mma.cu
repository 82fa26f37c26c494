// experts_mma.cu — tensor-core expert kernel: block-scaled MXFP8 MMA (tcgen05)
// for steps whose experts hold many token rows.
//
// The CUDA-core expert kernel streams an expert's weights once per 8-row tile,
// so an expert with hundreds of rows re-reads them and spends CUDA-core FMAs
// on every tile. Here each expert's rows are split into chunks of <= 16, 32,
// 64 or 96 rows, and one MMA per 32 K columns covers a whole chunk. The chunks
// of one expert run side by side on neighbouring blocks and read each weight
// block from HBM once (the others find it in L2). Tensor time is small next to
// the weight stream, so the kernel stays bound by HBM, also at one token row.
//
// Work units, in the order the step counter hands them out (MB = 1 weight
// block per unit for chunks of <= 64 rows, MB = 2 for the 96-row chunks):
//   gate/up unit (chunk c, block b):
//       MB = 1: rows [64b, 64b + 64) of W_gate and of W_up as the MMA's A
//       operand (M = 128: 64 gate rows, then 64 up rows);
//       MB = 2: rows [128b, 128b + 128) of W_gate as block 0 and the same rows
//       of W_up as block 1 (two M = 128 MMAs per K step on one token tile);
//       the chunk's token rows of x (MXFP8) as B (N = rows rounded up to 16).
//       Epilogue: g, u -> bf16, h = bf16(silu(g) * u), h -> MXFP8 along I,
//       one 32-group per warp. Then ready[c] is bumped.
//   down unit (chunk c, block b): rows [128 MB b, 128 MB (b + 1)) of W_down
//       as A (MB blocks of 128 rows); the chunk's rows of h (MXFP8) as B. It
//       waits (bounded) until ready[c] counts every gate/up unit of c.
//       Epilogue: o[pair][h] in fp32, then the fused combine of every (token
//       row, 128-row block) this unit completes.
// Dynamic schedule: every block takes its next unit from the step's counter
// when it is about to need it, so blocks that stream faster take more units
// and all blocks finish within about one unit of each other (a static split of
// 512 KB and 256 KB units left the last blocks 10 to 25 us behind the first).
// The counter hands out every gate/up unit before any down unit, so a down
// unit only waits on gate/up units that blocks have already taken, and those
// never wait. The waits cannot form a cycle, and every wait is bounded anyway.
// Experts come in the chunk list's order, the shared expert first: its down
// units are the last contribution to every token row they cover, and at the
// end of the order they left a few blocks combining every row after the
// others had finished.
//
// Warp roles (10 warps):
//   warp 0      TMA producer: one lane takes the block's units from the
//               counter and queues them for the other roles; it loads the A
//               tiles (128 bytes of K x 64 or 128 rows per box, 128-byte
//               swizzle) into a ring of K chunks (5 stages of two chunks
//               with 16- and 32-row chunks, 4 of two with 64-row chunks, 4 of
//               one chunk of two weight blocks with 96-row chunks).
//   warp 1      MMA issuer: one lane issues tcgen05.mma.kind::mxf8f6f4
//               .block_scale (K = 32 each, 4 per K chunk and weight block)
//               into one of two sets of TMEM accumulators and commits each
//               stage back to the ring.
//   warps 2-5   loaders: gather the chunk's token rows into the B ring slot
//               with cp.async in the 128-byte swizzled K-major layout, with
//               the stage's UE8M0 scale words of A and B (the MMA issuer
//               moves those into TMEM with tcgen05.cp).
//   warps 6-9   epilogue: read the accumulators (tcgen05.ld), run the unit's
//               epilogue, and hand them back to the MMA issuer.
//
// Pages followed:
// - "Beyond Day-0: Optimizing DeepSeek-V4.1 Flash in SGLang", 2.1: group-32
//   FP8 weights and scales reorganised for Blackwell MXFP8 (here the canonical
//   K-major layout feeds the block-scaled MMA directly, with no copy), and
//   the reduction fused with the MXFP8 quantisation of its output.
// - Same page, 3.1: SwiGLU with the original intermediate rounding.
// - "FlyDSL Mono Kernels for High-Interactivity LLM Serving in ATOM",
//   "MiniMax-M3: Connecting Attention and Experts": persistent blocks, the
//   down weights loaded before h is ready, and tagged ready counters.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include "combine.cuh"
#include "device.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kKC = 128;                    // bytes (E4M3 values) of K per stage: 4 MMAs of K = 32
constexpr int kBM = 128;                    // MMA M (weight rows per unit)
constexpr int kABytes = kBM * kKC;          // 16 KB
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpLoad = 2, kWarpEpi = 6, kMWarps = 10;
constexpr int kMThreads = kMWarps * 32;
constexpr int kLoaders = 128;               // threads of the loader warps
constexpr int kEpiThreads = 128;            // threads of the epilogue warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kScaleSlotCols = 32;     // per stage: SFA at +0 (4 columns), SFB at +16 (4 columns)
constexpr int kBarEpi = 2, kBarGate = 3;   // named barriers (0 is __syncthreads)
constexpr int kUnitQ = 4;                   // entries of the block's unit queue
static_assert(kMmaDownRows == kBM, "unit geometry");

// One work unit, decoded.
struct MUnit {
  int u;       // unit index (-1: no more units)
  int down;    // 0: gate/up, 1: down
  int chunk;   // index into chunk_list
  int blk;     // 64-row block of I (gate/up) or 128-row block of H (down)
  int e;       // expert (E: the shared expert; -1: no more units)
  int start;   // first rank of the chunk within the expert's rows
  int n;       // token rows of the chunk (1..128)
  int npad;    // n rounded up to 16 (the MMA's N)
  int nch;     // chunks of the expert
};

// One instantiation per chunk size. A chunk of at most NMAX token rows is the
// MMA's N. A stage holds KPS K-chunks of 128 (MB weight tiles of 16 KB and one
// NMAX-row token tile each): more chunks per stage spread the per-stage costs
// of the MMA issuer (one barrier wait, one commit) over more MMAs.
// MB weight blocks per unit (M = 128 each) share the stage's token tile: with
// MB = 2 a unit covers 128 rows of I (gate/up) or 256 rows of H (down), and
// each token tile lands once per 256 weight rows instead of once per 128.
// The ring holds STAGES stages; smaller token tiles leave room for more.
template <int NMAX_, int STAGES_, int KPS_, int MB_ = 1>
struct MmaCfg {
  static constexpr int NMAX = NMAX_;
  static constexpr int STAGES = STAGES_;
  static constexpr int KPS = KPS_;
  static constexpr int MB = MB_;
  static constexpr int NPR = (NMAX + 31) / 32;                 // pair ids per epilogue lane
  static constexpr int BBYTES = NMAX * kKC;
  static constexpr uint32_t ACC_COLS = NMAX < 32 ? 32 : NMAX;  // TMEM columns per accumulator (one M block)
  static constexpr uint32_t BUF_COLS = MB * ACC_COLS;          // one unit's accumulators
  static constexpr uint32_t SCALE_COL0 = 2 * BUF_COLS;
  static constexpr uint32_t SLOT_COLS = KPS * kScaleSlotCols;  // TMEM scale columns per stage
  struct Smem {
    uint8_t a[STAGES][KPS][MB][kABytes];  // weight tiles, 128-byte swizzled K-major (TMA)
    uint8_t b[STAGES][KPS][BBYTES];       // token-row tiles, same layout (cp.async)
    uint32_t sfa[STAGES][KPS][MB][128];   // a chunk's 4 UE8M0 codes (one per 32 K) per weight row, TMEM image order
    uint32_t sfb[STAGES][KPS][128];       // the same per token row (rows past NMAX unused)
    uint16_t xchg[2][16][64];             // bf16 u of one 16-column slice, [column][i]
    uint32_t jobs[NMAX];                  // token rows whose combine a down unit completed
    uint64_t full[STAGES];                // A landed (TMA bytes, producer arrival) and B + scale words in place
                                          // (128 loader arrivals): one wait per stage for the MMA issuer
    uint64_t empty[STAGES];               // the stage's MMAs are done (tcgen05.commit)
    uint64_t acc_full[2];                 // accumulators complete (tcgen05.commit)
    uint64_t acc_empty[2];                // accumulators read out (128 epilogue arrivals)
    uint64_t mma_done;                    // every MMA of the block finished (before TMEM is freed)
    uint64_t uq_full[kUnitQ];             // queue entry written (producer)
    uint64_t uq_empty[kUnitQ];            // queue entry read by every consumer (MMA lane, loaders, epilogue)
    MUnit uq[kUnitQ];                     // the block's units in order, decoded (e = -1: no more)
    uint32_t tmem_base;
    uint32_t n_jobs;
  };
  static constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;  // + alignment of the ring to 1024 bytes
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(SCALE_COL0 + STAGES * SLOT_COLS <= kTmemCols, "TMEM budget");
  static_assert(NMAX % 16 == 0 && NMAX <= 96 && BBYTES % 1024 == 0, "token tile geometry");
  static_assert(MB == 1 || MB == 2, "one or two weight blocks per unit");
  static_assert(STAGES <= 11, "cp_async_wait_n covers at most 10 newer groups");
};
using Cfg16 = MmaCfg<16, 5, 2>;
using Cfg32 = MmaCfg<32, 5, 2>;
using Cfg64 = MmaCfg<64, 4, 2>;
using Cfg96x2 = MmaCfg<96, 4, 1, 2>;
using Cfg16x2 = MmaCfg<16, 5, 1, 2>;  // MXFP4 weights
using Cfg32x2 = MmaCfg<32, 5, 1, 2>;

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 16-byte copy global -> shared through L2; src_bytes = 0 writes 16 zero bytes.
__device__ __forceinline__ void cp_async16_zfill(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

// 4-byte copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async4_zfill(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Generic-proxy writes of this thread (cp.async) before later async-proxy reads (tcgen05.mma).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Barrier over n threads that also returns the AND of v over them. Every
// control decision taken by a group of warps goes through one, so the group
// always takes the same path through its barriers.
__device__ __forceinline__ int bar_and(int id, int n, int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.s32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.s32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v), "r"(id), "r"(n)
      : "memory");
  return r;
}

__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart, start address 16-byte granular.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);  // start address
  d |= uint64_t(1) << 16;                 // leading byte offset (unused with a 128-byte swizzle)
  d |= uint64_t(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 bytes
  d |= uint64_t(1) << 46;                 // descriptor version
  d |= uint64_t(2) << 61;                 // 128-byte swizzle
  return d;
}

// D (+)= (A * SFA) x (B * SFB)^T for K = 32; sf_id picks the byte of the scale words.
__device__ __forceinline__ void mma_mxf8(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Shared-memory descriptor of a 32-row x 16-byte matrix, no swizzle: 8-row
// core matrices of 128 bytes, 128 bytes apart.
__device__ __forceinline__ uint64_t sf_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFFu);  // start address
  d |= uint64_t(1) << 16;                 // leading byte offset: 16 bytes
  d |= uint64_t(128 >> 4) << 32;          // stride byte offset: 8 rows x 16 bytes
  d |= uint64_t(1) << 46;                 // descriptor version
  return d;                               // no swizzle
}

// 32 TMEM lanes x 4 columns from shared memory (16 bytes per lane), the same
// in each of the four 32-lane quadrants.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 16 consecutive fp32 columns of the warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ units and schedule


// An expert with cnt rows is split into ceil(cnt/NMAX) chunks of nearly equal
// size. The units of one expert are consecutive: for each of its blocks in
// order, every chunk of the expert. Neighbouring units run at about the same
// time on neighbouring blocks, so the chunks of a multi-chunk expert read
// each weight block from HBM once and from L2 after that.
template <int NMAX>
__device__ __forceinline__ MUnit decode_unit(const ExpertArgs &a, int u, int n_chunks, int mbg, int hbd) {
  MUnit m;
  m.u = u;
  const int ng = n_chunks * mbg;
  int nb;  // blocks per chunk
  if (u < ng) {
    m.down = 0;
    nb = mbg;
  } else {
    u -= ng;
    m.down = 1;
    nb = hbd;
  }
  const int ci0 = u / nb;  // a chunk of the unit's expert
  if (!in_bounds(a.status, a.diag, 10, ci0, a.n_tiles_max)) {
    m.u = m.e = -1;
    return m;
  }
  const int ent = __ldcg(a.chunk_list + ci0);
  m.e = ent >> 16;
  if (!in_bounds(a.status, a.diag, 11, m.e, a.E + 1)) {
    m.u = m.e = -1;
    return m;
  }
  const int cbase = ci0 - (ent & 0xFFFF);  // the expert's first chunk
  const int cnt = __ldcg(a.counts + m.e);
  m.nch = (cnt + NMAX - 1) / NMAX;
  const int w = u - cbase * nb;  // unit within the expert's span of nch * nb units
  m.blk = w / m.nch;
  const int c = w - m.blk * m.nch;
  m.chunk = cbase + c;
  const int cs = (cnt + m.nch - 1) / m.nch;
  m.start = c * cs;
  m.n = min(cs, cnt - m.start);
  m.npad = (m.n + 15) & ~15;
  if (!in_bounds(a.status, a.diag, 12, m.chunk, a.n_tiles_max) ||
      !in_bounds(a.status, a.diag, 13, int64_t(m.start) + m.n - 1, a.Tmax) ||
      !in_bounds(a.status, a.diag, 14, m.n - 1, NMAX)) {
    m.u = m.e = -1;
  }
  return m;
}

__device__ __forceinline__ bool aborted(const ExpertArgs &a) { return ld_volatile(a.work + 1) != 0; }

__device__ __forceinline__ void fail(const ExpertArgs &a, int64_t site, int64_t unit, int64_t where, int64_t seen,
                                     int64_t expected, int64_t ns) {
  report_diag(a.status, a.diag, MOE_ERR_TIMEOUT, site, unit, where, seen, expected, ns, 0);
  atomicExch(a.work + 1, 1u);
}

// ------------------------------------------------------------------ unit queue
// Units are handed out while the kernel runs: the TMA producer takes the next
// unit index from the step's counter (work[0], zeroed by the route kernel) and
// passes it to the block's other roles through a queue of kUnitQ entries in
// shared memory. Blocks that stream faster take more units, so the blocks
// finish within about one unit of each other. The counter hands out every
// gate/up unit before any down unit, so a down unit only ever waits for gate/up
// units that some block has already taken.

// Entry i of the queue (blocking, bounded); e = -1 after a timeout.
template <class C>
__device__ __forceinline__ MUnit queue_pop(const ExpertArgs &a, typename C::Smem &sm, uint32_t i) {
  const uint32_t qs = i % kUnitQ;
  int64_t waited = 0;
  MUnit m = {};
  if (!mbar_wait(&sm.uq_full[qs], (i / kUnitQ) & 1u, a.timeout_ns, &waited)) {
    fail(a, kDiagQueueWait, -1, qs, i, -16, waited);
    m.u = m.e = -1;
    return m;
  }
  m = sm.uq[qs];
  mbar_arrive(&sm.uq_empty[qs]);
  return m;
}

// ------------------------------------------------------------------ TMA producer (one lane)

template <class C>
__device__ void mma_producer(const MmaMaps &maps, const ExpertArgs &a, typename C::Smem &sm, int n_chunks, int mbg,
                             int hbd) {
  constexpr int kMStages = C::STAGES;
  const uint64_t pol_first = l2_evict_first_policy(), pol_normal = l2_evict_normal_policy();
  // MXFP4 boxes move half the bytes (the transaction count is the packed
  // global bytes; each 16-code group lands in 16 bytes of shared memory)
  const uint32_t a_tx_bytes = a.fp4 ? kABytes / 2 : kABytes;
  const int total = n_chunks * (mbg + hbd);
  uint32_t g = 0;  // stages issued
  uint32_t q = 0;  // queue entries published
  // Decode unit u (-1, or past the last unit: the end of the work) into the
  // next queue entry. Consumers read the decoded unit from shared memory.
  const auto publish = [&](int u) -> MUnit {
    MUnit d = {};
    d.u = d.e = -1;
    if (u >= 0 && u < total && !aborted(a)) d = decode_unit<C::NMAX>(a, u, n_chunks, mbg, hbd);
    const uint32_t qs = q % kUnitQ;
    int64_t waited = 0;
    if (!mbar_wait(&sm.uq_empty[qs], ((q / kUnitQ) & 1u) ^ 1u, a.timeout_ns, &waited)) {
      fail(a, kDiagQueueWait, u, qs, q, -17, waited);
      d.u = d.e = -1;
      return d;  // not published: the consumers' waits end at their limit
    }
    sm.uq[qs] = d;
    mbar_arrive(&sm.uq_full[qs]);
    ++q;
    return d;
  };
  // Block b starts with unit b; the counter hands out units G, G + 1, ...
  MUnit m = publish(int(blockIdx.x));
  while (m.e >= 0) {
    const bool sh = m.e == a.E;
    // the chunks of a multi-chunk expert read the same weights at about the same time
    const uint64_t pol = m.nch > 1 ? pol_normal : pol_first;
    const int kcs = (m.down ? a.I : a.H) / kKC;
    const int nst = (kcs + C::KPS - 1) / C::KPS;  // stages of the unit
    // The next unit is taken four stages before this unit's last stage and
    // published two stages before it, so the other roles find it decoded
    // when they reach the end of this unit.
    const int st_take = nst > 4 ? nst - 4 : 0, st_pub = nst > 2 ? nst - 2 : 0;
    int nxt = -1;
    MUnit mn = {};
    mn.u = mn.e = -2;  // not published yet
    bool ok = true;
    for (int st = 0; st < nst; ++st) {
      if (st == st_take) nxt = int(gridDim.x + atomicAdd(a.work, 1u));
      if (st == st_pub) mn = publish(nxt);
      const int kc0 = st * C::KPS;
      const int s = int(g % kMStages);
      const uint32_t ph = (g / kMStages) & 1u;
      const int nck = kcs - kc0 < C::KPS ? kcs - kc0 : C::KPS;
      int64_t waited = 0;
      if (!mbar_wait(&sm.empty[s], ph ^ 1u, a.timeout_ns, &waited)) {
        fail(a, kDiagEmptyWait, m.u, s, kc0, -10, waited);
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(&sm.full[s], a_tx_bytes * uint32_t(nck * C::MB));
      for (int j = 0; j < nck; ++j) {
        const int kc = kc0 + j;
        if (C::MB == 2 && !m.down) {
          // gate rows 128 blk .. 128 blk + 127 into tile 0, the same rows of W_up into tile 1
          const int y = (sh ? 0 : m.e * a.I) + m.blk * kBM;
          if (in_bounds(a.status, a.diag, 15, y, int64_t(sh ? 1 : a.E) * a.I - (kBM - 1))) {
            tma_load_2d(sm.a[s][j][0], sh ? &maps.sh_gate2 : &maps.gate2, kc * kKC, y, &sm.full[s], pol);
            tma_load_2d(sm.a[s][j][C::MB - 1], sh ? &maps.sh_up2 : &maps.up2, kc * kKC, y, &sm.full[s], pol);
          }
          continue;
        }
#pragma unroll
        for (int mb = 0; mb < C::MB; ++mb) {
          if (!m.down) {
            const int y = (sh ? 0 : m.e * a.I) + (m.blk * C::MB + mb) * 64;
            if (!in_bounds(a.status, a.diag, 15, y, int64_t(sh ? 1 : a.E) * a.I - 63)) continue;
            tma_load_2d(sm.a[s][j][mb], sh ? &maps.sh_gate : &maps.gate, kc * kKC, y, &sm.full[s], pol);
            tma_load_2d(sm.a[s][j][mb] + kABytes / 2, sh ? &maps.sh_up : &maps.up, kc * kKC, y, &sm.full[s], pol);
          } else {
            const int y = (sh ? 0 : m.e * a.H) + (m.blk * C::MB + mb) * kBM;
            if (!in_bounds(a.status, a.diag, 16, y, int64_t(sh ? 1 : a.E) * a.H - (kBM - 1))) continue;
            tma_load_2d(sm.a[s][j][mb], sh ? &maps.sh_down : &maps.down, kc * kKC, y, &sm.full[s], pol);
          }
        }
      }
      ++g;
    }
    if (!ok) {
      // a failed unit ends the block's work (the abort flag is up); an end
      // entry follows the last unit published
      if (mn.e != -1) publish(-1);
      break;
    }
    m = mn;
  }
  // No copy may still be in flight when the block exits: wait for the last
  // load of every slot (already complete unless the MMA side stopped early).
  const uint32_t last = g < uint32_t(kMStages) ? g : uint32_t(kMStages);
  for (uint32_t j = 1; j <= last; ++j) {
    const uint32_t gg = g - j;
    mbar_wait(&sm.full[gg % kMStages], (gg / kMStages) & 1u, a.timeout_ns);
  }
}

// ------------------------------------------------------------------ MMA issuer (one lane)

template <class C>
__device__ void mma_issuer(const ExpertArgs &a, typename C::Smem &sm, uint32_t tmem, int n_chunks, int mbg,
                           int hbd) {
  constexpr int kMStages = C::STAGES;
  uint32_t g = 0, nu = 0;  // stages consumed, units done
  for (uint32_t i = 0;; ++i) {
    const MUnit m = queue_pop<C>(a, sm, i);
    if (m.e < 0 || aborted(a)) break;
    const int acc = int(nu & 1u);
    const uint32_t aph = (nu >> 1) & 1u;
    int64_t waited = 0;
    if (!mbar_wait(&sm.acc_empty[acc], aph ^ 1u, a.timeout_ns, &waited)) {
      fail(a, kDiagEmptyWait, m.u, acc, -1, -11, waited);
      break;
    }
    tmem_fence_after();
    const uint32_t d = tmem + uint32_t(acc) * C::BUF_COLS;
    // kind::mxf8f6f4, A E4M3 (or E2M1 for MXFP4 weights, format 5), B E4M3,
    // K-major, UE8M0 scales, N = npad, M = 128
    const uint32_t idesc = (1u << 23) | (uint32_t(m.npad >> 3) << 17) | (uint32_t(kBM >> 4) << 24) |
                           (a.fp4 ? (5u << 7) : 0u);
    const int kcs = (m.down ? a.I : a.H) / kKC;
    bool ok = true;
    for (int kc0 = 0; kc0 < kcs; kc0 += C::KPS) {
      const int s = int(g % kMStages);
      const uint32_t ph = (g / kMStages) & 1u;
      const int nck = kcs - kc0 < C::KPS ? kcs - kc0 : C::KPS;
      if (!mbar_wait(&sm.full[s], ph, a.timeout_ns, &waited)) {
        fail(a, kDiagFullWait, m.u, s, kc0, -12, waited);
        ok = false;
        break;
      }
      tmem_fence_after();
      for (int j = 0; j < nck; ++j) {
        // scale slot of the chunk: SFA of weight block mb at +8 mb (4 columns each), SFB at +16
        const uint32_t sfa = tmem + C::SCALE_COL0 + uint32_t(s) * C::SLOT_COLS + uint32_t(j) * kScaleSlotCols;
        const uint32_t sfb = sfa + 16;
        // the chunk's scale words into TMEM (in issue order before the MMAs that read them)
#pragma unroll
        for (int mb = 0; mb < C::MB; ++mb) tmem_cp_32x128b_x4(sfa + 8u * mb, sf_desc(smem_u32(sm.sfa[s][j][mb])));
        tmem_cp_32x128b_x4(sfb, sf_desc(smem_u32(sm.sfb[s][j])));
        const uint64_t bdesc = sw128_desc(smem_u32(sm.b[s][j]));
#pragma unroll
        for (int mb = 0; mb < C::MB; ++mb) {
          const uint64_t adesc = sw128_desc(smem_u32(sm.a[s][j][mb]));
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            // +32 bytes of K per step: +2 in the descriptor's 16-byte start-address field
            mma_mxf8(d + uint32_t(mb) * C::ACC_COLS, adesc + uint64_t(2 * k4), bdesc + uint64_t(2 * k4),
                     idesc | (uint32_t(k4) << 4) | (uint32_t(k4) << 29), sfa + 8u * mb, sfb,
                     (kc0 + j + k4) != 0 ? 1u : 0u);
          }
        }
      }
      mma_commit(&sm.empty[s]);
      ++g;
    }
    if (!ok) break;
    mma_commit(&sm.acc_full[acc]);
    ++nu;
  }
  // every MMA issued must finish before TMEM is freed
  mma_commit(&sm.mma_done);
  mbar_wait(&sm.mma_done, 0, a.timeout_ns);
}

// ------------------------------------------------------------------ loaders (warps 2-5)
// Thread tau (0..127) copies 16-byte column tau % 8 of rows tau/8 + 16 i of the
// B tile, and the stage's scale word (4 UE8M0 codes, one per 32 K) of weight
// row tau and of token row tau. The scale words go to shared memory in the
// order of their TMEM image (word 4 l + c holds row l + 32 c; the MMA issuer
// copies them with tcgen05.cp). Each thread runs its own pipeline and meets
// no other thread: it issues a stage as soon as the ring slot is free, and
// when it cannot issue, it waits for its oldest stage in flight and arrives
// on that stage's full barrier (fence.proxy.async first: the copies were written
// through the generic proxy, the MMA reads through the async proxy).

template <int NMAX, int MB>
struct LoaderRows {
  const uint8_t *b[NMAX / 16];  // row i: token (pair) row r = tau/8 + 16 i of the chunk, its K-major codes
  const uint8_t *sfa[MB];  // scale row of weight row tau of each weight block
  const uint8_t *sfb;      // scale row of token row tau (or NULL past the chunk)
};

template <int NMAX, int MB>
__device__ __forceinline__ LoaderRows<NMAX, MB> loader_rows(const ExpertArgs &a, int T, const MUnit &m, int tau) {
  LoaderRows<NMAX, MB> lr;
  const int32_t *rows = a.rows_of + int64_t(m.e) * a.Tmax + m.start;
  const int64_t tk = int64_t(T) * a.k;
  const int r0 = tau >> 3;
#pragma unroll
  for (int i = 0; i < NMAX / 16; ++i) {
    const int r = r0 + 16 * i;
    lr.b[i] = nullptr;
    if (r < m.n) {
      const int64_t p = __ldcg(rows + r);
      const int64_t t = p < tk ? p / a.k : p - tk;
      if (in_bounds(a.status, a.diag, 17, p, a.pairs_cap) && in_bounds(a.status, a.diag, 18, t, a.Tmax))
        lr.b[i] = m.down ? a.hq + p * a.I : a.xq + t * a.H;
    }
  }
  lr.sfb = nullptr;
  if (tau < m.n) {
    const int64_t p = __ldcg(rows + tau);
    const int64_t t = p < tk ? p / a.k : p - tk;
    if (in_bounds(a.status, a.diag, 17, p, a.pairs_cap) && in_bounds(a.status, a.diag, 18, t, a.Tmax))
      lr.sfb = m.down ? a.hs + p * (a.I / kGroup) : a.xs + t * (a.H / kGroup);
  }
  const bool sh = m.e == a.E;
#pragma unroll
  for (int mb = 0; mb < MB; ++mb) {
    if (!m.down) {
      // one block: rows 64 blk .. + 63 of W_gate then of W_up; two blocks: block 0 is
      // rows 128 blk .. + 127 of W_gate, block 1 the same rows of W_up
      int64_t row = (sh ? 0 : int64_t(m.e) * a.I) +
                    (MB == 2 ? int64_t(m.blk) * kBM + tau : int64_t(m.blk * MB + mb) * 64 + (tau & 63));
      if (!in_bounds(a.status, a.diag, 19, row, int64_t(sh ? 1 : a.E) * a.I)) row = 0;
      const bool gate = MB == 2 ? mb == 0 : tau < 64;
      const uint8_t *base = gate ? (sh ? a.sh_s_gate : a.s_gate) : (sh ? a.sh_s_up : a.s_up);
      lr.sfa[mb] = base + row * (a.H / kGroup);
    } else {
      int64_t row = (sh ? 0 : int64_t(m.e) * a.H) + int64_t(m.blk * MB + mb) * kBM + tau;
      if (!in_bounds(a.status, a.diag, 20, row, int64_t(sh ? 1 : a.E) * a.H)) row = 0;
      lr.sfa[mb] = (sh ? a.sh_s_down : a.s_down) + row * (a.I / kGroup);
    }
  }
  return lr;
}

// Issue the copies of stage slot s for K chunks kc0 .. kc0 + nck - 1 (one cp.async group).
template <class C>
__device__ __forceinline__ void loader_issue(typename C::Smem &sm, const MUnit &m, const LoaderRows<C::NMAX, C::MB> &lr,
                                             int s, int kc0, int nck, int tau, const void *zero_src) {
  const int c8 = tau & 7, r0 = tau >> 3;
  const int w = (tau & 31) * 4 + (tau >> 5);  // TMEM image order
#pragma unroll
  for (int j = 0; j < C::KPS; ++j) {
    if (j >= nck) break;
    const int kc = kc0 + j;
    uint8_t *bs = sm.b[s][j];
#pragma unroll
    for (int i = 0; i < C::NMAX / 16; ++i) {
      const int r = r0 + 16 * i;
      if (r < m.npad) {
        const bool v = lr.b[i] != nullptr;
        cp_async16_zfill(bs + r * kKC + ((c8 ^ (r & 7)) << 4), v ? lr.b[i] + kc * kKC + c8 * 16 : zero_src,
                         v ? 16u : 0u);
      }
    }
#pragma unroll
    for (int mb = 0; mb < C::MB; ++mb) cp_async4_zfill(&sm.sfa[s][j][mb][w], lr.sfa[mb] + kc * 4, 4u);
    cp_async4_zfill(&sm.sfb[s][j][w], lr.sfb ? lr.sfb + kc * 4 : zero_src, lr.sfb ? 4u : 0u);
  }
  cp_async_commit();
}

// Wait until at most n (<= 10) of this thread's copy groups are still in flight.
__device__ __forceinline__ void cp_async_wait_n(uint32_t n) {
  switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    case 7: cp_async_wait<7>(); break;
    case 8: cp_async_wait<8>(); break;
    case 9: cp_async_wait<9>(); break;
    default: cp_async_wait<10>(); break;
  }
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ int wait_chunk_ready(const ExpertArgs &a, int chunk, uint32_t target, int u) {
  const WaitClock wc;
  uint32_t seen;
  while ((seen = ld_acquire_gpu(a.ready + chunk)) < target) {
    if (wc.expired(a.timeout_ns)) {
      report_diag(a.status, a.diag, MOE_ERR_TIMEOUT, kDiagReadyWait, u, chunk, seen, target, wc.ns(), wc.cycles());
      atomicExch(a.work + 1, 1u);
      return 0;
    }
    __nanosleep(128);
  }
  return 1;
}

template <class C>
__device__ void mma_loaders(const ExpertArgs &a, int T, typename C::Smem &sm, int n_chunks, int mbg, int hbd) {
  constexpr int kMStages = C::STAGES;
  const int tau = int(threadIdx.x) - kWarpLoad * 32;
  const void *zero_src = a.xq;  // any valid address: zero-byte copies read nothing
  uint32_t g = 0, gc = 0;       // stages issued, stages signalled (this thread's)
  // this thread's oldest stage in flight: copies landed -> fence -> arrive
  auto complete_oldest = [&]() {
    cp_async_wait_n(g - gc - 1);
    fence_proxy_async();
    mbar_arrive(&sm.full[gc % kMStages]);
    ++gc;
  };
  MUnit m;
  LoaderRows<C::NMAX, C::MB> lr;
  int kc = 0, kcs = 0;
  uint32_t next = 0;  // queue entries read
  while (true) {
    if (kc == kcs) {  // start the next unit
      // the stages in flight keep reaching the MMA while the entry is not there yet
      if (gc < g && !mbar_test(&sm.uq_full[next % kUnitQ], (next / kUnitQ) & 1u)) {
        complete_oldest();
        continue;
      }
      m = queue_pop<C>(a, sm, next++);
      if (m.e < 0 || aborted(a)) break;
      if (m.down && ld_acquire_gpu(a.ready + m.chunk) < uint32_t(mbg)) {
        // h of the chunk is not complete: everything in flight reaches the MMA
        // before this thread waits on other blocks
        while (gc < g) complete_oldest();
        if (!wait_chunk_ready(a, m.chunk, uint32_t(mbg), m.u)) break;
      }
      lr = loader_rows<C::NMAX, C::MB>(a, T, m, tau);
      kc = 0;
      kcs = (m.down ? a.I : a.H) / kKC;
    }
    const int s = int(g % kMStages);
    const uint32_t ph = (g / kMStages) & 1u;
    if (g - gc < uint32_t(kMStages) && mbar_test(&sm.empty[s], ph ^ 1u)) {
      const int nck = kcs - kc < C::KPS ? kcs - kc : C::KPS;
      loader_issue<C>(sm, m, lr, s, kc, nck, tau, zero_src);
      ++g;
      kc += nck;
      continue;
    }
    if (gc < g) {
      complete_oldest();
      continue;
    }
    int64_t waited = 0;
    if (!mbar_wait(&sm.empty[s], ph ^ 1u, a.timeout_ns, &waited)) {
      fail(a, kDiagEmptyWait, -1, s, kc, -14, waited);
      break;
    }
  }
  while (gc < g) complete_oldest();
}

// ------------------------------------------------------------------ epilogue (warps 6-9)

// Pair id of accumulator column col (0 .. NMAX - 1): lane l of the warp holds
// the pair ids of columns l, 32 + l, 64 + l in prs[0], prs[1], prs[2].
template <int NPR>
__device__ __forceinline__ int pair_of_col(const int (&prs)[NPR], int col) {
  int src = prs[0];
  if constexpr (NPR == 2) src = col < 32 ? prs[0] : prs[1];
  if constexpr (NPR == 3) src = col < 32 ? prs[0] : (col < 64 ? prs[1] : prs[2]);
  return __shfl_sync(0xFFFFFFFFu, src, col & 31);
}

template <class C>
__device__ void mma_epilogue(const ExpertArgs &a, int T, typename C::Smem &sm, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, ew = warp - kWarpEpi;
  const int et = ew * 32 + lane;
  const int64_t tk = int64_t(T) * a.k;
  const uint32_t target = uint32_t(a.k + a.shared);
  const float lim = a.swiglu_limit;
  const int hcb = a.H / kBM;  // combine blocks (128 columns of y) per token row
  uint32_t nu = 0, xc = 0;    // units done, gate/up column slices done
  for (uint32_t i = 0;; ++i) {
    const MUnit m = queue_pop<C>(a, sm, i);
    // every epilogue thread read the same entry (or timed out): they leave together
    if (!bar_and(kBarEpi, kEpiThreads, m.e >= 0 ? 1 : 0)) break;
    const int acc = int(nu & 1u);
    const uint32_t aph = (nu >> 1) & 1u;
    // pair ids of columns lane, 32 + lane, ... of the chunk (-1 past its end), loaded before the wait
    const int32_t *rows = a.rows_of + int64_t(m.e) * a.Tmax + m.start;
    int prs[C::NPR];
#pragma unroll
    for (int r = 0; r < C::NPR; ++r) {
      prs[r] = 32 * r + lane < m.n ? __ldcg(rows + 32 * r + lane) : -1;
      if (prs[r] >= 0 && !in_bounds(a.status, a.diag, 21, prs[r], a.pairs_cap)) prs[r] = -1;
    }
    int ok = !aborted(a);
    if (ok) {
      int64_t waited = 0;
      ok = mbar_wait(&sm.acc_full[acc], aph, a.timeout_ns, &waited) ? 1 : 0;
      if (!ok) fail(a, kDiagFullWait, m.u, acc, -1, -15, waited);
    }
    if (!bar_and(kBarEpi, kEpiThreads, ok)) break;
    tmem_fence_after();
    const int slices = m.npad / 16;
    if (C::MB == 2 && !m.down) {
      // Two-block gate/up unit: accumulator 0 holds gate rows 128 blk + 32 q + lane
      // in this warp's TMEM lanes, accumulator 1 the same rows of the up
      // projection. Every warp forms h for its 32 rows (one MXFP8 group) itself.
      const uint32_t ta = tmem + (uint32_t(32 * q) << 16) + uint32_t(acc) * C::BUF_COLS;
      const int64_t col = int64_t(m.blk) * kBM + 32 * q + lane;
      for (int j = 0; j < slices; ++j) {
        float gv[16], uv[16];
        tmem_ld16(ta + uint32_t(16 * j), gv);
        tmem_ld16(ta + C::ACC_COLS + uint32_t(16 * j), uv);
#pragma unroll 4
        for (int c = 0; c < 16; ++c) {
          const int p = pair_of_col<C::NPR>(prs, 16 * j + c);
          if (p < 0) continue;  // the same for the whole warp
          float gb = bf16_bits_to_float(float_to_bf16_bits(gv[c]));
          float ub = bf16_bits_to_float(float_to_bf16_bits(uv[c]));
          if (lim > 0.0f) {  // clipped SwiGLU
            gb = fminf(gb, lim);
            ub = fminf(fmaxf(ub, -lim), lim);
          }
          const float silu = gb / (1.0f + expf(-gb));
          const uint16_t hb = float_to_bf16_bits(silu * ub);
          const uint32_t amax = __reduce_max_sync(0xFFFFFFFFu, uint32_t(hb) & 0x7FFFu);
          const uint32_t code = mx_scale_code(bf16_bits_to_float(uint16_t(amax)));
          a.hq[int64_t(p) * a.I + col] = float_to_e4m3(mx_unscale(bf16_bits_to_float(hb), code));
          if (lane == 0) a.hs[int64_t(p) * (a.I / kGroup) + m.blk * 4 + q] = uint8_t(code);
          if (a.h_bf16) a.h_bf16[int64_t(p) * a.I + col] = hb;
        }
      }
      tmem_fence_before();
      mbar_arrive(&sm.acc_empty[acc]);
      // every warp's h stores, then one release of the ready count
      named_bar(kBarEpi, kEpiThreads);
      if (et == 0 && m.chunk != a.skip_ready_tile) {
        __threadfence();
        red_release_gpu_add(a.ready + m.chunk, 1u);
      }
    } else if (!m.down) {
      // Per weight block mb (64 rows of I): lanes of quadrants 0, 1 hold gate
      // rows 64 blk + 32 q + lane; quadrants 2, 3 the up rows.
#pragma unroll 1
      for (int mb = 0; mb < C::MB; ++mb) {
        const uint32_t ta = tmem + (uint32_t(32 * q) << 16) + uint32_t(acc) * C::BUF_COLS + uint32_t(mb) * C::ACC_COLS;
        const int blk = m.blk * C::MB + mb;
        for (int j = 0; j < slices; ++j, ++xc) {
          float v[16];
          tmem_ld16(ta + uint32_t(16 * j), v);
          uint16_t(*xb)[64] = sm.xchg[xc & 1u];
          if (q >= 2) {
#pragma unroll
            for (int c = 0; c < 16; ++c) xb[c][32 * (q - 2) + lane] = float_to_bf16_bits(v[c]);
          }
          named_bar(kBarEpi, kEpiThreads);
          if (q < 2) {
            const int64_t col = int64_t(blk) * 64 + 32 * q + lane;
#pragma unroll 4
            for (int c = 0; c < 16; ++c) {
              const int p = pair_of_col<C::NPR>(prs, 16 * j + c);
              if (p < 0) continue;  // the same for the whole warp
              float gb = bf16_bits_to_float(float_to_bf16_bits(v[c]));
              float ub = bf16_bits_to_float(xb[c][32 * q + lane]);
              if (lim > 0.0f) {  // clipped SwiGLU
                gb = fminf(gb, lim);
                ub = fminf(fmaxf(ub, -lim), lim);
              }
              const float silu = gb / (1.0f + expf(-gb));
              const uint16_t hb = float_to_bf16_bits(silu * ub);
              const uint32_t amax = __reduce_max_sync(0xFFFFFFFFu, uint32_t(hb) & 0x7FFFu);
              const uint32_t code = mx_scale_code(bf16_bits_to_float(uint16_t(amax)));
              a.hq[int64_t(p) * a.I + col] = float_to_e4m3(mx_unscale(bf16_bits_to_float(hb), code));
              if (lane == 0) a.hs[int64_t(p) * (a.I / kGroup) + blk * 2 + q] = uint8_t(code);
              if (a.h_bf16) a.h_bf16[int64_t(p) * a.I + col] = hb;
            }
          }
        }
      }
      tmem_fence_before();
      mbar_arrive(&sm.acc_empty[acc]);
      if (q < 2) {
        // The two gate warps' h stores, then one release of the ready count: the
        // barrier orders them before the fence of the publishing thread.
        named_bar(kBarGate, 64);
        if (q == 0 && lane == 0 && m.chunk != a.skip_ready_tile) {
          __threadfence();
          red_release_gpu_add(a.ready + m.chunk, 1u);
        }
      }
    } else {
#pragma unroll 1
      for (int mb = 0; mb < C::MB; ++mb) {
        const uint32_t ta = tmem + (uint32_t(32 * q) << 16) + uint32_t(acc) * C::BUF_COLS + uint32_t(mb) * C::ACC_COLS;
        const int64_t h = int64_t(m.blk * C::MB + mb) * kBM + 32 * q + lane;
        for (int j = 0; j < slices; ++j) {
          float v[16];
          tmem_ld16(ta + uint32_t(16 * j), v);
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int p = pair_of_col<C::NPR>(prs, 16 * j + c);
            if (p >= 0) a.o[int64_t(p) * a.H + h] = v[c];
          }
        }
      }
      tmem_fence_before();
      mbar_arrive(&sm.acc_empty[acc]);
      // Count each pair in for (token row, block): after the barrier, the counting
      // thread's fence orders every warp's o stores of the unit before its count.
      // The last of a row's k (+ shared) pairs queues the row's combine.
      named_bar(kBarEpi, kEpiThreads);
      // epilogue warp w counts columns 32 w .. 32 w + 31
      int pc = ew == 0 ? prs[0] : -1;
      if constexpr (C::NPR == 2) pc = ew == 0 ? prs[0] : (ew == 1 ? prs[1] : -1);
      if constexpr (C::NPR == 3) pc = ew == 0 ? prs[0] : (ew == 1 ? prs[1] : (ew == 2 ? prs[2] : -1));
#pragma unroll 1
      for (int mb = 0; mb < C::MB; ++mb) {
        const int blk = m.blk * C::MB + mb;
        if (pc >= 0) {
          const int t = int(pc < tk ? pc / a.k : pc - tk);
          __threadfence();
          if (in_bounds(a.status, a.diag, 22, int64_t(t) * hcb + blk, a.comb_cap) &&
              atomicAdd(a.comb_cnt + int64_t(t) * hcb + blk, 1u) == target - 1u) {
            const uint32_t idx = atomicAdd(&sm.n_jobs, 1u);
            if (in_bounds(a.status, a.diag, 23, idx, C::NMAX)) sm.jobs[idx] = uint32_t(t);
          }
        }
        named_bar(kBarEpi, kEpiThreads);
        uint32_t nj = *reinterpret_cast<volatile uint32_t *>(&sm.n_jobs);
        if constexpr (kBoundsChecked) nj = min(nj, uint32_t(C::NMAX));  // entries past NMAX were not stored
        if (nj) {
          __threadfence();  // the other pairs' o stores, before these reads
          for (uint32_t jj = uint32_t(ew); jj < nj; jj += 4) {
            const int t = int(sm.jobs[jj]);
            if (!in_bounds(a.status, a.diag, 24, t, T)) continue;
            uint16_t yb[kBM / 32];
            combine_row_block<kBM / 32>(a.o, a.topk_w, a.y, T, a.k, a.shared, a.H, t, int64_t(blk) * kBM, lane, yb);
          }
        }
        named_bar(kBarEpi, kEpiThreads);
        if (et == 0) sm.n_jobs = 0;
        if constexpr (C::MB > 1) {
          if (mb + 1 < C::MB) named_bar(kBarEpi, kEpiThreads);  // the reset, before the next block's counts
        }
      }
    }
    ++nu;
  }
}

// ------------------------------------------------------------------ kernel

template <class C>
__global__ void __launch_bounds__(kMThreads, 1) experts_mma_kernel(const __grid_constant__ MmaMaps maps,
                                                                   const ExpertArgs a) {
  constexpr int kMStages = C::STAGES;
  extern __shared__ unsigned char mma_smem_raw[];
  typename C::Smem &sm =
      *reinterpret_cast<typename C::Smem *>((reinterpret_cast<uintptr_t>(mma_smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMStages; ++i) {
      mbar_init(&sm.full[i], 1 + kLoaders);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.acc_full[i], 1);
      mbar_init(&sm.acc_empty[i], kEpiThreads);
    }
    mbar_init(&sm.mma_done, 1);
    for (int i = 0; i < kUnitQ; ++i) {
      mbar_init(&sm.uq_full[i], 1);
      mbar_init(&sm.uq_empty[i], 1 + kLoaders + kEpiThreads);
    }
    sm.n_jobs = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // Everything below reads the router's outputs.
  pdl_wait_primary();
  // A dependent kernel (the residual-stream epilogue) may now be scheduled;
  // it waits for this grid to complete before it reads y.
  pdl_launch_dependents();
  // the step's row count: a.T, or the device-side value (clamped as the route kernel does)
  int T = a.T;
  if (a.d_T) {
    const int td = *reinterpret_cast<const volatile int32_t *>(a.d_T);
    T = td < 0 ? 0 : (td > a.Tmax ? a.Tmax : td);
  }
  const int n_chunks = __ldcg(a.n_chunks);
  // units per chunk: gate/up units of MB x 64 rows of I, down units of MB x 128 rows of H
  const int mbg = a.I / (64 * C::MB), hbd = a.H / (kBM * C::MB);
  if (warp == kWarpTma) {
    if (lane == 0) mma_producer<C>(maps, a, sm, n_chunks, mbg, hbd);
  } else if (warp == kWarpMma) {
    if (lane == 0) mma_issuer<C>(a, sm, tmem, n_chunks, mbg, hbd);
  } else if (warp < kWarpEpi) {
    mma_loaders<C>(a, T, sm, n_chunks, mbg, hbd);
  } else {
    mma_epilogue<C>(a, T, sm, tmem);
  }
  __syncwarp();
  tmem_fence_before();
  __syncthreads();
  tmem_fence_after();
  if (warp == kWarpMma)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// rows x k matrix of 8-bit codes (fp4 = false) or packed 4-bit codes (fp4 =
// true, two per byte), row-major; boxes of 128 codes x box_rows, 128-byte
// swizzle. Packed 4-bit boxes land as 16 codes per 16 bytes of shared memory
// (8 bytes of codes, 8 bytes of padding): the layout the block-scaled MMA
// reads E2M1 operands in, with the same 128-byte rows as 8-bit codes.
bool encode_rows(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *map, const void *base, uint64_t k, uint64_t rows,
                 uint32_t box_rows, bool fp4) {
  const cuuint64_t dims[2] = {k, rows};
  const cuuint64_t strides[1] = {fp4 ? k / 2 : k};
  const cuuint32_t box[2] = {uint32_t(kKC), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
             const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// K chunks of 128 codes, 64-row gate/up blocks, 128-row down blocks.
bool experts_mma_shape_supported(int H, int I) {
  return H >= 128 && I >= 128 && H % 128 == 0 && I % 128 == 0 && H <= 16384 && I <= 16384;
}

bool encode_mma_maps(const moe_config_t &c, const moe_weights_t &w, MmaMaps *maps) {
  memset(maps, 0, sizeof(MmaMaps));
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const uint64_t H = uint64_t(c.hidden), I = uint64_t(c.intermediate), E = uint64_t(c.num_experts);
  const bool f4 = c.weight_format == MOE_WEIGHTS_MXFP4;
  bool ok = encode_rows(enc, &maps->gate, w.w_gate, H, E * I, 64, f4) &&
            encode_rows(enc, &maps->up, w.w_up, H, E * I, 64, f4) &&
            encode_rows(enc, &maps->down, w.w_down, I, E * H, kBM, f4) &&
            encode_rows(enc, &maps->gate2, w.w_gate, H, E * I, kBM, f4) &&
            encode_rows(enc, &maps->up2, w.w_up, H, E * I, kBM, f4);
  if (ok && c.num_shared)
    ok = encode_rows(enc, &maps->sh_gate, w.sh_w_gate, H, I, 64, f4) &&
         encode_rows(enc, &maps->sh_up, w.sh_w_up, H, I, 64, f4) &&
         encode_rows(enc, &maps->sh_down, w.sh_w_down, I, H, kBM, f4) &&
         encode_rows(enc, &maps->sh_gate2, w.sh_w_gate, H, I, kBM, f4) &&
         encode_rows(enc, &maps->sh_up2, w.sh_w_up, H, I, kBM, f4);
  return ok;
}

namespace {

template <class C>
cudaError_t prepare_cfg() {
  return cudaFuncSetAttribute(experts_mma_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(C::SMEM_BYTES));
}

template <class C>
cudaError_t launch_cfg(const MmaMaps &maps, const ExpertArgs &a, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, experts_mma_kernel<C>, maps, a);
}

}  // namespace

// Chunk size. A chunk never holds more rows than the step (an expert has at
// most T rows), so T <= 16 uses 16-row chunks, up to 128 rows 32-row chunks
// (a 5-stage ring). Above 128 rows the hot experts hold many rows, and each
// chunk lands the expert's weight tiles in shared memory again, and each unit
// lands the chunk's token tile again: 96-row chunks with two 128-row weight
// blocks per unit (sharing one token tile; a 4-stage ring) land the fewest
// bytes, when H is a multiple of 256; otherwise 64-row chunks with one block.
int mma_chunk_rows(int T, int H) { return T <= 16 ? 16 : (T <= 128 ? 32 : (H % 256 == 0 ? 96 : 64)); }

cudaError_t prepare_experts_mma() {
  cudaError_t e = prepare_cfg<Cfg16>();
  if (e == cudaSuccess) e = prepare_cfg<Cfg32>();
  if (e == cudaSuccess) e = prepare_cfg<Cfg64>();
  if (e == cudaSuccess) e = prepare_cfg<Cfg96x2>();
  if (e == cudaSuccess) e = prepare_cfg<Cfg16x2>();
  if (e == cudaSuccess) e = prepare_cfg<Cfg32x2>();
  return e;
}

// Weight blocks per unit. MXFP8 weights: one block up to 128 rows (the
// 5-stage ring of two K chunks keeps more bytes in flight, which is what the
// HBM-bound row counts need), two above. MXFP4 weights: two blocks at every
// row count when H is a multiple of 256; same-box A/B, us per step:
// bs1_fp4 192.4 -> 169.8, bs4_fp4 565.7 -> 477.1, while MXFP8 lost 3-4 % at
// bs1 and bs4 with two blocks.
cudaError_t launch_experts_mma(const MmaMaps &maps, const ExpertArgs &a, int grid, int chunk_rows, cudaStream_t st) {
  const bool two = a.fp4 && a.H % 256 == 0;
  switch (chunk_rows) {
    case 16: return two ? launch_cfg<Cfg16x2>(maps, a, grid, st) : launch_cfg<Cfg16>(maps, a, grid, st);
    case 32: return two ? launch_cfg<Cfg32x2>(maps, a, grid, st) : launch_cfg<Cfg32>(maps, a, grid, st);
    case 64: return launch_cfg<Cfg64>(maps, a, grid, st);
    case 96: return launch_cfg<Cfg96x2>(maps, a, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
