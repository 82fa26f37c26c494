// moe_abi.cu — the C ABI: Guard + Build (moe_plan), Runtime (moe_forward), teardown.
//
// The four-stage plugin contract follows "SGLang's Low-Latency Mode Boosts
// DeepSeek-V4.1-Flash Speed by 1.56x on AMD", "Four stages keep megakernels
// outside core": Register, Guard, Build, Runtime.
// - Guard rejects unsupported shapes and devices with MOE_ERR_UNSUPPORTED. It
//   does not fall back.
// - Build allocates every scratch buffer once for max_rows. "Beyond Day-0:
//   Optimizing DeepSeek-V4.1 Flash in SGLang" 2.1 reuses scratch buffers
//   across calls to avoid re-initialisation.
// - Runtime enqueues two kernels:
//     1. route + place + quantise x;
//     2. a persistent expert kernel (gate/up, down and the fused combine),
//        launched with Programmatic Dependent Launch: the tensor-core kernel
//        (experts_mma.cu), or the CUDA-core GEMV kernel (experts.cu) when
//        the plan was built with MOE_FLAG_PATH_GEMV.
//   It allocates nothing and does not synchronise.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <new>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"
#include "moe.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


// Pure host checks of the Guard (no device access).
moe_status_t guard_config(const moe_config_t &c) {
  if (c.hidden <= 0 || c.intermediate <= 0 || c.num_experts <= 0 || c.top_k <= 0 || c.max_rows <= 0)
    return MOE_ERR_INVALID_ARG;
  if (c.num_shared != 0 && c.num_shared != 1) return MOE_ERR_INVALID_ARG;
  if ((c.flags & MOE_FLAG_PATH_GEMV) && (c.flags & MOE_FLAG_PATH_MMA)) return MOE_ERR_INVALID_ARG;
  if (c.weight_format != MOE_WEIGHTS_MXFP8 && c.weight_format != MOE_WEIGHTS_MXFP4) return MOE_ERR_INVALID_ARG;
  if (!(c.swiglu_limit == c.swiglu_limit)) return MOE_ERR_INVALID_ARG;  // NaN
  if (c.top_k > c.num_experts) return MOE_ERR_INVALID_ARG;
  if (!experts_mma_shape_supported(c.hidden, c.intermediate)) return MOE_ERR_UNSUPPORTED;
  if (c.flags & MOE_FLAG_PATH_GEMV) {  // the CUDA-core kernel: compiled MXFP8 shapes only
    if (!experts_shape_supported(c.hidden, c.intermediate)) return MOE_ERR_UNSUPPORTED;
    if (c.weight_format != MOE_WEIGHTS_MXFP8) return MOE_ERR_UNSUPPORTED;
  }
  if (c.num_experts + c.num_shared > kRouteThreads) return MOE_ERR_UNSUPPORTED;
  if (c.top_k > 32) return MOE_ERR_UNSUPPORTED;
  if (c.max_rows > 4096) return MOE_ERR_UNSUPPORTED;
  const int words = (c.max_rows + 31) / 32;
  if (route_smem_bytes(c.num_experts, words) > kRouteSmemMax) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t guard_weights(const moe_config_t &c, const moe_weights_t &w) {
  const void *routed[6] = {w.w_gate, w.s_gate, w.w_up, w.s_up, w.w_down, w.s_down};
  const void *shared[6] = {w.sh_w_gate, w.sh_s_gate, w.sh_w_up, w.sh_s_up, w.sh_w_down, w.sh_s_down};
  for (const void *p : routed)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  for (const void *p : shared) {
    if (c.num_shared && (!p || !aligned16(p))) return MOE_ERR_INVALID_ARG;
    if (!c.num_shared && p) return MOE_ERR_INVALID_ARG;
  }
  if (c.weight_format == MOE_WEIGHTS_MXFP4) {  // packed 4-bit tensor maps want 32-byte aligned rows
    const void *codes[6] = {w.w_gate, w.w_up, w.w_down, w.sh_w_gate, w.sh_w_up, w.sh_w_down};
    for (const void *p : codes)
      if (p && (reinterpret_cast<uintptr_t>(p) & 31u)) return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

void destroy_plan(Plan *p) {
  if (!p) return;
  if (p->events_created) {
    for (int i = 0; i < kMaxTimedCalls; ++i) {
      if (p->ev_start[i]) cudaEventDestroy(p->ev_start[i]);
      if (p->ev_stop[i]) cudaEventDestroy(p->ev_stop[i]);
    }
  }
  if (p->arena) cudaFree(p->arena);
  if (p->status_host) cudaFreeHost(p->status_host);
  delete p;
}

moe_status_t copy_taps(Plan *p, const moe_taps_t *t, int T, cudaStream_t st) {
  if (!t) return MOE_OK;
  const moe_config_t &c = p->cfg;
  const int64_t P = int64_t(T) * c.top_k + int64_t(T) * c.num_shared;
  const int words = (T + 31) / 32;
  auto cp = [&](void *dst, const void *src, size_t bytes) -> bool {
    if (!dst || bytes == 0) return true;
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st) == cudaSuccess;
  };
  bool ok = true;
  ok &= cp(t->topk_ids, p->s.topk_ids, size_t(T) * c.top_k * 4);
  ok &= cp(t->topk_w, p->s.topk_w, size_t(T) * c.top_k * 4);
  ok &= cp(t->counts, p->s.counts, size_t(c.num_experts) * 4);
  ok &= cp(t->slot, p->s.slot, size_t(T) * c.top_k * 4);
  ok &= cp(t->xq, p->s.xq, size_t(T) * c.hidden);
  ok &= cp(t->xs, p->s.xs, size_t(T) * (c.hidden / 32));
  ok &= cp(t->hq, p->s.hq, size_t(P) * c.intermediate);
  ok &= cp(t->hs, p->s.hs, size_t(P) * (c.intermediate / 32));
  ok &= cp(t->h_bf16, p->s.h_bf16, size_t(P) * c.intermediate * 2);
  ok &= cp(t->o, p->s.o, size_t(P) * c.hidden * 4);
  if (t->bitmap) {
    // plan rows are ceil(max_rows/32) words wide; the tap is ceil(T/32) wide
    ok &= cudaMemcpy2DAsync(t->bitmap, size_t(words) * 4, p->s.bitmap, size_t(p->words) * 4, size_t(words) * 4,
                            c.num_experts, cudaMemcpyDeviceToDevice, st) == cudaSuccess;
  }
  return ok ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

namespace moe {
// The Guard's host-only checks, for the other entry points of the library.
moe_status_t guard_host(const moe_config_t &c, const moe_weights_t &w) {
  const moe_status_t g = guard_config(c);
  return g != MOE_OK ? g : guard_weights(c, w);
}
}  // namespace moe

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char *moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_OOM: return "MOE_ERR_OOM";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_plan(const moe_config_t *config, const moe_weights_t *weights, void *cuda_stream,
                      void **plan_out) {
  (void)cuda_stream;
  if (plan_out) *plan_out = nullptr;
  if (!config || !weights || !plan_out) return MOE_ERR_INVALID_ARG;
  const moe_config_t c = *config;
  moe_status_t g = guard_config(c);
  if (g != MOE_OK) return g;
  g = guard_weights(c, *weights);
  if (g != MOE_OK) return g;

  // ---- device part of the Guard
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;

  // ---- Build
  Plan *p = new (std::nothrow) Plan();
  if (!p) return MOE_ERR_OOM;
  memset(p, 0, sizeof(Plan));
  p->cfg = c;
  p->w = *weights;
  p->device = dev;
  p->num_sms = sms;
  p->timeout_ns = c.wait_timeout_ns > 0 ? c.wait_timeout_ns : 200000000LL;
  p->mma_min_rows = (c.flags & MOE_FLAG_PATH_GEMV) ? 0x7FFFFFFF : (c.flags & MOE_FLAG_PATH_MMA) ? 1 : kMmaMinRowsDefault;
  const int Tm = c.max_rows, E = c.num_experts, k = c.top_k, H = c.hidden, I = c.intermediate;
  p->words = (Tm + 31) / 32;
  const int64_t pairs_routed = int64_t(Tm) * k;
  p->pairs_max = pairs_routed + int64_t(Tm) * c.num_shared;
  const int64_t active_max = pairs_routed < E ? pairs_routed : E;
  p->n_tiles_max = int(pairs_routed / kTileRows + active_max + (c.num_shared ? (Tm + kTileRows - 1) / kTileRows : 0));

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  const size_t o_ids = take(pairs_routed * 4), o_w = take(pairs_routed * 4);
  const size_t o_bm = take(size_t(E) * p->words * 4), o_cnt = take(size_t(E + 1) * 4);
  const size_t o_slot = take(pairs_routed * 4), o_rows = take(size_t(E + 1) * Tm * 4);
  const size_t o_tl = take(size_t(p->n_tiles_max) * 4), o_nt = take(4);
  const size_t o_cl = take(size_t(p->n_tiles_max) * 4), o_nc = take(4);
  const size_t o_ready = take(size_t(p->n_tiles_max) * 4), o_work = take(16), o_status = take(4);
  const int down_blocks = experts_down_blocks(H, I) > H / kMmaDownRows ? experts_down_blocks(H, I) : H / kMmaDownRows;
  p->comb_per_row_max = down_blocks;
  const size_t o_comb = take(size_t(Tm) * down_blocks * 4);
  const size_t o_diag = take(8 * 8);
  const size_t o_xq = take(size_t(Tm) * H), o_xs = take(size_t(Tm) * (H / 32));
  const size_t o_hq = take(size_t(p->pairs_max) * I), o_hs = take(size_t(p->pairs_max) * (I / 32));
  const size_t o_hb = take(size_t(p->pairs_max) * I * 2), o_o = take(size_t(p->pairs_max) * H * 4);
  const size_t o_xd = take(size_t(Tm) * H * 2), o_ld = take(size_t(Tm) * E * 4), o_yd = take(size_t(Tm) * H * 2);
  const size_t o_lp = take(size_t(Tm) * E * 4), o_rg = take(size_t(p->words) * 4);
  p->arena_bytes = off;
  if (cudaMalloc(&p->arena, off) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return MOE_ERR_OOM;
  }
  unsigned char *base = static_cast<unsigned char *>(p->arena);
  Scratch &s = p->s;
  s.topk_ids = reinterpret_cast<int32_t *>(base + o_ids);
  s.topk_w = reinterpret_cast<float *>(base + o_w);
  s.bitmap = reinterpret_cast<uint32_t *>(base + o_bm);
  s.counts = reinterpret_cast<int32_t *>(base + o_cnt);
  s.slot = reinterpret_cast<int32_t *>(base + o_slot);
  s.rows_of = reinterpret_cast<int32_t *>(base + o_rows);
  s.tile_list = reinterpret_cast<int32_t *>(base + o_tl);
  s.n_tiles = reinterpret_cast<int32_t *>(base + o_nt);
  s.chunk_list = reinterpret_cast<int32_t *>(base + o_cl);
  s.n_chunks = reinterpret_cast<int32_t *>(base + o_nc);
  s.ready = reinterpret_cast<uint32_t *>(base + o_ready);
  s.comb_cnt = reinterpret_cast<uint32_t *>(base + o_comb);
  s.work = reinterpret_cast<uint32_t *>(base + o_work);
  s.status = reinterpret_cast<int32_t *>(base + o_status);
  s.diag = reinterpret_cast<int64_t *>(base + o_diag);
  s.xq = base + o_xq;
  s.xs = base + o_xs;
  s.hq = base + o_hq;
  s.hs = base + o_hs;
  s.h_bf16 = reinterpret_cast<uint16_t *>(base + o_hb);
  s.o = reinterpret_cast<float *>(base + o_o);
  s.x_dev = base + o_xd;
  s.logits_dev = reinterpret_cast<float *>(base + o_ld);
  s.y_dev = base + o_yd;
  s.logits_proj = reinterpret_cast<float *>(base + o_lp);
  s.rg_cnt = reinterpret_cast<uint32_t *>(base + o_rg);
  if (cudaMemset(p->arena, 0, off) != cudaSuccess) {
    destroy_plan(p);
    return MOE_ERR_CUDA;
  }
  if (prepare_route() != cudaSuccess ||
      (experts_shape_supported(H, I) && prepare_experts(H, I) != cudaSuccess) || prepare_experts_mma() != cudaSuccess ||
      prepare_residual_norm(H) != cudaSuccess) {
    destroy_plan(p);
    return MOE_ERR_CUDA;
  }
  if (!encode_mma_maps(c, *weights, &p->maps)) {
    destroy_plan(p);
    return MOE_ERR_CUDA;
  }
  if (cudaHostAlloc(reinterpret_cast<void **>(&p->status_host), 4, cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    p->status_host = nullptr;
    destroy_plan(p);
    return MOE_ERR_OOM;
  }
  if (cudaHostGetDevicePointer(reinterpret_cast<void **>(&p->status_mapped), p->status_host, 0) != cudaSuccess) {
    destroy_plan(p);
    return MOE_ERR_CUDA;
  }
  if (c.flags & MOE_FLAG_TIMING) {
    for (int i = 0; i < kMaxTimedCalls; ++i) {
      if (cudaEventCreate(&p->ev_start[i]) != cudaSuccess || cudaEventCreate(&p->ev_stop[i]) != cudaSuccess) {
        p->events_created = true;
        destroy_plan(p);
        return MOE_ERR_CUDA;
      }
    }
    p->events_created = true;
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    destroy_plan(p);
    return MOE_ERR_CUDA;
  }
  *plan_out = p;
  return MOE_OK;
}

}  // extern "C"

namespace {

// A named NVTX range over one entry-point call (no cost unless a profiler is
// attached): profilers can pick out each step's launches by it.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

// Enqueues one step: the route kernel, then an expert kernel with PDL.
// T sizes the grids. With d_T set, the kernels read the step's row count
// from device memory (clamped to max_rows) and the tensor-core kernel runs.
// io (or NULL): the fused router projection and residual-stream epilogue;
// with io set, logits is ignored and the tensor-core kernel runs.
moe_status_t enqueue_step(Plan *p, const void *x, const float *logits, int32_t T, const int32_t *d_T, void *y,
                          bool h_tap, int32_t *d_status, cudaStream_t st, const moe_fused_io_t *io = nullptr) {
  const moe_config_t &c = p->cfg;
  Scratch &s = p->s;
  int32_t *status = d_status ? d_status : s.status;
  const bool mma = d_T != nullptr || io != nullptr || T >= p->mma_min_rows;
  const bool proj = io && io->w_router;
  const int n_streams = io ? io->num_streams : 0;

  RouteArgs ra;
  ra.logits = proj ? (io->logits ? io->logits : s.logits_proj) : (io ? io->logits : logits);
  ra.x = static_cast<const uint16_t *>(x);
  ra.w_router = proj ? static_cast<const uint16_t *>(io->w_router) : nullptr;
  ra.rg_cnt = s.rg_cnt;
  ra.n_eblk = (c.num_experts + kRouterExperts - 1) / kRouterExperts;
  ra.T = T;
  ra.d_T = d_T;
  ra.H = c.hidden;
  ra.E = c.num_experts;
  ra.k = c.top_k;
  ra.shared = c.num_shared;
  ra.words = p->words;
  ra.Tmax = c.max_rows;
  ra.topk_ids = s.topk_ids;
  ra.topk_w = s.topk_w;
  ra.bitmap = s.bitmap;
  ra.counts = s.counts;
  ra.slot = s.slot;
  ra.rows_of = s.rows_of;
  ra.tile_list = s.tile_list;
  ra.n_tiles = s.n_tiles;
  ra.chunk_list = mma ? s.chunk_list : nullptr;
  ra.n_chunks = s.n_chunks;
  ra.chunk_rows = mma_chunk_rows(T, c.hidden);
  ra.ready = s.ready;
  ra.n_tiles_max = p->n_tiles_max;
  ra.comb_cnt = s.comb_cnt;
  ra.comb_per_row = mma ? c.hidden / kMmaDownRows : experts_down_blocks(c.hidden, c.intermediate);
  ra.work = s.work;
  ra.ticket = s.work + 2;
  ra.status = status;
  ra.diag = s.diag;
  ra.xq = s.xq;
  ra.xs = s.xs;
  if (launch_route(ra, st) != cudaSuccess) return MOE_ERR_CUDA;

  ExpertArgs ea;
  ea.w_gate = p->w.w_gate;
  ea.s_gate = p->w.s_gate;
  ea.w_up = p->w.w_up;
  ea.s_up = p->w.s_up;
  ea.w_down = p->w.w_down;
  ea.s_down = p->w.s_down;
  ea.sh_w_gate = p->w.sh_w_gate;
  ea.sh_s_gate = p->w.sh_s_gate;
  ea.sh_w_up = p->w.sh_w_up;
  ea.sh_s_up = p->w.sh_s_up;
  ea.sh_w_down = p->w.sh_w_down;
  ea.sh_s_down = p->w.sh_s_down;
  ea.T = T;
  ea.d_T = d_T;
  ea.H = c.hidden;
  ea.I = c.intermediate;
  ea.E = c.num_experts;
  ea.k = c.top_k;
  ea.Tmax = c.max_rows;
  ea.counts = s.counts;
  ea.rows_of = s.rows_of;
  ea.tile_list = s.tile_list;
  ea.n_tiles = s.n_tiles;
  ea.chunk_list = s.chunk_list;
  ea.n_chunks = s.n_chunks;
  ea.xq = s.xq;
  ea.xs = s.xs;
  ea.hq = s.hq;
  ea.hs = s.hs;
  ea.h_bf16 = h_tap ? s.h_bf16 : nullptr;
  ea.o = s.o;
  ea.ready = s.ready;
  ea.comb_cnt = s.comb_cnt;
  ea.topk_w = s.topk_w;
  ea.y = static_cast<uint16_t *>(y);
  ea.shared = c.num_shared;
  ea.work = s.work;
  ea.status = status;
  ea.diag = s.diag;
  ea.timeout_ns = p->timeout_ns;
  ea.skip_ready_tile = (c.flags & MOE_FLAG_TEST_SKIP_READY) ? 0 : -1;
  ea.fp4 = c.weight_format == MOE_WEIGHTS_MXFP4 ? 1 : 0;
  ea.swiglu_limit = c.swiglu_limit;
  ea.n_tiles_max = p->n_tiles_max;
  ea.pairs_cap = p->pairs_max;
  ea.comb_cap = int64_t(c.max_rows) * p->comb_per_row_max;
  // test hook of the bounds-checked build: the checks see half of the combine
  // counters this step uses, so one trips at an index still inside the buffer
  if (c.flags & MOE_FLAG_TEST_BOUNDS) ea.comb_cap = int64_t(T) * ra.comb_per_row / 2;
  const bool timed = (c.flags & MOE_FLAG_TIMING) && p->timed_calls < kMaxTimedCalls;
  if (timed && cudaEventRecord(p->ev_start[p->timed_calls], st) != cudaSuccess) return MOE_ERR_CUDA;
  const cudaError_t le = mma ? launch_experts_mma(p->maps, ea, p->num_sms, ra.chunk_rows, st) : launch_experts(ea, p->num_sms, st);
  if (le != cudaSuccess) return MOE_ERR_CUDA;
  if (timed) {
    if (cudaEventRecord(p->ev_stop[p->timed_calls], st) != cudaSuccess) return MOE_ERR_CUDA;
    ++p->timed_calls;
  }
  if (n_streams) {  // the epilogue: one block per row, launched to overlap the expert kernel's end
    ResidArgs na;
    na.y = static_cast<const uint16_t *>(y);
    na.resid_in = static_cast<const uint16_t *>(io->resid_in);
    na.resid_out = static_cast<uint16_t *>(io->resid_out);
    na.mix_res = io->mix_res;
    na.mix_post = io->mix_post;
    na.mix_pre = io->mix_pre;
    na.norm_w = static_cast<const uint16_t *>(io->norm_weight);
    na.rms_eps = io->rms_eps;
    na.zq = io->zq;
    na.zs = io->zs;
    na.z_bf16 = static_cast<uint16_t *>(io->z);
    na.T = T;
    na.H = c.hidden;
    na.S = n_streams;
    if (launch_residual_norm(na, st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_forward(void *plan, const void *x, const float *logits, int32_t T, void *y,
                         const moe_taps_t *taps, int32_t *d_status, void *cuda_stream) {
  const NvtxRange nvtx_range("moe_forward");
  Plan *p = static_cast<Plan *>(plan);
  if (!p) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > p->cfg.max_rows) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !logits || !y || !aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(logits) & 3u))
    return MOE_ERR_INVALID_ARG;
  if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(p->device);
  if (!dg.ok) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const moe_status_t r = enqueue_step(p, x, logits, T, nullptr, y, taps && taps->h_bf16, d_status, st);
  if (r != MOE_OK) return r;
  return copy_taps(p, taps, T, st);
}

moe_status_t moe_forward_dev(void *plan, const void *x, const float *logits, const int32_t *d_T, void *y,
                             int32_t *d_status, void *cuda_stream) {
  const NvtxRange nvtx_range("moe_forward_dev");
  Plan *p = static_cast<Plan *>(plan);
  if (!p || !d_T || (reinterpret_cast<uintptr_t>(d_T) & 3u)) return MOE_ERR_INVALID_ARG;
  if (p->cfg.flags & MOE_FLAG_PATH_GEMV) return MOE_ERR_UNSUPPORTED;
  if (!x || !logits || !y || !aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(logits) & 3u))
    return MOE_ERR_INVALID_ARG;
  if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(p->device);
  if (!dg.ok) return MOE_ERR_CUDA;
  return enqueue_step(p, x, logits, p->cfg.max_rows, d_T, y, false, d_status, static_cast<cudaStream_t>(cuda_stream));
}

moe_status_t moe_forward_fused(void *plan, const void *x, int32_t T, const moe_fused_io_t *io, void *y,
                               const moe_taps_t *taps, int32_t *d_status, void *cuda_stream) {
  const NvtxRange nvtx_range("moe_forward_fused");
  Plan *p = static_cast<Plan *>(plan);
  if (!p || !io) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > p->cfg.max_rows) return MOE_ERR_INVALID_ARG;
  if (p->cfg.flags & MOE_FLAG_PATH_GEMV) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  const auto a4 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 3u) == 0; };
  if (!x || !y || !aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  if (io->w_router) {
    if (!aligned16(io->w_router) || (io->logits && !a4(io->logits))) return MOE_ERR_INVALID_ARG;
  } else if (!io->logits || !a4(io->logits)) {
    return MOE_ERR_INVALID_ARG;
  }
  const int S = io->num_streams;
  if (S < 0 || S > kMaxStreams) return MOE_ERR_INVALID_ARG;
  if (S > 0) {
    if (!io->resid_in || !io->resid_out || !io->norm_weight || !io->zq || !io->zs) return MOE_ERR_INVALID_ARG;
    if (!aligned16(io->resid_in) || !aligned16(io->resid_out) || !aligned16(io->norm_weight) || !aligned16(io->zq) ||
        (io->z && !aligned16(io->z)))
      return MOE_ERR_INVALID_ARG;
    if (!a4(io->mix_res) || !a4(io->mix_post) || !a4(io->mix_pre)) return MOE_ERR_INVALID_ARG;
    if (!(io->rms_eps >= 0.0f) || io->rms_eps > 3.4e38f) return MOE_ERR_INVALID_ARG;  // NaN, negative or infinite
  }
  if (d_status && !a4(d_status)) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(p->device);
  if (!dg.ok) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const moe_status_t r = enqueue_step(p, x, nullptr, T, nullptr, y, taps && taps->h_bf16, d_status, st, io);
  if (r != MOE_OK) return r;
  return copy_taps(p, taps, T, st);
}

moe_status_t moe_forward_host(void *plan, const void *x_host, const float *logits_host, int32_t T, void *y_host,
                              void *cuda_stream) {
  const NvtxRange nvtx_range("moe_forward_host");
  Plan *p = static_cast<Plan *>(plan);
  if (!p) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > p->cfg.max_rows) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x_host || !logits_host || !y_host) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(p->device);
  if (!dg.ok) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const moe_config_t &c = p->cfg;
  const size_t xb = size_t(T) * c.hidden * 2, lb = size_t(T) * c.num_experts * 4;
  // Pinned (page-locked, mapped) host memory is in the device's address
  // space: the kernels read x and the logits and write y there directly, over
  // the host link, with no copy operation. Other host memory goes through
  // plan-owned device buffers.
  const auto mapped = [](const void *h) -> const void * {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
  };
  const void *x_dev = mapped(x_host);
  const void *l_dev = mapped(logits_host);
  void *y_dev = const_cast<void *>(mapped(y_host));
  if (!x_dev || !aligned16(x_dev)) {
    if (cudaMemcpyAsync(p->s.x_dev, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess) return MOE_ERR_CUDA;
    x_dev = p->s.x_dev;
  }
  if (!l_dev || !aligned16(l_dev)) {
    if (cudaMemcpyAsync(p->s.logits_dev, logits_host, lb, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    l_dev = p->s.logits_dev;
  }
  const bool y_staged = !y_dev || !aligned16(y_dev);
  if (y_staged) y_dev = p->s.y_dev;
  // The step's status goes straight to the plan's pinned word (the route
  // kernel sets it at the start of the step; errors replace it).
  *reinterpret_cast<volatile int32_t *>(p->status_host) = MOE_ERR_CUDA;
  moe_status_t r = moe_forward(plan, x_dev, static_cast<const float *>(l_dev), T, y_dev, nullptr, p->status_mapped,
                               cuda_stream);
  if (r != MOE_OK) return r;
  if (y_staged && cudaMemcpyAsync(y_host, p->s.y_dev, xb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status_t>(*reinterpret_cast<volatile int32_t *>(p->status_host));
}

moe_status_t moe_quantize_mxfp8(const void *x, int64_t rows, int32_t cols, uint8_t *q, uint8_t *s, void *cuda_stream) {
  if (rows < 0 || cols <= 0 || cols % 32) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !s || !aligned16(x) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (launch_quantize(static_cast<const uint16_t *>(x), rows, cols, q, s, static_cast<cudaStream_t>(cuda_stream)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_quantize_mxfp4(const void *x, int64_t rows, int32_t cols, uint8_t *q, uint8_t *s, void *cuda_stream) {
  if (rows < 0 || cols <= 0 || cols % 32) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !s || !aligned16(x) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  if (launch_quantize_fp4(static_cast<const uint16_t *>(x), rows, cols, q, s,
                          static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_kernel_times(void *plan, double *expert_ms_out, int32_t *launches_out) {
  Plan *p = static_cast<Plan *>(plan);
  if (!p || !expert_ms_out || !launches_out) return MOE_ERR_INVALID_ARG;
  if (!(p->cfg.flags & MOE_FLAG_TIMING)) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(p->device);
  double total = 0.0;
  for (int i = 0; i < p->timed_calls; ++i) {
    if (cudaEventSynchronize(p->ev_stop[i]) != cudaSuccess) return MOE_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p->ev_start[i], p->ev_stop[i]) != cudaSuccess) return MOE_ERR_CUDA;
    total += ms;
  }
  *expert_ms_out = total;
  *launches_out = p->timed_calls;
  p->timed_calls = 0;
  return MOE_OK;
}

moe_status_t moe_plan_status(void *plan, int32_t *status_out) {
  Plan *p = static_cast<Plan *>(plan);
  if (!p || !status_out) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(p->device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, p->s.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  *status_out = v;
  return MOE_OK;
}

moe_status_t moe_plan_diagnostics(void *plan, int64_t *out8) {
  Plan *p = static_cast<Plan *>(plan);
  if (!p || !out8) return MOE_ERR_INVALID_ARG;
  DeviceGuard dg(p->device);
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(out8, p->s.diag, 8 * sizeof(int64_t), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_destroy(void *plan) {
  Plan *p = static_cast<Plan *>(plan);
  if (!p) return MOE_OK;
  DeviceGuard dg(p->device);
  const bool ok = cudaDeviceSynchronize() == cudaSuccess;
  destroy_plan(p);
  return ok ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
