// static_scratch.cu — the MoE step without any allocation: scratch lives in a
// fixed device array that is part of this library.
//
// Who needs this. Some callers cannot call cudaMalloc at the point where they
// want to run the step:
//  - a serving process whose allocator has already reserved almost all device
//    memory (for example for a KV cache) and forbids further allocations;
//  - code that must never trigger the device-wide synchronisation and latency
//    spikes cudaMalloc/cudaFree can cause;
//  - code loaded as a plugin that is only handed input and output buffers.
// moe_plan allocates its scratch once (cudaMalloc), which such callers cannot
// do. moe_forward_static_scratch runs the same kernels (route, and experts with the
// fused combine) on the fixed array below instead. It allocates nothing, and it
// calls no allocating library routine.
//
// Cost and limits:
//  - The array is MOE_STATIC_SCRATCH_BYTES (8 MiB). Every GPU that loads the
//    library holds it until the process exits.
//  - A step whose scratch does not fit is rejected with MOE_ERR_UNSUPPORTED,
//    before any device work.
//  - All calls share the one array. Calls whose work overlaps on the GPU (two
//    streams, or two host threads) race and corrupt each other's results.
//    Serialise them.
//  - Everything that must start at zero is cleared by the step's first
//    kernel: the per-tile ready counts, the work and abort words, the status
//    word and the diagnostics.
// Set-up. The first call on a device checks the device and records its SM
// count, with that device current. Every call then looks up the array's device
// address with cudaGetSymbolAddress and sets the kernels' dynamic
// shared-memory limits with cudaFuncSetAttribute: host-side calls that
// allocate nothing, repeated so that a cudaDeviceReset (which reloads the
// module) never leaves a stale address or a lost attribute behind. The first
// call on a device may load this library's device code: make it before any
// stream capture that includes a call.
// Status: with d_status NULL the step writes its status into the array,
// where no call reads it back; pass d_status to see device-side errors.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"
#include "moe.h"

namespace moe {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  bool done = false;
  int num_sms = 0;
};

DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

// Once per device, with that device current: the device check and its SM count.
moe_status_t setup_device(int dev, int *num_sms) {
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup &d = g_setup[dev];
  if (!d.done) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;
    d.num_sms = sms;
    d.done = true;
  }
  *num_sms = d.num_sms;
  return MOE_OK;
}

// Every call, with the device current: the array's device address on this
// device (host code cannot use g_static_scratch itself), and the shared-memory
// limits of the two kernels the step launches. Host-side only; allocates nothing.
moe_status_t bind_scratch(int H, int I, unsigned char **scratch) {
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) return MOE_ERR_CUDA;
  if (prepare_experts(H, I) != cudaSuccess || prepare_route() != cudaSuccess) return MOE_ERR_CUDA;
  *scratch = static_cast<unsigned char *>(ptr);
  return MOE_OK;
}

struct Layout {
  size_t ids, w, bm, cnt, slot, rows, tl, nt, ready, comb, work, status, diag, xq, xs, hq, hs, o, total;
};

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// The array starts with a control area that keeps its value between calls of
// any shape: the route kernel's phase-2 ticket, which every step leaves at
// zero (the array itself starts zeroed). The step's buffers follow it.
constexpr size_t kControlBytes = 256;

// Scratch for a T-row step (the same buffers moe_plan sizes for max_rows = T).
Layout layout_for(const moe_config_t &c, int T, int words, int n_tiles_max) {
  Layout L{};
  size_t off = kControlBytes;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += up256(bytes);
    return o;
  };
  const int64_t pairs_routed = int64_t(T) * c.top_k;
  const int64_t pairs = pairs_routed + int64_t(T) * c.num_shared;
  L.ids = take(pairs_routed * 4);
  L.w = take(pairs_routed * 4);
  L.bm = take(size_t(c.num_experts) * words * 4);
  L.cnt = take(size_t(c.num_experts + 1) * 4);
  L.slot = take(pairs_routed * 4);
  L.rows = take(size_t(c.num_experts + 1) * T * 4);
  L.tl = take(size_t(n_tiles_max) * 4);
  L.nt = take(4);
  L.ready = take(size_t(n_tiles_max) * 4);
  L.comb = take(size_t(T) * experts_down_blocks(c.hidden, c.intermediate) * 4);
  L.work = take(8);
  L.status = take(4);
  L.diag = take(64);
  L.xq = take(size_t(T) * c.hidden);
  L.xs = take(size_t(T) * (c.hidden / 32));
  L.hq = take(size_t(pairs) * c.intermediate);
  L.hs = take(size_t(pairs) * (c.intermediate / 32));
  L.o = take(size_t(pairs) * c.hidden * 4);
  L.total = off;
  return L;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_forward_static_scratch(const moe_config_t *config, const moe_weights_t *weights,
                                                   const void *x, const float *logits, int32_t T, void *y,
                                                   int32_t *d_status, void *cuda_stream) {
  if (!config || !weights) return MOE_ERR_INVALID_ARG;
  moe_config_t c = *config;
  if (T < 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  c.max_rows = T;
  const moe_status_t g = guard_host(c, *weights);
  if (g != MOE_OK) return g;
  // this entry point runs the CUDA-core GEMV kernel: its compiled MXFP8 shapes only
  if (!experts_shape_supported(c.hidden, c.intermediate) || c.weight_format != MOE_WEIGHTS_MXFP8)
    return MOE_ERR_UNSUPPORTED;
  if (!x || !logits || !y || !aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(logits) & 3u))
    return MOE_ERR_INVALID_ARG;
  if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return MOE_ERR_INVALID_ARG;
  const int words = (T + 31) / 32;
  const int64_t pairs_routed = int64_t(T) * c.top_k;
  const int64_t active_max = pairs_routed < c.num_experts ? pairs_routed : c.num_experts;
  const int n_tiles_max =
      int(pairs_routed / kTileRows + active_max + (c.num_shared ? (T + kTileRows - 1) / kTileRows : 0));
  const Layout L = layout_for(c, T, words, n_tiles_max);
  if (L.total > size_t(MOE_STATIC_SCRATCH_BYTES)) return MOE_ERR_UNSUPPORTED;  // does not fit the fixed array

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int num_sms = 0;
  const moe_status_t sg = setup_device(dev, &num_sms);
  if (sg != MOE_OK) return sg;
  unsigned char *base = nullptr;
  const moe_status_t bs = bind_scratch(c.hidden, c.intermediate, &base);
  if (bs != MOE_OK) return bs;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int32_t *status = d_status ? d_status : reinterpret_cast<int32_t *>(base + L.status);

  RouteArgs ra;
  ra.logits = logits;
  ra.x = static_cast<const uint16_t *>(x);
  ra.w_router = nullptr;  // logits are an input here
  ra.rg_cnt = nullptr;
  ra.n_eblk = 1;
  ra.T = T;
  ra.d_T = nullptr;
  ra.H = c.hidden;
  ra.E = c.num_experts;
  ra.k = c.top_k;
  ra.shared = c.num_shared;
  ra.words = words;
  ra.Tmax = T;
  ra.topk_ids = reinterpret_cast<int32_t *>(base + L.ids);
  ra.topk_w = reinterpret_cast<float *>(base + L.w);
  ra.bitmap = reinterpret_cast<uint32_t *>(base + L.bm);
  ra.counts = reinterpret_cast<int32_t *>(base + L.cnt);
  ra.slot = reinterpret_cast<int32_t *>(base + L.slot);
  ra.rows_of = reinterpret_cast<int32_t *>(base + L.rows);
  ra.tile_list = reinterpret_cast<int32_t *>(base + L.tl);
  ra.n_tiles = reinterpret_cast<int32_t *>(base + L.nt);
  ra.chunk_list = nullptr;  // this entry point always runs the CUDA-core expert kernel
  ra.n_chunks = nullptr;
  ra.chunk_rows = kChunkRowsMax;
  ra.ready = reinterpret_cast<uint32_t *>(base + L.ready);
  ra.n_tiles_max = n_tiles_max;
  ra.comb_cnt = reinterpret_cast<uint32_t *>(base + L.comb);
  ra.comb_per_row = experts_down_blocks(c.hidden, c.intermediate);
  ra.work = reinterpret_cast<uint32_t *>(base + L.work);
  ra.ticket = reinterpret_cast<uint32_t *>(base);  // control area: zero between steps
  ra.status = status;
  ra.diag = reinterpret_cast<int64_t *>(base + L.diag);
  ra.xq = base + L.xq;
  ra.xs = base + L.xs;
  if (launch_route(ra, st) != cudaSuccess) return MOE_ERR_CUDA;

  ExpertArgs ea;
  ea.w_gate = weights->w_gate;
  ea.s_gate = weights->s_gate;
  ea.w_up = weights->w_up;
  ea.s_up = weights->s_up;
  ea.w_down = weights->w_down;
  ea.s_down = weights->s_down;
  ea.sh_w_gate = weights->sh_w_gate;
  ea.sh_s_gate = weights->sh_s_gate;
  ea.sh_w_up = weights->sh_w_up;
  ea.sh_s_up = weights->sh_s_up;
  ea.sh_w_down = weights->sh_w_down;
  ea.sh_s_down = weights->sh_s_down;
  ea.T = T;
  ea.d_T = nullptr;
  ea.H = c.hidden;
  ea.I = c.intermediate;
  ea.E = c.num_experts;
  ea.k = c.top_k;
  ea.Tmax = T;
  ea.counts = ra.counts;
  ea.rows_of = ra.rows_of;
  ea.tile_list = ra.tile_list;
  ea.n_tiles = ra.n_tiles;
  ea.chunk_list = nullptr;
  ea.n_chunks = nullptr;
  ea.xq = ra.xq;
  ea.xs = ra.xs;
  ea.hq = base + L.hq;
  ea.hs = base + L.hs;
  ea.h_bf16 = nullptr;
  ea.o = reinterpret_cast<float *>(base + L.o);
  ea.ready = ra.ready;
  ea.comb_cnt = ra.comb_cnt;
  ea.topk_w = ra.topk_w;
  ea.y = static_cast<uint16_t *>(y);
  ea.shared = c.num_shared;
  ea.work = ra.work;
  ea.status = status;
  ea.diag = ra.diag;
  ea.timeout_ns = c.wait_timeout_ns > 0 ? c.wait_timeout_ns : 200000000LL;
  ea.skip_ready_tile = -1;
  ea.fp4 = 0;
  ea.swiglu_limit = c.swiglu_limit;
  ea.n_tiles_max = n_tiles_max;
  ea.pairs_cap = pairs_routed + int64_t(T) * c.num_shared;
  ea.comb_cap = int64_t(T) * experts_down_blocks(c.hidden, c.intermediate);
  if (launch_experts(ea, num_sms, st) != cudaSuccess) return MOE_ERR_CUDA;

  return MOE_OK;
}
