// libmoe_mxfp4.so — C ABI entry points (declared in include/moe_mxfp4.h).
//
// One translation unit: the kernels live in the headers included below.  The
// host code validates arguments before any CUDA call, lays out the per-call
// scratch, and enqueues the steps of the layer on the caller's stream:
//   route_topk -> route_permute -> act quant/gather -> GEMM1 -> GEMM2 -> combine
// (for T <= 32 the first three are one kernel; GEMM1 and GEMM2 are one
// cooperative launch on layers with a handful of work items per SM).  MXFP8
// mode runs the GEMMs on tcgen05 block-scaled MMA fed by TMA; bf16 mode
// decodes the weights to bf16 in tensor memory and runs tcgen05 kind::f16.
// Beside the layer: the router GEMM, a dense MXFP8 projection, the
// verification of a drafted block, and a chain of layers in one call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>
#include <utility>

#include "combine.cuh"
#include "common.cuh"
#include "dense_tc.cuh"
#include "fmt.cuh"
#include "gemm_bf16.cuh"
#include "gemm_tc.cuh"
#include "pad.cuh"
#include "quant.cuh"
#include "route.cuh"
#include "route_small.cuh"
#include "verify.cuh"

namespace moe {

__device__ int g_status;  // first device-side error since the last get_status

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int* status = nullptr;
  void* ws = nullptr;  // library-owned scratch cache
  size_t ws_bytes = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_allocs{0};  // device allocations of the scratch cache

// records the step markers of moe_opts around the kernels of one call
struct Steps {
  const moe_opts* o;
  cudaStream_t s;
  int i = 0;
  void mark() {
    if (o && o->step_events && i < o->n_step_events) cudaEventRecord(o->step_events[i], s);
    ++i;
  }
  void launched(int n = 1) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <int kN>
bool set_bf16_smem() {
  const int bytes = (int)BfCfg<kN>::kSmem;
  return cudaFuncSetAttribute(gemm_bf16_kernel<kN, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
         cudaFuncSetAttribute(gemm_bf16_kernel<kN, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess;
}

// Token-chunk width (slots per GEMM work item): narrow chunks keep the weight
// pipeline deepest; from kWideMinTokens tokens on, experts get many tokens and
// wide chunks cut the MMA instructions per token (MXFP8 mode) or the decodes
// of each expert's weights (bf16 mode).
int chunk_for(int act, int T) {
  if (T < kWideMinTokens) return kChunkNarrow;
  return act == MOE_ACT_MXFP8 ? kChunkWide : kChunkBf16Wide;
}

// the fused small-block routing kernel's largest shared memory (T = 32,
// E = MOE_MAX_E, k = MOE_MAX_K), for every instantiation
static_assert(kSmallRouteTokens * MOE_MAX_K <= 1024,
              "the small-block routing ranks one assignment per thread");
bool set_small_route_smem() {
  const int tk = kSmallRouteTokens * MOE_MAX_K;
  const int bytes = (int)small_route_smem(kSmallRouteTokens, MOE_MAX_E, MOE_MAX_K,
                                          std::min(MOE_MAX_E, tk) + tk / kChunkNarrow + 1)
                        .total;
  bool ok = true;
  auto set = [&](auto kernel) {
    ok = ok && cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    bytes) == cudaSuccess;
  };
  set(route_act_small_kernel<4, true>);
  set(route_act_small_kernel<12, true>);
  set(route_act_small_kernel<32, true>);
  set(route_act_small_kernel<4, false>);
  set(route_act_small_kernel<12, false>);
  set(route_act_small_kernel<32, false>);
  set(route_act_small_layers_kernel<4, true>);
  set(route_act_small_layers_kernel<12, true>);
  set(route_act_small_layers_kernel<32, true>);
  set(route_act_small_layers_kernel<4, false>);
  set(route_act_small_layers_kernel<12, false>);
  set(route_act_small_layers_kernel<32, false>);
  return ok;
}

template <int kN>
bool set_gemm_smem() {
  const int bytes = (int)TcCfg<kN>::kSmem;
  static_assert(tc_smem_bytes<kN, kModeLayer>() <= 232448, "shared memory of the layer launch");
  return cudaFuncSetAttribute(gemm_tc_kernel<kN, kModeGemm1>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
         cudaFuncSetAttribute(gemm_tc_kernel<kN, kModeGemm2>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
         cudaFuncSetAttribute(gemm_tc_kernel<kN, kModeBoth>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
         cudaFuncSetAttribute(gemm_tc_kernel<kN, kModeLayer>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)tc_smem_bytes<kN, kModeLayer>()) == cudaSuccess &&
         cudaFuncSetAttribute(gemm_chain_kernel<kN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)tc_smem_bytes<kN, kModeLayer>()) == cudaSuccess;
}

// Launches `kernel` (a persistent kernel whose CTAs wait on one another) as a
// cooperative launch of one CTA per SM: every CTA is resident at once or the
// launch fails without running (cudaErrorCooperativeLaunchTooLarge).  Also
// programmatic when the driver accepts both attributes and it is not the
// call's first kernel.
template <typename P>
cudaError_t launch_cooperative(void (*kernel)(P), int grid, size_t smem, cudaStream_t stream,
                               const P& prm, bool first) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = first ? 1 : 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, prm);
  if (e == cudaSuccess || e == cudaErrorCooperativeLaunchTooLarge || first) return e;
  (void)cudaGetLastError();  // the combination was refused: cooperative only
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, prm);
}

// Launches `kernel` with programmatic stream serialization: it may be
// scheduled while the previous kernel in the stream still runs and orders
// itself with grid_dependency_wait() (every kernel launched this way calls it
// before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Returns the launch's error (cudaSuccess when enqueued).  `first`: the
// call's first kernel (an ordinary launch, never overlapping earlier work).
template <int kN>
cudaError_t launch_gemm(int mode, int grid, cudaStream_t stream, const TcParams& prm,
                        bool first = false) {
  const size_t smem = TcCfg<kN>::kSmem;
  if (mode == kModeGemm1)
    return launch_pdl(gemm_tc_kernel<kN, kModeGemm1>, dim3(grid), dim3(kTcThreads), smem, stream,
                      prm);
  if (mode == kModeGemm2)
    return launch_pdl(gemm_tc_kernel<kN, kModeGemm2>, dim3(grid), dim3(kTcThreads), smem, stream,
                      prm);
  // Both GEMMs (and, for the whole-layer mode, the combine and maybe the
  // routing) in one launch: CTAs wait for other CTAs' work, so every CTA must
  // be resident at once (a cooperative launch).  When programmatic, CTAs that
  // start early block in grid_dependency_wait() before any cross-CTA wait,
  // and the preceding kernel never waits on them.
  if (mode == kModeLayer)
    return launch_cooperative(gemm_tc_kernel<kN, kModeLayer>, grid,
                              tc_smem_bytes<kN, kModeLayer>(), stream, prm, first);
  return launch_cooperative(gemm_tc_kernel<kN, kModeBoth>, grid, smem, stream, prm, first);
}

constexpr int kRouterNMax = 128;                        // router tokens per work item
// projection tokens per work item: up to 32 tokens a small B tile, so that
// more stages of weights are in flight (11 against 7: T = 8 20.8 -> 18 us);
// above, 128 (256-token items, one wave at T = 256, were slower: 35 -> 37 us)
constexpr int kDenseNSmall = 32, kDenseNMax = 128;
int dense_n_for(int T) { return T <= kDenseNSmall ? kDenseNSmall : kDenseNMax; }
constexpr int64_t kRouterPartBytes = 24ll << 20;       // cap on router split partials
constexpr int64_t kDensePartBytes = 64ll << 20;        // cap on projection split partials

// Work decomposition of a dense split-K GEMM: 128-row weight tiles x token
// blocks x K splits.  The split count minimises a simple time model (µs):
// waves of work items x (K blocks per item x a stage's bytes at the ~45 GB/s an
// SM ingests by TMA + 2 of fixed cost per item), plus the fp32 partials
// written and read back at about 5 TB/s; under a cap on the partials' bytes,
// and only splits that leave no item empty.
struct DensePlan {
  int m_tiles, n_blocks, k_splits, kb_per_split, kb_total;
};

DensePlan plan_dense(int64_t M, int64_t T, int kb_total, int n_max, int sms, int64_t cap) {
  DensePlan P{};
  P.m_tiles = (int)((M + 127) / 128);
  P.n_blocks = (int)((T + n_max - 1) / n_max);
  P.kb_total = kb_total;
  const int64_t base = (int64_t)P.m_tiles * P.n_blocks;
  const int64_t split_bytes = T * M * 4;
  const int64_t rows_b = (std::min<int64_t>(T, n_max) + 15) & ~int64_t(15);
  const double stage_us = (double)(128 * 128 + rows_b * 128) / 45.0e3;
  int best = 1;
  double best_t = -1.0;
  for (int ks = 1; ks <= std::min(kb_total, kDenseMaxSplits); ++ks) {
    if (ks > 1 && split_bytes * ks > cap) break;
    const int per = (kb_total + ks - 1) / ks;
    if ((kb_total + per - 1) / per != ks) continue;
    const int64_t items = base * ks;
    const double t = (double)((items + sms - 1) / sms) * (stage_us * per + 2.0) +
                     (ks > 1 ? 2.0 * (double)(split_bytes * ks) / 5.0e6 : 0.0);
    if (best_t < 0.0 || t < best_t) {
      best_t = t;
      best = ks;
    }
  }
  P.kb_per_split = (kb_total + best - 1) / best;
  P.k_splits = (kb_total + P.kb_per_split - 1) / P.kb_per_split;
  return P;
}

// bytes of router partials a layer of this shape may need (any device)
int64_t router_part_bytes(int64_t T, int64_t E) {
  return std::max<int64_t>(T * E * 4, std::min<int64_t>(kRouterPartBytes,
                                                         (int64_t)kDenseMaxSplits * T * E * 4));
}

// token rows per activation TMA box: no wider than the token count needs
int box_rows_for(int64_t T) { return T <= 16 ? 16 : T <= 32 ? 32 : kDenseBoxRowsB; }

// current device; checks compute capability 10.3 and caches per-device data
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_NO_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return MOE_ERR_NO_DEVICE;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status) != cudaSuccess)
      return MOE_ERR_CUDA;
    const int permute_smem = (35 * MOE_MAX_E + 35) * (int)sizeof(int);
    if (cudaFuncSetAttribute(route_permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             permute_smem) != cudaSuccess ||
        cudaFuncSetAttribute(route_permute_layers_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             permute_smem) != cudaSuccess ||
        !set_small_route_smem() ||
        !set_gemm_smem<kChunkNarrow>() || !set_gemm_smem<kChunkWide>() ||
        cudaFuncSetAttribute(dense_tc_kernel<kDenseBf16, kRouterNMax>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)DenseCfg<kDenseBf16, kRouterNMax>::kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(dense_tc_kernel<kDenseMxf8, kDenseNSmall>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)DenseCfg<kDenseMxf8, kDenseNSmall>::kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(dense_tc_kernel<kDenseMxf8, kDenseNMax>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)DenseCfg<kDenseMxf8, kDenseNMax>::kSmem) != cudaSuccess ||
        !set_bf16_smem<kChunkNarrow>() || !set_bf16_smem<kChunkBf16Wide>())
      return MOE_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  return MOE_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2D row-major map: `inner` elements per row, `rows` rows, `stride` bytes
// between rows, box of box_inner x box_rows, 128-byte swizzle
int make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
             uint64_t rows, uint64_t stride, uint32_t box_inner, uint32_t box_rows,
             CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
             CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
  auto enc = tensor_map_encoder();
  if (!enc) return MOE_ERR_CUDA;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {stride};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

struct Layout {
  size_t topk_idx, topk_w, cnt, off, perm, pos, chunks, done, meta, xq, xs, hq, hs, yp, part,
      rlogits, sync, total;
  int max_chunks;
};

// routed: the layer computes its router logits (split-K partials in `part`)
Layout layout_for(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int act_mode,
                  bool routed = false) {
  Layout L{};
  const int64_t TK = T * k;
  const int64_t act_bytes = act_mode == MOE_ACT_BF16 ? 2 : 1;
  L.max_chunks = (int)(std::min<int64_t>(E, TK) + TK / kChunkNarrow + 1);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.topk_idx = take(TK * 4);
  L.topk_w = take(TK * 4);
  L.cnt = take(E * 4);
  L.off = take((E + 1) * 4);
  L.perm = take(TK * 4);
  L.pos = take(TK * 4);
  L.chunks = take((size_t)L.max_chunks * 16);
  L.done = take((size_t)L.max_chunks * 4);
  L.meta = take(64 * 4);
  L.xq = take(TK * H * act_bytes);
  L.xs = take(TK * (H / 32));
  L.hq = take(TK * I * act_bytes);
  L.hs = take(TK * (I / 32));
  L.yp = take(TK * H * 4);
  L.part = take(routed ? (size_t)router_part_bytes(T, E) : 0);
  L.rlogits = take(routed ? (size_t)(T * E * 4) : 0);
  // the whole-layer launch's barrier words and its flags per (chunk, GEMM1
  // tile pair, epilogue warp)
  L.sync = take(kGridSyncBytes + (size_t)L.max_chunks * (I / 128) * 4 * 8);
  L.total = o;
  return L;
}

Work carve(void* base, const Layout& L) {
  uint8_t* b = static_cast<uint8_t*>(base);
  Work w;
  w.topk_idx = reinterpret_cast<int32_t*>(b + L.topk_idx);
  w.topk_w = reinterpret_cast<float*>(b + L.topk_w);
  w.cnt = reinterpret_cast<int32_t*>(b + L.cnt);
  w.off = reinterpret_cast<int32_t*>(b + L.off);
  w.perm = reinterpret_cast<int32_t*>(b + L.perm);
  w.pos = reinterpret_cast<int32_t*>(b + L.pos);
  w.chunks = reinterpret_cast<int4*>(b + L.chunks);
  w.done = reinterpret_cast<int32_t*>(b + L.done);
  w.meta = reinterpret_cast<int32_t*>(b + L.meta);
  w.xq = b + L.xq;
  w.xs = b + L.xs;
  w.hq = b + L.hq;
  w.hs = b + L.hs;
  w.yp = reinterpret_cast<float*>(b + L.yp);
  w.part = reinterpret_cast<float*>(b + L.part);
  w.rlogits = reinterpret_cast<float*>(b + L.rlogits);
  w.sync = b + L.sync;
  w.max_chunks = L.max_chunks;
  return w;
}

// K steps of the next layer's first GEMM1 item each CTA prefetches into L2
// (2 x 8 KB of packed weights per step; 148 CTAs x 8 steps ~ 19 MB)
constexpr int kChainPrefetchStages = 8;

// A chain of n layers: n routing blocks one stride apart (a routing block is
// the first regions of a layer's layout, topk_idx .. meta), then the rest of
// one layer's layout (the activation buffers the layers share in turn), then
// two bf16 [T, H] buffers that carry the residual stream between layers.
struct ChainLayout {
  Layout base;
  size_t route_block, act_shift, xb[2], total;
};

ChainLayout chain_layout(int64_t n, int64_t T, int64_t H, int64_t I, int64_t E, int64_t k,
                         int act_mode) {
  ChainLayout C{};
  C.base = layout_for(T, H, I, E, k, act_mode);
  C.route_block = C.base.xq;
  C.act_shift = (size_t)(n - 1) * C.route_block;  // the base layout follows the last block
  const size_t x_bytes = align256((size_t)(T * H * 2));
  C.xb[0] = C.act_shift + C.base.total;
  C.xb[1] = C.xb[0] + x_bytes;
  C.total = C.xb[1] + x_bytes;
  return C;
}

// layer l's view of a chain workspace: its own routing block, the shared rest
Work carve_chain(void* base, const ChainLayout& C, int l) {
  uint8_t* b = static_cast<uint8_t*>(base);
  Work w = carve(b + C.act_shift, C.base);
  uint8_t* r = b + (size_t)l * C.route_block;
  const Layout& L = C.base;
  w.topk_idx = reinterpret_cast<int32_t*>(r + L.topk_idx);
  w.topk_w = reinterpret_cast<float*>(r + L.topk_w);
  w.cnt = reinterpret_cast<int32_t*>(r + L.cnt);
  w.off = reinterpret_cast<int32_t*>(r + L.off);
  w.perm = reinterpret_cast<int32_t*>(r + L.perm);
  w.pos = reinterpret_cast<int32_t*>(r + L.pos);
  w.chunks = reinterpret_cast<int4*>(r + L.chunks);
  w.done = reinterpret_cast<int32_t*>(r + L.done);
  w.meta = reinterpret_cast<int32_t*>(r + L.meta);
  return w;
}

// the public form of a layout: routing arrays `route_shift` bytes and the
// activation buffers `act_shift` bytes after the layout's own offsets
moe_workspace_layout public_layout(const Layout& L, size_t route_shift, size_t act_shift) {
  moe_workspace_layout o{};
  o.topk_idx = route_shift + L.topk_idx;
  o.topk_w = route_shift + L.topk_w;
  o.cnt = route_shift + L.cnt;
  o.off = route_shift + L.off;
  o.perm = route_shift + L.perm;
  o.pos = route_shift + L.pos;
  o.xq = act_shift + L.xq;
  o.xs = act_shift + L.xs;
  o.hq = act_shift + L.hq;
  o.hs = act_shift + L.hs;
  o.yp = act_shift + L.yp;
  o.logits = L.rlogits < L.sync ? act_shift + L.rlogits : SIZE_MAX;  // routed layouts only
  o.x_stream[0] = o.x_stream[1] = SIZE_MAX;
  return o;
}

// library-owned scratch of at least `bytes` on this device
int cached_workspace(DeviceState* d, size_t bytes, void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (d->ws_bytes < bytes) {
    if (d->ws) cudaFree(d->ws);  // synchronizes: no call still uses it
    d->ws = nullptr;
    d->ws_bytes = 0;
    if (cudaMalloc(&d->ws, bytes) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_NO_MEMORY;
    }
    g_allocs.fetch_add(1, std::memory_order_relaxed);
    d->ws_bytes = bytes;
  }
  *out = d->ws;
  return MOE_OK;
}

int validate_shape(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
  if (k > E) return MOE_ERR_INVALID_ARG;
  if (k > MOE_MAX_K || E > MOE_MAX_E) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (H % 32 || I % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (T * k > (int64_t)1 << 30 || T * k * H > ((int64_t)1 << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

int launch_status() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// widths the GEMM kernels take directly (their FP4 weight rows are TMA-loaded
// 128 elements at a time); other multiples of 32 run on zero-padded copies
bool tc_widths(int64_t H, int64_t I) { return H % 128 == 0 && I % 128 == 0; }

int64_t round128(int64_t v) { return (v + 127) / 128 * 128; }

// A layer run on zero-padded copies (H or I rounded up to a multiple of 128,
// or FP4 weights only 16-byte aligned): the padded layer's own scratch first
// (so its routing arrays and activation buffers sit where the layout of the
// padded shape puts them), then the copies of the weights, x, y and the router
// weights (routed layers).
struct PadLayout {
  int64_t Hp, Ip;
  Layout inner;
  size_t w13, w13s, w2, w2s, x, y, wr, total;
};

PadLayout pad_layout(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int act,
                     bool routed) {
  PadLayout P{};
  P.Hp = round128(H);
  P.Ip = round128(I);
  P.inner = layout_for(T, P.Hp, P.Ip, E, k, act, routed);
  size_t o = P.inner.total;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  P.w13 = take((size_t)(E * 2 * P.Ip * P.Hp / 2));
  P.w13s = take((size_t)(E * 2 * P.Ip * P.Hp / 32));
  P.w2 = take((size_t)(E * P.Hp * P.Ip / 2));
  P.w2s = take((size_t)(E * P.Hp * P.Ip / 32));
  P.x = take((size_t)(T * P.Hp * 2));
  P.y = take((size_t)(T * P.Hp * 2));
  P.wr = take(routed ? (size_t)(E * P.Hp * 2) : 0);
  P.total = o;
  return P;
}

// scratch bytes of a layer call whose FP4 weights are 32-byte aligned
size_t layer_bytes(int64_t T, int64_t H, int64_t I, int64_t E, int64_t k, int act, bool routed) {
  return tc_widths(H, I) ? layout_for(T, H, I, E, k, act, routed).total
                         : pad_layout(T, H, I, E, k, act, routed).total;
}

int grid_for(int64_t work, int per_block, int cap) {
  int64_t g = (work + per_block - 1) / per_block;
  return (int)std::max<int64_t>(1, std::min<int64_t>(g, cap));
}

// Router logits [T, E] = x [T, H] (bf16) times W_r^T (W_r [E, H] bf16): a
// split-K GEMM into part[ks][t][e], then one kernel that sums the partials in
// a fixed order into `logits` and, for k > 0, runs step (1) on them into
// topk_idx / topk_w.  The first kernels of a call.
int enqueue_router(const void* x_bf16, const void* w_router, int T, int H, int E, float* part,
                   float* logits, DeviceState* d, cudaStream_t s, unsigned long long timeout_ns,
                   Steps& st, int k = 0, int32_t* topk_idx = nullptr, float* topk_w = nullptr) {
  const DensePlan P =
      plan_dense(E, T, H / 64, kRouterNMax, d->sms, router_part_bytes(T, E));
  DenseParams dp{};
  int rc;
  if ((rc = make_map(&dp.map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_router, H, E,
                     (uint64_t)H * 2, 64, 128)) ||
      (rc = make_map(&dp.map_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x_bf16, H, T,
                     (uint64_t)H * 2, 64, box_rows_for(T))))
    return rc;
  dp.box_rows_b = box_rows_for(T);
  dp.part = part;
  dp.M = E;
  dp.T = T;
  dp.m_tiles = P.m_tiles;
  dp.n_blocks = P.n_blocks;
  dp.k_splits = P.k_splits;
  dp.kb_per_split = P.kb_per_split;
  dp.kb_total = P.kb_total;
  dp.status = d->status;
  dp.timeout_ns = timeout_ns;
  const int items = P.m_tiles * P.n_blocks * P.k_splits;
  st.mark();
  dense_tc_kernel<kDenseBf16, kRouterNMax>
      <<<std::min(items, d->sms), kDenseThreads, DenseCfg<kDenseBf16, kRouterNMax>::kSmem, s>>>(
          dp);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  st.launched();
  if (P.k_splits > kTopkMaxSplits) return MOE_ERR_UNSUPPORTED_SHAPE;  // (kDenseMaxSplits)
  st.mark();
  const int vec = E % 4 == 0 ? 4 : 1;
  const dim3 grid(std::min(T, d->sms * 8));
  // above one token per SM (and up to 384 experts), two CTAs per SM
  const bool two = T > d->sms && E <= 384;
  const dim3 block(std::min(two ? kTopkThreads2 : kTopkThreads,
                            (kTopkGroups * (E / vec) + 31) / 32 * 32));
  auto go = [&](auto kernel) {
    return launch_pdl(kernel, grid, block, 0, s, (const float*)part, P.k_splits, T, E, k, logits,
                      topk_idx, topk_w, d->status);
  };
  const cudaError_t e =
      two ? (vec == 4 ? (E <= 128 ? go(splitk_topk_kernel<4, 4, 2>)
                                  : go(splitk_topk_kernel<12, 4, 2>))
                      : (E <= 128 ? go(splitk_topk_kernel<4, 1, 2>)
                                  : go(splitk_topk_kernel<12, 1, 2>)))
      : vec == 4 ? (E <= 128   ? go(splitk_topk_kernel<4, 4, 1>)
                    : E <= 384 ? go(splitk_topk_kernel<12, 4, 1>)
                               : go(splitk_topk_kernel<32, 4, 1>))
                 : (E <= 128   ? go(splitk_topk_kernel<4, 1, 1>)
                    : E <= 384 ? go(splitk_topk_kernel<12, 1, 1>)
                               : go(splitk_topk_kernel<32, 1, 1>));
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  st.launched();
  return MOE_OK;
}

// step (1): top-k + softmax into topk_idx / topk_w (see enqueue_route); an
// ordinary launch when it is the call's first kernel, else programmatic
int enqueue_topk(const float* logits, bool first, int T, int E, int k, int32_t* topk_idx,
                 float* topk_w, DeviceState* d, cudaStream_t s, Steps& st) {
  const dim3 grid(grid_for((int64_t)T * 32, 256, 1 << 30));
  st.mark();
  auto topk = [&](auto kernel) {
    if (first) {
      kernel<<<grid, 256, 0, s>>>(logits, T, E, k, topk_idx, topk_w, d->status);
      return cudaGetLastError();
    }
    return launch_pdl(kernel, grid, dim3(256), 0, s, logits, T, E, k, topk_idx, topk_w,
                      d->status);
  };
  const cudaError_t te = E <= 128   ? topk(route_topk_kernel<4>)
                         : E <= 384 ? topk(route_topk_kernel<12>)
                                    : topk(route_topk_kernel<32>);
  if (te != cudaSuccess) return MOE_ERR_CUDA;
  st.launched();
  return MOE_OK;
}

// Routing steps (1)-(4) into w; `first`: the top-k is the call's first kernel;
// `topk_done`: step (1) already ran (the router's last kernel), only (2)-(4)
int enqueue_route(const float* logits, bool first, int T, int E, int k, int chunk_max,
                  const Work& w, DeviceState* d, cudaStream_t s, Steps& st,
                  bool topk_done = false) {
  int rc = topk_done ? MOE_OK : enqueue_topk(logits, first, T, E, k, w.topk_idx, w.topk_w, d, s, st);
  if (rc) return rc;
  st.mark();
  const size_t smem = (size_t)(35 * E + 35) * sizeof(int);
  if (launch_pdl(route_permute_kernel, dim3(1), dim3(1024), smem, s, w.topk_idx, T, k, E, w.cnt,
                 w.off, w.perm, w.pos, w.chunks, w.max_chunks, chunk_max, w.meta, w.done,
                 d->status) != cudaSuccess)
    return MOE_ERR_CUDA;
  st.launched();
  return launch_status();
}

// CTAs of the small-block routing kernel: step a4 has T * ceil(H / 1024)
// token-major warp units; each CTA's warps T..31 take one unit while warps
// 0..T-1 run the top-k (all 32 warps take units after the routing when
// T = 32), so this many CTAs cover the units in one round.  One CTA when there
// is no a4 (routing alone).
int small_route_grid(int T_act, int H, int sms) {
  const int64_t units = (int64_t)T_act * ((H / 32 + 31) / 32);
  const int per = T_act < kSmallRouteTokens ? kSmallRouteTokens - T_act : kSmallRouteTokens;
  return grid_for(units, per, sms);
}

// Steps a1-a4 in one launch for a block of T <= kSmallRouteTokens tokens
// (route_act_small_kernel); `first`: the call's first kernel (ordinary launch);
// x == nullptr: routing alone (no a4)
int enqueue_route_act_small(const float* logits, bool first, int act, const uint16_t* x, int T,
                            int H, int E, int k, int chunk_max, const Work& w, DeviceState* d,
                            cudaStream_t s, Steps& st) {
  const dim3 grid(small_route_grid(x ? T : 0, H, d->sms));
  const size_t smem = small_route_smem(T, E, k, w.max_chunks).total;
  st.mark();
  auto go = [&](auto kernel) {
    if (first) {
      kernel<<<grid, 1024, smem, s>>>(logits, x, T, H, E, k, w.max_chunks, chunk_max, w.topk_idx,
                                      w.topk_w, w.cnt, w.off, w.perm, w.pos, w.chunks, w.meta,
                                      w.done, w.xq, w.xs, d->status);
      return cudaGetLastError();
    }
    return launch_pdl(kernel, grid, dim3(1024), smem, s, logits, x, T, H, E, k, w.max_chunks,
                      chunk_max, w.topk_idx, w.topk_w, w.cnt, w.off, w.perm, w.pos, w.chunks,
                      w.meta, w.done, w.xq, w.xs, d->status);
  };
  cudaError_t e;
  if (act == MOE_ACT_MXFP8)
    e = E <= 128 ? go(route_act_small_kernel<4, true>)
        : E <= 384 ? go(route_act_small_kernel<12, true>)
                   : go(route_act_small_kernel<32, true>);
  else
    e = E <= 128 ? go(route_act_small_kernel<4, false>)
        : E <= 384 ? go(route_act_small_kernel<12, false>)
                   : go(route_act_small_kernel<32, false>);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  st.launched();
  return MOE_OK;
}

// Routing steps (1)-(4) of every layer of a chain in two launches (the first
// an ordinary launch: it starts the call); layer l's routing block lies
// l * stride bytes after layer 0's (w0)
int enqueue_route_layers(const float* const* logits, int n, int T, int E, int k, int chunk_max,
                         const Work& w0, int64_t stride, DeviceState* d, cudaStream_t s,
                         Steps& st) {
  LayerLogits lg{};
  for (int l = 0; l < n; ++l) lg.p[l] = logits[l];
  const dim3 grid(grid_for((int64_t)T * 32, 256, 1 << 30), n);
  st.mark();
  auto topk = [&](auto kernel) {
    kernel<<<grid, 256, 0, s>>>(lg, T, E, k, w0.topk_idx, w0.topk_w, stride, d->status);
    return cudaGetLastError();
  };
  const cudaError_t te = E <= 128   ? topk(route_topk_layers_kernel<4>)
                         : E <= 384 ? topk(route_topk_layers_kernel<12>)
                                    : topk(route_topk_layers_kernel<32>);
  if (te != cudaSuccess) return MOE_ERR_CUDA;
  st.launched();
  st.mark();
  const size_t smem = (size_t)(35 * E + 35) * sizeof(int);
  if (launch_pdl(route_permute_layers_kernel, dim3(n), dim3(1024), smem, s,
                 (const int32_t*)w0.topk_idx, T, k, E, w0.cnt, w0.off, w0.perm, w0.pos, w0.chunks,
                 w0.max_chunks, chunk_max, w0.meta, w0.done, stride, d->status) != cudaSuccess)
    return MOE_ERR_CUDA;
  st.launched();
  return launch_status();
}

// Routing of every layer of a chain over a block of T <= kSmallRouteTokens
// tokens, and layer 0's step a4, in one ordinary launch (the call's first):
// route_act_small_layers_kernel; layer l's routing block lies l * stride
// bytes after layer 0's (w0)
int enqueue_route_act_small_layers(const float* const* logits, int n, int act, const uint16_t* x,
                                   int T, int H, int E, int k, int chunk_max, const Work& w0,
                                   int64_t stride, DeviceState* d, cudaStream_t s, Steps& st) {
  LayerLogits lg{};
  for (int l = 0; l < n; ++l) lg.p[l] = logits[l];
  // layer 0's CTAs, then one CTA per later layer
  const int g0 = small_route_grid(T, H, d->sms);
  const dim3 grid(g0 + n - 1);
  const size_t smem = small_route_smem(T, E, k, w0.max_chunks).total;
  st.mark();
  auto go = [&](auto kernel) {
    kernel<<<grid, 1024, smem, s>>>(lg, x, T, H, E, k, w0.max_chunks, chunk_max, w0.topk_idx,
                                    w0.topk_w, w0.cnt, w0.off, w0.perm, w0.pos, w0.chunks,
                                    w0.meta, w0.done, w0.xq, w0.xs, stride, g0, d->status);
    return cudaGetLastError();
  };
  cudaError_t e;
  if (act == MOE_ACT_MXFP8)
    e = E <= 128 ? go(route_act_small_layers_kernel<4, true>)
        : E <= 384 ? go(route_act_small_layers_kernel<12, true>)
                   : go(route_act_small_layers_kernel<32, true>);
  else
    e = E <= 128 ? go(route_act_small_layers_kernel<4, false>)
        : E <= 384 ? go(route_act_small_layers_kernel<12, false>)
                   : go(route_act_small_layers_kernel<32, false>);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  st.launched();
  return MOE_OK;
}

// The path MOE_PATH_AUTO takes: one launch for both GEMMs when the bound on
// GEMM work items per SM is at most kPersistentItemsPerSm, else two.  One
// launch removes the gap and the tail between the GEMMs and fills GEMM1's last
// wave with GEMM2 items; with many items per SM the two specialised launches
// stream weights faster (measured, µs, L2 emptied: full per-expert shape at
// T = 64, 108 items per SM: one launch 913.5, two 919.8; at T = 256, 121 per
// SM: 1265.6 against 1258.7).  The bound uses at most min(T*k, E) touched
// experts.
#ifndef MOE_PERSISTENT_ITEMS_PER_SM
#define MOE_PERSISTENT_ITEMS_PER_SM 110
#endif
constexpr int kPersistentItemsPerSm = MOE_PERSISTENT_ITEMS_PER_SM;
int auto_path(int T, int H, int I, int E, int k, int act, int sms) {
  if (act != MOE_ACT_MXFP8) return MOE_PATH_MULTI;  // the bf16 GEMMs are two launches
  const int64_t TK = (int64_t)T * k;
  const bool wide = T >= kWideMinTokens;
  const int64_t chunk_bound = std::min<int64_t>(TK, E) + TK / (wide ? kChunkWide : kChunkNarrow);
  const int64_t item_bound = chunk_bound * (I / 128 + (H + 255) / 256);
  return item_bound <= (int64_t)kPersistentItemsPerSm * sms ? MOE_PATH_GEMMS : MOE_PATH_MULTI;
}

// step a4: x rows into slot order, MXFP8-quantised or copied as bf16; each
// token's row is read once and written to its k slots (pos from the routing)
int enqueue_act(int act, const uint16_t* x, const Work& w, int T, int H, int k, DeviceState* d,
                cudaStream_t stream, Steps& st) {
  const int64_t units = (int64_t)T * ((H / 32 + 31) / 32);
  const dim3 grid(grid_for(units, 8, d->sms * 8));
  st.mark();
  const cudaError_t qe =
      act == MOE_ACT_MXFP8
          ? launch_pdl(act_tokens_kernel<true>, grid, dim3(256), 0, stream, x,
                       (const int32_t*)w.pos, T, k, (int64_t)H, w.xq, w.xs, d->status)
          : launch_pdl(act_tokens_kernel<false>, grid, dim3(256), 0, stream, x,
                       (const int32_t*)w.pos, T, k, (int64_t)H, w.xq, w.xs, d->status);
  if (qe != cudaSuccess) return MOE_ERR_CUDA;
  st.launched();
  return MOE_OK;
}

// The MXFP8 GEMMs' parameters: phase 0 = GEMM1 (gate/up rows paired, SwiGLU
// epilogue into hq/hs), phase 1 = GEMM2 (output rows r and r + 128 paired,
// fp32 rows into yp)
// `two_launch`: the GEMMs run as two launches (the large layers); GEMM2's
// weight copies then promote L2 fills to 128 bytes instead of 256 (one box,
// back to back: full_t256 1275 -> 1267.5 us, GEMM2 417 -> 408 us; GEMM1 is
// faster with 256, 842 against 853 us, and so are the one-launch GEMMs of the
// small layers)
int mxfp8_gemm_params(const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2,
                      const uint8_t* w2s, int T, int H, int I, int E, int k, const Work& w,
                      DeviceState* d, unsigned long long timeout_ns, TcParams& p,
                      bool two_launch = false) {
  const int TK = T * k;
  TcPhase& g1 = p.ph[0];
  TcPhase& g2 = p.ph[1];
  const CUtensorMapL2promotion wp2 =
      two_launch ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  int rc;
  if ((rc = make_map(&g1.map_w, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w13, H, (uint64_t)E * 2 * I,
                     H / 2, 128, 128)) ||
      (rc = make_map(&g1.map_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.xq, H, TK, H, 128, kBoxRowsB)) ||
      (rc = make_map(&g2.map_w, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w2, I, (uint64_t)E * H,
                     I / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B, wp2)) ||
      (rc = make_map(&g2.map_x, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.hq, I, TK, I, 128, kBoxRowsB)))
    return rc;
  g1.w_sf = w13s;
  g1.x_sf = w.xs;
  g1.K = H;
  g1.R = 2 * I;
  g1.m_tiles = I / 128;
  g1.m_stride = 128;
  g1.half = I;
  g1.out_dim = I;
  g1.rows_total = E * 2 * I;
  g2.w_sf = w2s;
  g2.x_sf = w.hs;
  g2.K = I;
  g2.R = H;
  g2.m_tiles = (H + 255) / 256;  // an odd last tile pairs with rows past the expert
  g2.m_stride = 256;
  g2.half = 128;
  g2.out_dim = H;
  g2.rows_total = E * H;
  p.chunks = w.chunks;
  p.meta = w.meta;
  p.hq = w.hq;
  p.hs = w.hs;
  p.yp = w.yp;
  p.status = d->status;
  p.timeout_ns = timeout_ns;
  return MOE_OK;
}

std::atomic<uint32_t> g_calls{0};  // host call number: the salt of the grid barriers' tags

// the barrier words of a persistent launch (in the call's scratch) and a new salt
void set_grid_sync(TcParams& p, const Work& w) {
  p.sync.counter = reinterpret_cast<uint32_t*>(w.sync);
  p.sync.abort = reinterpret_cast<uint64_t*>(w.sync + 8);
  p.sync.flags = reinterpret_cast<uint64_t*>(w.sync + 16);
  p.sync.chunk_flags = reinterpret_cast<uint64_t*>(w.sync + kGridSyncBytes);
  p.sync.salt = g_calls.fetch_add(1, std::memory_order_relaxed) + 1;
}
constexpr int kLayerLaunchTooLarge = 1;   // enqueue_layer: the cooperative launch was refused

// The whole layer in one persistent launch (MXFP8 mode): both GEMMs and the
// combine; with `route_in` (T <= kSmallRouteTokens) also the routing and the
// activation step, and with `w_router` the router in front (its logits are
// written to `logits`).  Without `route_in` the routing kernels have run
// before (w holds their arrays).
int enqueue_layer(const float* logits, const uint16_t* x, const uint8_t* w13, const uint8_t* w13s,
                  const uint8_t* w2, const uint8_t* w2s, int T, int H, int I, int E, int k,
                  bool route_in, bool first, const Work& w, void* y, DeviceState* d,
                  cudaStream_t stream, unsigned long long timeout_ns, const moe_opts* opts,
                  Steps& st, const void* w_router = nullptr) {
  TcParams p{};
  int rc;
  if ((rc = mxfp8_gemm_params(w13, w13s, w2, w2s, T, H, I, E, k, w, d, timeout_ns, p))) return rc;
  p.gemm1_done = w.done;
  p.ph[1].dep_target = 4 * p.ph[0].m_tiles;  // four epilogue warps publish per tile pair
  if (opts && (opts->debug_flags & MOE_DEBUG_FORCE_DEP_TIMEOUT))
    p.ph[1].dep_target = INT_MAX;  // never reached: the dependency wait runs out
  if (route_in) {
    LayerRouteParams& r = p.route;
    r.logits = logits;
    r.x = x;
    r.w_router = static_cast<const uint16_t*>(w_router);
    r.T = T;
    r.E = E;
    r.k = k;
    r.chunk_max = kChunkNarrow;
    r.max_chunks = w.max_chunks;
    r.topk_idx = w.topk_idx;
    r.topk_w = w.topk_w;
    r.cnt = w.cnt;
    r.off = w.off;
    r.perm = w.perm;
    r.pos = w.pos;
    r.chunks = w.chunks;
    r.meta = w.meta;
    r.xq = w.xq;
    r.xs = w.xs;
  }
  set_grid_sync(p, w);
  p.pos = w.pos;
  p.gate = w.topk_w;
  p.y = static_cast<uint16_t*>(y);
  p.T = T;
  p.H = H;
  p.k = k;
  if (d->sms > kMaxGridSync) return MOE_ERR_UNSUPPORTED_SHAPE;
  const bool wide = T >= kWideMinTokens;
  st.mark();
  const cudaError_t e = wide ? launch_gemm<kChunkWide>(kModeLayer, d->sms, stream, p, first)
                             : launch_gemm<kChunkNarrow>(kModeLayer, d->sms, stream, p, first);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    // the GPU cannot hold every CTA at once (e.g. a partitioned device):
    // nothing ran, the caller takes the multi-launch path
    return e == cudaErrorCooperativeLaunchTooLarge ? kLayerLaunchTooLarge : MOE_ERR_CUDA;
  }
  st.launched();
  return launch_status();
}

// steps a5-a7: the two grouped GEMMs (one persistent launch or two)
// `next` (a chained layer, MXFP8 mode): the last GEMM launch prefetches the
// next layer's first GEMM1 weight tiles into L2
// `chunks_before`: the chunk list was final before the kernel in front of the
// GEMMs started (that kernel is the activation step or a combine), so a GEMM1
// launch may start its weight stream before its dependency wait (GEMM2
// launches always may; the both-GEMMs launch does not: the copy code cost its
// stages more than the early start gained).
int enqueue_gemms(int act, int path, const uint8_t* w13, const uint8_t* w13s, const uint8_t* w2,
                  const uint8_t* w2s, int T, int H, int I, int E, int k, const Work& w,
                  DeviceState* d, cudaStream_t stream, unsigned long long timeout_ns,
                  const moe_opts* opts, Steps& st, const NextGemm1* next = nullptr,
                  bool chunks_before = false) {
  const int TK = T * k;
  const bool wide = act == MOE_ACT_MXFP8 && T >= kWideMinTokens;
  const bool bf_wide = chunk_for(act, T) == kChunkBf16Wide;
  int rc = MOE_OK;
  if (act == MOE_ACT_MXFP8) {
    // both GEMMs in one launch: the chain's MOE_PATH_PERSISTENT asks for it
    // too (the chain has no whole-layer launch)
    bool persistent = path == MOE_PATH_GEMMS || path == MOE_PATH_PERSISTENT ||
                      (path == MOE_PATH_AUTO &&
                       auto_path(T, H, I, E, k, act, d->sms) == MOE_PATH_GEMMS);
    TcParams p{};
    if ((rc = mxfp8_gemm_params(w13, w13s, w2, w2s, T, H, I, E, k, w, d, timeout_ns, p,
                                !persistent)))
      return rc;
    TcPhase g1 = p.ph[0], g2 = p.ph[1];
    auto launch = [&](int mode, const TcParams& prm) {
      const cudaError_t e = wide ? launch_gemm<kChunkWide>(mode, d->sms, stream, prm)
                                 : launch_gemm<kChunkNarrow>(mode, d->sms, stream, prm);
      if (e == cudaSuccess) st.launched();
      return e;
    };
    p.early_chunks = chunks_before ? 1 : 0;
    if (persistent) {  // both GEMMs in one launch
      g2.dep_target = 4 * g1.m_tiles;  // four epilogue warps publish per tile pair
      if (opts && (opts->debug_flags & MOE_DEBUG_FORCE_DEP_TIMEOUT))
        g2.dep_target = INT_MAX;  // never reached: the dependency wait runs out
      p.gemm1_done = w.done;
      p.ph[0] = g1;
      p.ph[1] = g2;
      if (next) p.next = *next;
      st.mark();
      const cudaError_t e = launch(kModeBoth, p);
      if (e == cudaErrorCooperativeLaunchTooLarge) {
        // the GPU cannot hold every CTA at once (e.g. a partitioned device):
        // nothing ran, so take the two-launch path
        (void)cudaGetLastError();
        persistent = false;
      } else if (e != cudaSuccess) {
        return MOE_ERR_CUDA;
      }
    }
    if (!persistent) {
      p.gemm1_done = nullptr;
      p.ph[1] = TcPhase{};
      p.ph[0] = g1;
      p.next = NextGemm1{};  // only the layer's last launch prefetches
      st.mark();
      if (launch(kModeGemm1, p) != cudaSuccess) return MOE_ERR_CUDA;
      p.ph[0] = g2;
      p.next = next ? *next : NextGemm1{};
      p.early_chunks = 1;  // GEMM1 ran after the routing finished
      st.mark();
      if (launch(kModeGemm2, p) != cudaSuccess) return MOE_ERR_CUDA;
    }
  } else {
    // bf16 activations: weights decoded to bf16 in TMEM, kind::f16 MMA
    BfParams b1{}, b2{};
    if ((rc = make_map(&b1.map_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w13, H / 2, (uint64_t)E * 2 * I,
                       H / 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_64B)) ||
        (rc = make_map(&b1.map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w.xq, H, TK, (uint64_t)H * 2,
                       64, 16)) ||
        (rc = make_map(&b2.map_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w2, I / 2, (uint64_t)E * H, I / 2,
                       64, 128, CU_TENSOR_MAP_SWIZZLE_64B)) ||
        (rc = make_map(&b2.map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w.hq, I, TK, (uint64_t)I * 2,
                       64, 16)))
      return rc;
    for (BfParams* b : {&b1, &b2}) {
      b->chunks = reinterpret_cast<const int4*>(w.chunks);
      b->meta = w.meta;
      b->status = d->status;
      b->timeout_ns = timeout_ns;
    }
    b1.w_sf = w13s;
    b1.stall_decode = opts && (opts->debug_flags & MOE_DEBUG_STALL_DECODE) ? 1 : 0;
    b1.hq = reinterpret_cast<uint16_t*>(w.hq);
    b1.K = H;
    b1.R = 2 * I;
    b1.m_tiles = I / 128;
    b1.m_stride = 128;
    b1.half = I;
    b1.out_dim = I;
    b1.rows_total = E * 2 * I;
    b2.w_sf = w2s;
    b2.yp = w.yp;
    b2.K = I;
    b2.R = H;
    b2.m_tiles = (H + 255) / 256;  // an odd last tile pairs with rows past the expert
    b2.m_stride = 256;
    b2.half = 128;
    b2.out_dim = H;
    b2.rows_total = E * H;
    st.mark();
    if ((bf_wide ? launch_pdl(gemm_bf16_kernel<kChunkBf16Wide, true>, dim3(d->sms),
                              dim3(kBfThreads), BfCfg<kChunkBf16Wide>::kSmem, stream, b1)
                 : launch_pdl(gemm_bf16_kernel<kChunkNarrow, true>, dim3(d->sms),
                              dim3(kBfThreads), BfCfg<kChunkNarrow>::kSmem, stream, b1)) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    st.launched();
    st.mark();
    if ((bf_wide ? launch_pdl(gemm_bf16_kernel<kChunkBf16Wide, false>, dim3(d->sms),
                              dim3(kBfThreads), BfCfg<kChunkBf16Wide>::kSmem, stream, b2)
                 : launch_pdl(gemm_bf16_kernel<kChunkNarrow, false>, dim3(d->sms),
                              dim3(kBfThreads), BfCfg<kChunkNarrow>::kSmem, stream, b2)) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    st.launched();
  }
  return MOE_OK;
}

int forward_padded(const void* x_bf16, const float* logits, const uint8_t* w13,
                   const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s, int T, int H, int I,
                   int E, int k, void* y, cudaStream_t stream, const moe_opts* opts,
                   const void* w_router);

// The layer.  Exactly one of `logits` (router logits [T, E]) and `w_router`
// (router weights [E, H] bf16: the router GEMM runs in front of the top-k)
// is given.
int forward_impl(const void* x_bf16, const float* logits, const uint8_t* w13, const uint8_t* w13s,
                 const uint8_t* w2, const uint8_t* w2s, int T, int H, int I, int E, int k,
                 void* y, cudaStream_t stream, const moe_opts* opts,
                 const void* w_router = nullptr) {
  if (!x_bf16 || (!logits == !w_router) || !w13 || !w13s || !w2 || !w2s || !y)
    return MOE_ERR_INVALID_ARG;
  int rc = validate_shape(T, H, I, E, k);
  if (rc) return rc;
  const bool routed = w_router != nullptr;
  if (routed && !aligned(w_router, 16)) return MOE_ERR_ALIGNMENT;
  const int act = opts ? opts->act_mode : MOE_ACT_MXFP8;
  const int path = opts ? opts->path : MOE_PATH_AUTO;
  if (act != MOE_ACT_MXFP8 && act != MOE_ACT_BF16) return MOE_ERR_INVALID_ARG;
  if (path < MOE_PATH_AUTO || path > MOE_PATH_GEMMS) return MOE_ERR_INVALID_ARG;
  if (!aligned(w13, 16) || !aligned(w2, 16) || !aligned(x_bf16, 16) || !aligned(logits, 16) ||
      !aligned(w13s, 16) || !aligned(w2s, 16) || !aligned(y, 16))
    return MOE_ERR_ALIGNMENT;
  if (opts && opts->workspace && !aligned(opts->workspace, 256)) return MOE_ERR_ALIGNMENT;
  if (!tc_widths(H, I) || !aligned(w13, 32) || !aligned(w2, 32))
    return forward_padded(x_bf16, logits, w13, w13s, w2, w2s, T, H, I, E, k, y, stream, opts,
                          w_router);
  const Layout L = layout_for(T, H, I, E, k, act, routed);
  if (opts && opts->workspace && opts->workspace_bytes < L.total) return MOE_ERR_NO_MEMORY;
  if (T == 0) return MOE_OK;

  DeviceState* d = nullptr;
  if ((rc = device_state(&d))) return rc;
  void* ws = opts ? opts->workspace : nullptr;
  if (!ws && (rc = cached_workspace(d, L.total, &ws))) return rc;
  const Work w = carve(ws, L);

  const unsigned long long timeout_ns =
      (opts && (opts->debug_flags & MOE_DEBUG_SHORT_TIMEOUT)) ? 1000000ull : 2000000000ull;
  Steps st{opts, stream};
  const float* lg = routed ? w.rlogits : logits;
  const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
  // wide token chunks cut the MMA instructions per token when experts get
  // many tokens (large T); narrow chunks keep the weight pipeline deepest
  const int chunk = chunk_for(act, T);
  const bool split = opts && (opts->debug_flags & MOE_DEBUG_SPLIT_ROUTING);
  // the whole layer in one launch (explicit MOE_PATH_PERSISTENT); the other
  // paths run routing, GEMMs and combine as stream-ordered kernels, the GEMMs
  // as one launch (MOE_PATH_GEMMS) or two
  const bool persistent = act == MOE_ACT_MXFP8 && path == MOE_PATH_PERSISTENT;
  const int gemm_path =
      act != MOE_ACT_MXFP8 ? MOE_PATH_MULTI
      : path == MOE_PATH_AUTO ? auto_path(T, H, I, E, k, act, d->sms)
      : path == MOE_PATH_PERSISTENT ? MOE_PATH_MULTI  // (only after a refused layer launch)
                                    : path;
  // the whole layer in one launch: for T <= 32 also the routing (steps a1-a4)
  const bool route_in = persistent && T <= kSmallRouteTokens && !split;
  if (route_in) {  // (with the router inside too when the layer is routed)
    rc = enqueue_layer(lg, x, w13, w13s, w2, w2s, T, H, I, E, k, true, true, w, y, d, stream,
                       timeout_ns, opts, st, w_router);
    if (rc != kLayerLaunchTooLarge) {
      if (rc) return rc;
      st.mark();
      return launch_status();
    }
  }
  // the router's last kernel also runs step (1) when the split routing
  // kernels follow (the small-block kernel routes from the logits itself)
  const bool small_route = T <= kSmallRouteTokens && !split;
  if (routed && (rc = enqueue_router(x_bf16, w_router, T, H, E, w.part, w.rlogits, d, stream,
                                     timeout_ns, st, small_route ? 0 : k, w.topk_idx,
                                     w.topk_w)))
    return rc;
  if (small_route) {
    if ((rc = enqueue_route_act_small(lg, !routed, act, x, T, H, E, k, chunk, w, d, stream, st)))
      return rc;
  } else if ((rc = enqueue_route(lg, !routed, T, E, k, chunk, w, d, stream, st, routed)) ||
             (rc = enqueue_act(act, x, w, T, H, k, d, stream, st))) {
    return rc;
  }
  if (persistent && !route_in) {
    rc = enqueue_layer(lg, x, w13, w13s, w2, w2s, T, H, I, E, k, false, false, w, y, d, stream,
                       timeout_ns, opts, st);
    if (rc != kLayerLaunchTooLarge) {
      if (rc) return rc;
      st.mark();
      return launch_status();
    }
  }
  // (the small-block routing kernel writes the chunk list right before the
  // GEMMs; the split path's activation step runs after it is final; the GEMM
  // kernels of wide chunks, T >= kWideMinTokens, have no early copies)
  const bool chunks_before = !small_route && T < kWideMinTokens;
  if ((rc = enqueue_gemms(act, gemm_path, w13, w13s, w2, w2s, T, H, I, E, k, w, d, stream,
                          timeout_ns, opts, st, nullptr, chunks_before)))
    return rc;
  const int cap = d->sms * 8;
  st.mark();
  if (launch_pdl(combine_kernel, dim3(grid_for((int64_t)T * H / 4, 256, cap)), dim3(256), 0,
                 stream, (const float*)w.yp, (const int32_t*)w.pos, (const float*)w.topk_w, T, H,
                 k, static_cast<uint16_t*>(y)) != cudaSuccess)
    return MOE_ERR_CUDA;
  st.launched();
  st.mark();
  return launch_status();
}

// The layer on zero-padded copies: weights, x (and the router weights) are
// copied into the scratch with H and I rounded up to multiples of 128 (gate
// rows to [0, I), up rows to [Ip, Ip + I) of each expert's padded w13), the
// padded layer runs, and y keeps the first H columns of its padded output.
// The added weights and activations are zero, so every real output is the
// same sum as without them.  The copies are made on every call (one read and
// one write of the weights): a path for shapes the GEMMs cannot take, not a
// fast one.
int forward_padded(const void* x_bf16, const float* logits, const uint8_t* w13,
                   const uint8_t* w13s, const uint8_t* w2, const uint8_t* w2s, int T, int H, int I,
                   int E, int k, void* y, cudaStream_t stream, const moe_opts* opts,
                   const void* w_router) {
  const bool routed = w_router != nullptr;
  const int act = opts ? opts->act_mode : MOE_ACT_MXFP8;
  const PadLayout P = pad_layout(T, H, I, E, k, act, routed);
  if (opts && opts->workspace && opts->workspace_bytes < P.total) return MOE_ERR_NO_MEMORY;
  if (T == 0) return MOE_OK;
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  void* ws = opts ? opts->workspace : nullptr;
  if (!ws && (rc = cached_workspace(d, P.total, &ws))) return rc;
  uint8_t* b = static_cast<uint8_t*>(ws);
  const int64_t Hp = P.Hp, Ip = P.Ip;
  const dim3 grid(d->sms * 4), block(256);
  Steps st{nullptr, stream};
  // the first copy is an ordinary launch: the previous call may still use
  // the scratch; the others (and the padded layer's kernels) follow in order
  bool first = true;
  auto pad = [&](const void* src, uint8_t* dst, int64_t groups, int64_t src_rows,
                 int64_t dst_rows, int64_t src_row_bytes, int64_t dst_row_bytes, int64_t n0,
                 int64_t d1 = 0, int64_t n1 = 0, int64_t s1 = 0) {
    const PadSpec ps{static_cast<const uint8_t*>(src), dst, groups, src_rows, dst_rows,
                     src_row_bytes, dst_row_bytes, 0, n0, 0, d1, n1, s1};
    cudaError_t e;
    if (first) {
      pad_rows_kernel<<<grid, block, 0, stream>>>(ps);
      e = cudaGetLastError();
    } else {
      e = launch_pdl(pad_rows_kernel, grid, block, 0, stream, ps);
    }
    first = false;
    st.launched();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  };
  if ((rc = pad(w13, b + P.w13, E, 2 * I, 2 * Ip, H / 2, Hp / 2, I, Ip, I, I)) ||
      (rc = pad(w13s, b + P.w13s, E, 2 * I, 2 * Ip, H / 32, Hp / 32, I, Ip, I, I)) ||
      (rc = pad(w2, b + P.w2, E, H, Hp, I / 2, Ip / 2, H)) ||
      (rc = pad(w2s, b + P.w2s, E, H, Hp, I / 32, Ip / 32, H)) ||
      (rc = pad(x_bf16, b + P.x, 1, T, T, 2 * H, 2 * Hp, T)) ||
      (routed && (rc = pad(w_router, b + P.wr, 1, E, E, 2 * H, 2 * Hp, E))))
    return rc;
  moe_opts o = opts ? *opts : moe_opts{};
  o.act_mode = act;
  o.workspace = ws;
  o.workspace_bytes = P.inner.total;
  if ((rc = forward_impl(b + P.x, logits, b + P.w13, b + P.w13s, b + P.w2, b + P.w2s, T,
                         (int)Hp, (int)Ip, E, k, b + P.y, stream, &o,
                         routed ? b + P.wr : nullptr)))
    return rc;
  return pad(b + P.y, static_cast<uint8_t*>(y), 1, T, T, 2 * Hp, 2 * H, T);
}

// A chain of layers over one token block: x_0 = x, x_{l+1} = bf16_RNE(y_l +
// residual * x_l), y = x_n.  Routing depends only on each layer's logits, so
// every layer is routed first, all layers at once (two launches, or at T <= 32
// one that also runs layer 0's activation step); then per
// layer the GEMMs run and the combine writes layer l+1's activation rows
// directly (combine_next_kernel).
int chain_impl(int n, const void* x_bf16, const float* const* logits,
               const uint8_t* const* w13, const uint8_t* const* w13s, const uint8_t* const* w2,
               const uint8_t* const* w2s, int T, int H, int I, int E, int k, int residual,
               void* y, cudaStream_t stream, const moe_opts* opts) {
  if (n < 1 || n > MOE_MAX_CHAIN || !x_bf16 || !logits || !w13 || !w13s || !w2 || !w2s || !y ||
      (residual != 0 && residual != 1))
    return MOE_ERR_INVALID_ARG;
  int rc = validate_shape(T, H, I, E, k);
  if (rc) return rc;
  if (!tc_widths(H, I)) return MOE_ERR_UNSUPPORTED_SHAPE;  // chains take no padded layers
  const int act = opts ? opts->act_mode : MOE_ACT_MXFP8;
  const int path = opts ? opts->path : MOE_PATH_AUTO;
  if (act != MOE_ACT_MXFP8 && act != MOE_ACT_BF16) return MOE_ERR_INVALID_ARG;
  if (path < MOE_PATH_AUTO || path > MOE_PATH_GEMMS) return MOE_ERR_INVALID_ARG;
  if (!aligned(x_bf16, 16) || !aligned(y, 16)) return MOE_ERR_ALIGNMENT;
  for (int l = 0; l < n; ++l) {
    if (!logits[l] || !w13[l] || !w13s[l] || !w2[l] || !w2s[l]) return MOE_ERR_INVALID_ARG;
    if (!aligned(logits[l], 16) || !aligned(w13[l], 32) || !aligned(w2[l], 32) ||
        !aligned(w13s[l], 16) || !aligned(w2s[l], 16))
      return MOE_ERR_ALIGNMENT;
  }
  const ChainLayout C = chain_layout(n, T, H, I, E, k, act);
  if (opts && opts->workspace) {
    if (!aligned(opts->workspace, 256)) return MOE_ERR_ALIGNMENT;
    if (opts->workspace_bytes < C.total) return MOE_ERR_NO_MEMORY;
  }
  if (T == 0) return MOE_OK;

  DeviceState* d = nullptr;
  if ((rc = device_state(&d))) return rc;
  void* ws = opts ? opts->workspace : nullptr;
  if (!ws && (rc = cached_workspace(d, C.total, &ws))) return rc;
  uint16_t* xb[2] = {reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + C.xb[0]),
                     reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + C.xb[1])};
  const unsigned long long timeout_ns =
      (opts && (opts->debug_flags & MOE_DEBUG_SHORT_TIMEOUT)) ? 1000000ull : 2000000000ull;
  Steps st{opts, stream};
  const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
  const bool small_route =
      T <= kSmallRouteTokens && !(opts && (opts->debug_flags & MOE_DEBUG_SPLIT_ROUTING));
  if (small_route) {
    if ((rc = enqueue_route_act_small_layers(logits, n, act, x, T, H, E, k, chunk_for(act, T),
                                             carve_chain(ws, C, 0), (int64_t)C.route_block, d,
                                             stream, st)))
      return rc;
  } else {
    if ((rc = enqueue_route_layers(logits, n, T, E, k, chunk_for(act, T),
                                   carve_chain(ws, C, 0), (int64_t)C.route_block, d, stream,
                                   st)))
      return rc;
    if ((rc = enqueue_act(act, x, carve_chain(ws, C, 0), T, H, k, d, stream, st))) return rc;
  }
  if (act == MOE_ACT_MXFP8 && path == MOE_PATH_PERSISTENT) {
    // Whole layers in one launch: up to kMaxLaunchLayers layers per launch,
    // each layer's combine writing the next layer's act1 rows (and, with the
    // residual, the stream) inside the launch.
    const bool wide = T >= kWideMinTokens;
    for (int l0 = 0; l0 < n; l0 += kMaxLaunchLayers) {
      const int nl = std::min(kMaxLaunchLayers, n - l0);
      ChainParams cp{};
      const Work w0 = carve_chain(ws, C, l0);
      if ((rc = mxfp8_gemm_params(w13[l0], w13s[l0], w2[l0], w2s[l0], T, H, I, E, k, w0, d,
                                  timeout_ns, cp.p)))
        return rc;
      cp.p.ph[1].dep_target = 4 * cp.p.ph[0].m_tiles;
      if (opts && (opts->debug_flags & MOE_DEBUG_FORCE_DEP_TIMEOUT))
        cp.p.ph[1].dep_target = INT_MAX;  // never reached: the dependency wait runs out
      set_grid_sync(cp.p, w0);
      cp.p.route.xq = w0.xq;  // the combines write the next layers' act1 rows here
      cp.p.route.xs = w0.xs;
      cp.p.T = T;
      cp.p.H = H;
      cp.p.k = k;
      for (int i = 0; i < nl; ++i) {
        const int l = l0 + i;
        const Work wl = carve_chain(ws, C, l);
        ChainLayer& L = cp.lay[i];
        if ((rc = make_map(&L.map_w[0], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w13[l], H,
                           (uint64_t)E * 2 * I, H / 2, 128, 128)) ||
            (rc = make_map(&L.map_w[1], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w2[l], I,
                           (uint64_t)E * H, I / 2, 128, 128)))
          return rc;
        L.w_sf[0] = w13s[l];
        L.w_sf[1] = w2s[l];
        L.chunks = wl.chunks;
        L.meta = wl.meta;
        L.pos = wl.pos;
        L.gate = wl.topk_w;
        const bool last = l == n - 1;
        L.x_res = residual ? (l == 0 ? x : xb[l & 1]) : nullptr;
        L.x_out = last ? static_cast<uint16_t*>(y) : residual ? xb[(l + 1) & 1] : nullptr;
        L.pos_next = last ? nullptr : carve_chain(ws, C, l + 1).pos;
      }
      cp.n_layers = nl;
      if (d->sms > kMaxGridSync) return MOE_ERR_UNSUPPORTED_SHAPE;
      st.mark();
      const cudaError_t e =
          wide ? launch_cooperative(gemm_chain_kernel<kChunkWide>, d->sms,
                                    tc_smem_bytes<kChunkWide, kModeLayer>(), stream, cp, false)
               : launch_cooperative(gemm_chain_kernel<kChunkNarrow>, d->sms,
                                    tc_smem_bytes<kChunkNarrow, kModeLayer>(), stream, cp,
                                    false);
      if (e != cudaSuccess) {
        (void)cudaGetLastError();
        // (a device that cannot hold every CTA at once: nothing of this launch ran)
        return e == cudaErrorCooperativeLaunchTooLarge ? MOE_ERR_UNSUPPORTED_SHAPE
                                                        : MOE_ERR_CUDA;
      }
      st.launched();
    }
    st.mark();
    return launch_status();
  }
  const int64_t threads = (int64_t)T * H / 4;
  for (int l = 0; l < n; ++l) {
    const Work w = carve_chain(ws, C, l);
    NextGemm1 nx{};
    if (l + 1 < n) {  // the next layer's first GEMM1 weight tiles, prefetched into L2
      const Work wn = carve_chain(ws, C, l + 1);
      if ((rc = make_map(&nx.map_w, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, w13[l + 1], H,
                         (uint64_t)E * 2 * I, H / 2, 128, 128)))
        return rc;
      nx.chunks = wn.chunks;
      nx.meta = wn.meta;
      nx.R = 2 * I;
      nx.m_tiles = I / 128;
      nx.m_stride = 128;
      nx.half = I;
      nx.stages = std::min(kChainPrefetchStages, H / 128);
    }
    // every layer was routed before the chain's first GEMMs; the kernel in
    // front of layer l's GEMMs is the previous layer's combine, or for layer 0
    // the activation step (or the small-block routing, which writes the lists)
    const bool chunks_before = (l > 0 || !small_route) && T < kWideMinTokens;
    if ((rc = enqueue_gemms(act, path, w13[l], w13s[l], w2[l], w2s[l], T, H, I, E, k, w, d,
                            stream, timeout_ns, opts, st, l + 1 < n ? &nx : nullptr,
                            chunks_before)))
      return rc;
    const bool last = l == n - 1;
    const uint16_t* x_res = residual ? (l == 0 ? x : xb[l & 1]) : nullptr;
    uint16_t* x_out = last ? static_cast<uint16_t*>(y) : residual ? xb[(l + 1) & 1] : nullptr;
    const int32_t* pos_next = last ? nullptr : carve_chain(ws, C, l + 1).pos;
    st.mark();
    const dim3 grid(grid_for(threads, 256, d->sms * 8));
    const cudaError_t e =
        act == MOE_ACT_MXFP8
            ? launch_pdl(combine_next_kernel<true>, grid, dim3(256), 0, stream,
                         (const float*)w.yp, (const int32_t*)w.pos, (const float*)w.topk_w, T, H,
                         k, x_res, x_out, pos_next, w.xq, w.xs, d->status)
            : launch_pdl(combine_next_kernel<false>, grid, dim3(256), 0, stream,
                         (const float*)w.yp, (const int32_t*)w.pos, (const float*)w.topk_w, T, H,
                         k, x_res, x_out, pos_next, w.xq, w.xs, d->status);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    st.launched();
  }
  st.mark();
  return launch_status();
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_mxfp4_forward(const void* x_bf16, const float* router_logits, const uint8_t* w13_fp4,
                      const uint8_t* w13_e8m0, const uint8_t* w2_fp4, const uint8_t* w2_e8m0,
                      int T, int H, int I, int E, int k, void* y_bf16, cudaStream_t stream) {
  return forward_impl(x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H, I, E, k,
                      y_bf16, stream, nullptr);
}

int moe_mxfp4_forward_ex(const void* x_bf16, const float* router_logits, const uint8_t* w13_fp4,
                         const uint8_t* w13_e8m0, const uint8_t* w2_fp4, const uint8_t* w2_e8m0,
                         int T, int H, int I, int E, int k, void* y_bf16, cudaStream_t stream,
                         const moe_opts* opts) {
  return forward_impl(x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H, I, E, k,
                      y_bf16, stream, opts);
}

size_t moe_mxfp4_workspace_size(int T, int H, int I, int E, int k, int act_mode) {
  if (validate_shape(T, H, I, E, k) != MOE_OK) return 0;
  if (act_mode != MOE_ACT_MXFP8 && act_mode != MOE_ACT_BF16) return 0;
  return layer_bytes(T, H, I, E, k, act_mode, false);
}

size_t moe_mxfp4_workspace_size_padded(int T, int H, int I, int E, int k, int act_mode,
                                       int routed) {
  if (validate_shape(T, H, I, E, k) != MOE_OK) return 0;
  if (act_mode != MOE_ACT_MXFP8 && act_mode != MOE_ACT_BF16) return 0;
  if (routed != 0 && routed != 1) return 0;
  return pad_layout(T, H, I, E, k, act_mode, routed == 1).total;
}

int moe_mxfp4_forward_chain(int n_layers, const void* x_bf16, const float* const* router_logits,
                            const uint8_t* const* w13_fp4, const uint8_t* const* w13_e8m0,
                            const uint8_t* const* w2_fp4, const uint8_t* const* w2_e8m0, int T,
                            int H, int I, int E, int k, int residual, void* y_bf16,
                            cudaStream_t stream, const moe_opts* opts) {
  return chain_impl(n_layers, x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H, I,
                    E, k, residual, y_bf16, stream, opts);
}

size_t moe_mxfp4_workspace_size_chain(int n_layers, int T, int H, int I, int E, int k,
                                      int act_mode) {
  if (n_layers < 1 || n_layers > MOE_MAX_CHAIN) return 0;
  if (validate_shape(T, H, I, E, k) != MOE_OK || !tc_widths(H, I)) return 0;
  if (act_mode != MOE_ACT_MXFP8 && act_mode != MOE_ACT_BF16) return 0;
  return chain_layout(n_layers, T, H, I, E, k, act_mode).total;
}

int moe_mxfp4_select_path(int T, int H, int I, int E, int k, int act_mode) {
  int rc = validate_shape(T, H, I, E, k);
  if (rc) return rc;
  if (act_mode != MOE_ACT_MXFP8 && act_mode != MOE_ACT_BF16) return MOE_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  if ((rc = device_state(&d))) return rc;
  return auto_path(T, (int)round128(H), (int)round128(I), E, k, act_mode, d->sms);
}

int mxfp4_quantize(const float* w, int64_t rows, int64_t K, uint8_t* out_fp4, uint8_t* out_e8m0,
                   cudaStream_t stream) {
  if (!w || !out_fp4 || !out_e8m0 || rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(w, 16) || !aligned(out_fp4, 16)) return MOE_ERR_ALIGNMENT;
  if (rows == 0) return MOE_OK;
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  const int64_t nblocks = rows * (K / 32);
  mxfp4_quantize_kernel<<<grid_for(nblocks, 256, d->sms * 16), 256, 0, stream>>>(
      w, nblocks, out_fp4, out_e8m0);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return launch_status();
}

int moe_mxfp4_route(const float* router_logits, int T, int E, int k, int32_t* topk_idx,
                    float* topk_w, int32_t* cnt, int32_t* off, int32_t* perm, int32_t* pos,
                    cudaStream_t stream) {
  if (!router_logits || !topk_idx || !topk_w || !cnt || !off || !perm || !pos)
    return MOE_ERR_INVALID_ARG;
  int rc = validate_shape(T, 128, 128, E, k);
  if (rc) return rc;
  if (T == 0) return MOE_OK;
  DeviceState* d = nullptr;
  if ((rc = device_state(&d))) return rc;
  const Layout L = layout_for(T, 128, 128, E, k, MOE_ACT_MXFP8);
  void* ws = nullptr;
  if ((rc = cached_workspace(d, L.total, &ws))) return rc;
  Work w = carve(ws, L);
  w.topk_idx = topk_idx;
  w.topk_w = topk_w;
  w.cnt = cnt;
  w.off = off;
  w.perm = perm;
  w.pos = pos;
  Steps st{nullptr, stream};
  // the kernels the forward runs for this T
  if (T <= kSmallRouteTokens) {
    if ((rc = enqueue_route_act_small(router_logits, true, MOE_ACT_MXFP8, nullptr, T, 128, E, k,
                                      kChunkNarrow, w, d, stream, st)))
      return rc;
    return launch_status();
  }
  return enqueue_route(router_logits, true, T, E, k, kChunkNarrow, w, d, stream, st);
}

int moe_mxfp8_quantize_rows(const void* x_bf16, int64_t rows, int64_t K, uint8_t* codes,
                            uint8_t* scales, cudaStream_t stream) {
  if (!x_bf16 || !codes || !scales || rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x_bf16, 16) || !aligned(codes, 16)) return MOE_ERR_ALIGNMENT;
  if (rows == 0) return MOE_OK;
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  mxfp8_rows_kernel<<<grid_for(rows * ((K / 32 + 31) / 32), 8, d->sms * 8), 256, 0, stream>>>(
      static_cast<const uint16_t*>(x_bf16), nullptr, rows, K, rows, codes, scales, d->status);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return launch_status();
}

int moe_mxfp4_forward_routed(const void* x_bf16, const void* w_router_bf16,
                             const uint8_t* w13_fp4, const uint8_t* w13_e8m0,
                             const uint8_t* w2_fp4, const uint8_t* w2_e8m0, int T, int H, int I,
                             int E, int k, void* y_bf16, cudaStream_t stream,
                             const moe_opts* opts) {
  if (!w_router_bf16) return MOE_ERR_INVALID_ARG;
  return forward_impl(x_bf16, nullptr, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H, I, E, k, y_bf16,
                      stream, opts, w_router_bf16);
}

size_t moe_mxfp4_workspace_size_routed(int T, int H, int I, int E, int k, int act_mode) {
  if (validate_shape(T, H, I, E, k) != MOE_OK) return 0;
  if (act_mode != MOE_ACT_MXFP8 && act_mode != MOE_ACT_BF16) return 0;
  return layer_bytes(T, H, I, E, k, act_mode, true);
}

int moe_router_topk(const void* x_bf16, const void* w_router_bf16, int T, int H, int E, int k,
                    float* logits_out, int32_t* topk_idx, float* topk_w, cudaStream_t stream) {
  if (!x_bf16 || !w_router_bf16 || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  int rc = validate_shape(T, H, 128, E, k);
  if (rc) return rc;
  if (H % 128) return MOE_ERR_UNSUPPORTED_SHAPE;  // the router GEMM's K tiles
  if (!aligned(x_bf16, 16) || !aligned(w_router_bf16, 16)) return MOE_ERR_ALIGNMENT;
  if (T == 0) return MOE_OK;
  DeviceState* d = nullptr;
  if ((rc = device_state(&d))) return rc;
  const size_t part_bytes = align256((size_t)router_part_bytes(T, E));
  void* ws = nullptr;
  if ((rc = cached_workspace(d, part_bytes + (size_t)T * E * 4, &ws))) return rc;
  float* part = static_cast<float*>(ws);
  float* lg = logits_out ? logits_out : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                                                   part_bytes);
  Steps st{nullptr, stream};
  return enqueue_router(x_bf16, w_router_bf16, T, H, E, part, lg, d, stream, 2000000000ull, st, k,
                        topk_idx, topk_w);
}

int mxfp8_quantize(const float* w, int64_t rows, int64_t K, uint8_t* out_e4m3, uint8_t* out_e8m0,
                   cudaStream_t stream) {
  if (!w || !out_e4m3 || !out_e8m0 || rows < 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (K % 32) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(w, 16) || !aligned(out_e4m3, 16)) return MOE_ERR_ALIGNMENT;
  if (rows == 0) return MOE_OK;
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  mxfp8_rows_f32_kernel<<<grid_for(rows, 8, d->sms * 8), 256, 0, stream>>>(w, rows, K, out_e4m3,
                                                                          out_e8m0);
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return launch_status();
}

int moe_fp8_dense_forward(const void* x_bf16, const uint8_t* w_e4m3, const uint8_t* w_e8m0,
                          int T, int K, int N, void* y_bf16, cudaStream_t stream) {
  if (!x_bf16 || !w_e4m3 || !w_e8m0 || !y_bf16 || T < 0 || K <= 0 || N <= 0)
    return MOE_ERR_INVALID_ARG;
  if (K % 128 || N % 4) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x_bf16, 16) || !aligned(w_e4m3, 16) || !aligned(w_e8m0, 16) || !aligned(y_bf16, 16))
    return MOE_ERR_ALIGNMENT;
  if (T == 0) return MOE_OK;
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  const int n_max = dense_n_for(T);
  const DensePlan P = plan_dense(N, T, K / 128, n_max, d->sms, kDensePartBytes);
  const size_t xq_bytes = align256((size_t)T * K), xs_bytes = align256((size_t)T * (K / 32));
  const size_t part_bytes = (size_t)P.k_splits * T * N * 4;
  void* ws = nullptr;
  if ((rc = cached_workspace(d, xq_bytes + xs_bytes + part_bytes, &ws))) return rc;
  uint8_t* xq = static_cast<uint8_t*>(ws);
  uint8_t* xs = xq + xq_bytes;
  float* part = reinterpret_cast<float*>(xs + xs_bytes);

  mxfp8_rows_kernel<<<grid_for((int64_t)T * ((K / 32 + 31) / 32), 8, d->sms * 8), 256, 0,
                      stream>>>(
      static_cast<const uint16_t*>(x_bf16), nullptr, T, K, T, xq, xs, d->status);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);

  DenseParams dp{};
  if ((rc = make_map(&dp.map_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, w_e4m3, K, N, K, 128, 128)) ||
      (rc = make_map(&dp.map_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, K, T, K, 128,
                     box_rows_for(T))))
    return rc;
  dp.box_rows_b = box_rows_for(T);
  dp.a_sf = w_e8m0;
  dp.b_sf = xs;
  dp.part = part;
  dp.M = N;
  dp.T = T;
  dp.m_tiles = P.m_tiles;
  dp.n_blocks = P.n_blocks;
  dp.k_splits = P.k_splits;
  dp.kb_per_split = P.kb_per_split;
  dp.kb_total = P.kb_total;
  dp.status = d->status;
  dp.timeout_ns = 2000000000ull;
  const int items = P.m_tiles * P.n_blocks * P.k_splits;
  auto go = [&](auto kernel, size_t smem) {
    return launch_pdl(kernel, dim3(std::min(items, d->sms)), dim3(kDenseThreads), smem, stream,
                      dp);
  };
  const cudaError_t e =
      n_max == kDenseNSmall
          ? go(dense_tc_kernel<kDenseMxf8, kDenseNSmall>, DenseCfg<kDenseMxf8, kDenseNSmall>::kSmem)
          : go(dense_tc_kernel<kDenseMxf8, kDenseNMax>, DenseCfg<kDenseMxf8, kDenseNMax>::kSmem);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (launch_pdl(splitk_reduce_bf16_kernel, dim3(grid_for((int64_t)T * N / 4, 256, d->sms * 8)),
                 dim3(256), 0, stream, (const float*)part, P.k_splits, T, N,
                 static_cast<uint16_t*>(y_bf16)) != cudaSuccess)
    return MOE_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_verify_block(const float* p, const float* q, const int32_t* draft, const float* u,
                     const uint64_t* U, int S, int g, int64_t V, int32_t* n_acc, int32_t* tokens,
                     cudaStream_t stream) {
  if (!p || !q || !draft || !u || !U || !n_acc || !tokens) return MOE_ERR_INVALID_ARG;
  if (S < 0 || g < 1 || g > MOE_VERIFY_MAX_DRAFT || V < 1 || V > INT32_MAX)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(p, 4) || !aligned(q, 4) || !aligned(draft, 4) || !aligned(u, 4) ||
      !aligned(U, 8) || !aligned(n_acc, 4) || !aligned(tokens, 4))
    return MOE_ERR_ALIGNMENT;
  if (S == 0) return MOE_OK;
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  if (V > (int64_t)kVerifyMaxChunks * kVerifyRange) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int chunks = (int)((V + kVerifyRange - 1) / kVerifyRange);
  const size_t part_bytes = align256((size_t)S * chunks * 8);
  const size_t count_bytes = align256((size_t)S * 4);
  void* ws = nullptr;
  if ((rc = cached_workspace(d, part_bytes + count_bytes + (size_t)S * 4, &ws))) return rc;
  VerifyParams P{};
  P.p = p;
  P.q = q;
  P.draft = draft;
  P.u = u;
  P.U = U;
  P.S = S;
  P.g = g;
  P.V = V;
  P.chunks = chunks;
  P.chunk_len = kVerifyRange;
  P.part = static_cast<uint64_t*>(ws);
  P.count = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + part_bytes);
  int32_t* jpos = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + part_bytes + count_bytes);
  P.n_acc = n_acc;
  P.tokens = tokens;
  P.status = d->status;
  verify_decide_kernel<<<(S + 7) / 8, 256, 0, stream>>>(P, jpos);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (launch_pdl(verify_draw_kernel, dim3(S * chunks), dim3(kVerifyDrawThreads), 0, stream, P,
                 (const int32_t*)jpos) != cudaSuccess)
    return MOE_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return launch_status();
}

int moe_mxfp4_get_status(cudaStream_t stream) {
  DeviceState* d = nullptr;
  int rc = device_state(&d);
  if (rc) return rc;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int zero = 0;
  if (v != 0 && cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return MOE_ERR_CUDA;
  return v;
}

uint64_t moe_mxfp4_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

uint64_t moe_mxfp4_alloc_count(void) { return g_allocs.load(std::memory_order_relaxed); }

int moe_mxfp4_workspace_layout(int T, int H, int I, int E, int k, int act_mode,
                               moe_workspace_layout* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  int rc = validate_shape(T, H, I, E, k);
  if (rc) return rc;
  if (act_mode != MOE_ACT_MXFP8 && act_mode != MOE_ACT_BF16) return MOE_ERR_INVALID_ARG;
  // a padded layer's routing arrays and buffers are those of the padded shape
  const Layout L = layout_for(T, round128(H), round128(I), E, k, act_mode);
  *out = public_layout(L, 0, 0);
  out->total = layer_bytes(T, H, I, E, k, act_mode, false);
  return MOE_OK;
}

int moe_mxfp4_workspace_layout_routed(int T, int H, int I, int E, int k, int act_mode,
                                      moe_workspace_layout* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  int rc = validate_shape(T, H, I, E, k);
  if (rc) return rc;
  if (act_mode != MOE_ACT_MXFP8 && act_mode != MOE_ACT_BF16) return MOE_ERR_INVALID_ARG;
  // a padded layer's routing arrays and buffers are those of the padded shape
  const Layout L = layout_for(T, round128(H), round128(I), E, k, act_mode, true);
  *out = public_layout(L, 0, 0);
  out->total = layer_bytes(T, H, I, E, k, act_mode, true);
  return MOE_OK;
}

int moe_mxfp4_workspace_layout_chain(int n_layers, int layer, int T, int H, int I, int E, int k,
                                     int act_mode, moe_workspace_layout* out) {
  if (!out || n_layers < 1 || n_layers > MOE_MAX_CHAIN || layer < 0 || layer >= n_layers)
    return MOE_ERR_INVALID_ARG;
  int rc = validate_shape(T, H, I, E, k);
  if (rc) return rc;
  if (act_mode != MOE_ACT_MXFP8 && act_mode != MOE_ACT_BF16) return MOE_ERR_INVALID_ARG;
  if (!tc_widths(H, I)) return MOE_ERR_UNSUPPORTED_SHAPE;
  const ChainLayout C = chain_layout(n_layers, T, H, I, E, k, act_mode);
  *out = public_layout(C.base, (size_t)layer * C.route_block, C.act_shift);
  out->x_stream[0] = C.xb[0];
  out->x_stream[1] = C.xb[1];
  out->total = C.total;
  return MOE_OK;
}

// ---------------------------------------------------------------- no-alloc entry point
//
// Scratch for moe_mxfp4_forward_noalloc: a fixed-size array in the module's
// global memory, created on every device that loads the library and kept
// until the process exits.  Host code must not pass g_noalloc_scratch itself
// to a kernel (in host code the name is a host-side stand-in, not a device
// address); the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

namespace moe {
namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices];

// device address of g_noalloc_scratch on the current device (looked up once
// per device, with that device current)
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}
}  // namespace
}  // namespace moe

int moe_mxfp4_forward_noalloc(const void* x_bf16, const float* router_logits,
                              const uint8_t* w13_fp4, const uint8_t* w13_e8m0,
                              const uint8_t* w2_fp4, const uint8_t* w2_e8m0, int T, int H, int I,
                              int E, int k, void* y_bf16, cudaStream_t stream) {
  // argument errors first, in moe_mxfp4_forward's order (pointers, shape,
  // alignment), then the scratch size
  if (!x_bf16 || !router_logits || !w13_fp4 || !w13_e8m0 || !w2_fp4 || !w2_e8m0 || !y_bf16)
    return MOE_ERR_INVALID_ARG;
  int rc = validate_shape(T, H, I, E, k);
  if (rc) return rc;
  if (!aligned(w13_fp4, 16) || !aligned(w2_fp4, 16) || !aligned(x_bf16, 16) ||
      !aligned(router_logits, 16) || !aligned(w13_e8m0, 16) || !aligned(w2_e8m0, 16) ||
      !aligned(y_bf16, 16))
    return MOE_ERR_ALIGNMENT;
  const bool padded = !tc_widths(H, I) || !aligned(w13_fp4, 32) || !aligned(w2_fp4, 32);
  if ((padded ? pad_layout(T, H, I, E, k, MOE_ACT_MXFP8, false).total
              : layout_for(T, H, I, E, k, MOE_ACT_MXFP8).total) >
      (size_t)MOE_NOALLOC_SCRATCH_BYTES)
    return MOE_ERR_NO_MEMORY;  // needs more scratch than the static array holds
  if (T == 0) return forward_impl(x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H,
                                  I, E, k, y_bf16, stream, nullptr);
  DeviceState* d = nullptr;
  if ((rc = device_state(&d))) return rc;
  void* scratch = nullptr;
  if ((rc = noalloc_scratch(&scratch))) return rc;
  moe_opts o{};
  o.act_mode = MOE_ACT_MXFP8;
  o.path = MOE_PATH_AUTO;
  o.workspace = scratch;
  o.workspace_bytes = MOE_NOALLOC_SCRATCH_BYTES;
  return forward_impl(x_bf16, router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0, T, H, I, E, k,
                      y_bf16, stream, &o);
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_NO_MEMORY: return "MOE_ERR_NO_MEMORY";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_DEVICE_FAULT: return "MOE_ERR_DEVICE_FAULT";
    case MOE_ERR_NO_DEVICE: return "MOE_ERR_NO_DEVICE";
    default: return "MOE_ERR_UNKNOWN";
  }
}

}  // extern "C"
