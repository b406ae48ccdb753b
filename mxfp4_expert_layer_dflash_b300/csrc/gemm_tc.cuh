// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05), MXFP8 mode.
//
// Swap-AB: the expert's weight rows fill the 128-row MMA dimension (A) and the
// expert's tokens (a chunk of slots, padded to 16) are N, so the tiny
// decode-time token count never pads the weight side.  A is FP4 (E2M1)
// straight from HBM: TMA's 16U4_ALIGN16B mode expands each 16-element group
// into the 16-byte-aligned form the MMA reads, so no thread touches the
// weights.  B is the MXFP8-E4M3 activation tile.  The E8M0 scales of both
// operands are written into TMEM by a scale warpgroup and applied by the MMA
// per 32 elements (kind::mxf8f6f4, block_scale).  Decode is bound by weight
// bandwidth (ai.appwright.xyz, "第1層"); the pipeline keeps several weight
// tiles in flight per SM while the tensor cores work on earlier ones (the
// load/compute overlap of dothoosh.com, "TileRT").
//
// One kernel body runs one or two phases:
//   phase GEMM1: z = W13_e x, h = silu(gate) * up, MXFP8-requantised into
//                hq/hs (gate rows [r, r+128) paired with up rows [I+r, I+r+128),
//                so the epilogue has both operands for the same row and token);
//   phase GEMM2: yp = W2_e h (fp32), output rows [r, r+128) paired with
//                [r+128, r+256).
// The multi-kernel path launches it once per phase; the persistent path runs
// both phases in one launch (the single resident engine kernel of dothoosh.com,
// "TileRT", for this layer): every CTA walks its GEMM1 items, then its GEMM2
// items, and a GEMM2 item waits (bounded) until all GEMM1 items of its token
// chunk have published h.  Each CTA finishes its GEMM1 items before any GEMM2
// item and the launch is cooperative (all CTAs resident), so every wait is on
// work that is running.
// Two weight boxes per pipeline round keep the fixed cost of a round small
// against the bytes it moves.
//
// Warp roles (384 threads, one CTA per SM, persistent over work items):
//   warp 0      TMA producer (weight tiles + activation tile): the warp walks
//               the fills convergently, one elected lane issues each copy
//   warp 2      TMEM owner and MMA issuer, convergent like the producer (a
//               single lane in a divergent branch issues MMAs far slower)
//   warps 4-7   scale stagers: warp w owns TMEM lanes 32*(w%4).. and writes the
//               E8M0 words of each stage there with tcgen05.st, loading them
//               from global memory four to eight stages ahead into registers
//   warps 8-11  epilogue: TMEM -> registers -> SwiGLU + MXFP8 requant, or fp32
// Work item = (chunk of one expert's slots, one pair of weight tiles).
//
// Scale placement in TMEM (checked on the device by a layout probe): the MMA
// reads the A scale of row m from lane m, column sfa + m/32, and the B scale
// of token n from lane 32q + n%32 of every lane quarter q, column sfb + n/32;
// the byte inside the 32-bit word is the instruction descriptor's scale id
// (one per 32-element block of the 128-element stage).
#pragma once

#include <cuda.h>

#include <climits>

#include "combine.cuh"
#include "common.cuh"
#include "fmt.cuh"
#include "grid_sync.cuh"
#include "ptx.cuh"
#include "route_layer.cuh"

namespace moe {

constexpr int kTcThreads = 384;
constexpr int kBlockK = 128;   // K elements per stage: one TMA box of FP4
constexpr int kBoxRowsB = 16;  // activation rows per TMA box
constexpr int kSfGroup = 4;    // fills per scale load group (16 bytes of scales per row)

struct TcPhase {
  CUtensorMap map_w;  // FP4 weights [E*R rows, K], 16U4_ALIGN16B, box {128, 128}, SW128
  CUtensorMap map_x;  // E4M3 activations [T*k rows, K], u8, box {128, 16}, SW128
  const uint8_t* w_sf;  // [E*R, K/32]
  const uint8_t* x_sf;  // [T*k, K/32]
  int K;           // reduction length
  int R;           // weight rows per expert (2I or H)
  int m_tiles;     // tile pairs per expert (I/128 for GEMM1, ceil(H/256) for GEMM2)
  int m_stride;    // weight rows between consecutive tile pairs (128 or 256)
  int half;        // row offset of the second tile of a pair (I or 128)
  int out_dim;     // row length of the output (I or H)
  int rows_total;  // E * R: weight rows in the tensor (guards an odd last tile pair)
  int dep_target;  // (GEMM2 of a persistent launch) GEMM1 publications per chunk to wait
                   // for: 4 epilogue warps x tile pairs
};

// A chain of layers: the next layer's GEMM1, whose first weight tiles the
// last GEMM launch of a layer prefetches into L2 once its own copies are
// issued — the weight stream continues while the layer's tail, the hand-off
// kernel and the next launch run (the pipeline kept in flight across
// operators: dothoosh.com, section "TileRT").
struct NextGemm1 {
  CUtensorMap map_w;    // the next layer's w13, as TcPhase::map_w
  const int4* chunks;   // the next layer's chunk list (routed before this launch)
  const int32_t* meta;
  int R, m_tiles, m_stride, half;
  int stages;           // K steps of the CTA's first next-layer item to prefetch (0: off)
};

struct TcParams {
  TcPhase ph[2];  // [0] = the launch's (first) GEMM, [1] = GEMM2 of a persistent launch
  const int4* chunks;
  const int32_t* meta;  // meta[0] = chunk count
  uint8_t* hq;          // [T*k, I] E4M3
  uint8_t* hs;          // [T*k, I/32]
  float* yp;            // [T*k, H]
  int* gemm1_done;      // [chunks] GEMM1 epilogue-warp publications per chunk (persistent path)
  int early_chunks;     // the chunk list was final before the preceding kernel ran: the
                        // producer may read it, and issue weight tiles, before the wait
  int* status;
  unsigned long long timeout_ns;
  NextGemm1 next;       // next.stages == 0 unless this is a chained layer's last GEMM launch
  // ---- the whole-layer launch (kModeLayer): GEMM1, GEMM2 and the combine,
  // and for T <= 32 also the routing and the activation step
  LayerRouteParams route;  // route.T > 0: steps a1-a4 run inside the launch
  GridSync sync;           // grid-wide barriers (act1 rows written; GEMM2 outputs written)
  const int32_t* pos;      // routing done before the launch: [T*k] slots
  const float* gate;       // [T*k] gates
  uint16_t* y;             // [T, H] bf16 output of the combine
  int T, H, k;
};

template <int kNMax>
struct TcCfg {
  static constexpr int kA = 2;                 // A tiles per stage
  static constexpr int kATile = 128 * 128;     // unpacked FP4 tile bytes
  static constexpr int kBTile = kNMax * 128;
  static constexpr int kStageBytes = kA * kATile + kBTile;  // multiple of 1024
  static constexpr int kStages = (232448 - 1024 - 256) / kStageBytes;
  static constexpr int kAccCols = kA * kNMax;  // one accumulator buffer (gate|up or lo|hi)
  static constexpr int kSfStride = 16;         // TMEM columns per stage of scales
  // accumulators are double-buffered when TMEM has room for two
  static constexpr int kAccBufs = 2 * kAccCols + kStages * kSfStride <= 512 ? 2 : 1;
  static constexpr int kSfBase = kAccBufs * kAccCols;   // TMEM column of stage 0's scales
  static constexpr int kSfbCol = 4 * kA;       // B scales after the A scale columns
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kTxA = 128 * 64;   // packed bytes of one weight box
  static constexpr int kWords = kA + kNMax / 32;  // scale words per lane per stage
  static constexpr int kBarBytes = 256;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kBarBytes;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kNMax % 32 == 0 && kNMax <= 128, "B-scale columns per stage");
  static_assert(kSfBase + kStages * kSfStride <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

// Kernel modes: one GEMM per launch, both GEMMs in one persistent launch, or
// whole layers in one persistent launch (both GEMMs, then the combine; with
// the routing and the activation step in front for a single layer of T <= 32
// tokens, and between layers for a chain).
constexpr int kModeGemm1 = 0, kModeGemm2 = 1, kModeBoth = 2, kModeLayer = 3;

// One layer of a chained launch: its weights, its routing (done before the
// launch), and where its combine reads the residual and writes its output.
struct ChainLayer {
  CUtensorMap map_w[2];      // w13 (GEMM1), w2 (GEMM2); as TcPhase::map_w
  const uint8_t* w_sf[2];    // their E8M0 scales
  const int4* chunks;        // the layer's chunk list
  const int32_t* meta;       // meta[0] = chunk count
  const int32_t* pos;        // [T*k] slots
  const float* gate;         // [T*k] gates
  const uint16_t* x_res;     // [T, H] residual added to the layer's sum, or null
  uint16_t* x_out;           // [T, H] the layer's bf16 output, or null
  const int32_t* pos_next;   // the next layer's slots (the combine writes its act1 rows), or null
};

// A chain of up to kMaxLaunchLayers layers in one launch: the shared
// parameters (shapes, activation tensor maps, scratch, barrier words) and the
// layers.
struct ChainParams {
  TcParams p;
  ChainLayer lay[kMaxLaunchLayers];
  int n_layers;
};

// shared memory of a launch in mode kMode: the whole-layer launch with
// narrow chunks also keeps its own routing (LayerRouteState)
template <int kNMax, int kMode>
constexpr size_t tc_smem_bytes() {
  return TcCfg<kNMax>::kSmem +
         (kMode == kModeLayer && kNMax == kChunkNarrow ? sizeof(LayerRouteState) : 0);
}

// position of a work item in a launch's sequence (layer, item): published by
// the producer, compared by the scale stagers; increases along the sequence
__device__ __forceinline__ int item_seq(int layer, int item) { return (layer << 20) | item; }

// Walks the (layer, work item, k-stage) sequence of one CTA over all phases
// (kPhases is 1 for single-GEMM launches, so the phase folds to a constant).
// `span`: continue into the next layers after one's items end (else stop).
template <int kPhases>
struct FillCursor {
  // per-launch constants, copied once (no parameter-space reads per item)
  const int4* chunks;
  const uint32_t* packed;  // the chunk list in shared memory (whole-layer launch), or null
  const ChainLayer* lay;   // chained layers, or null
  int n_layers, layer_end;
  int step, first, n0, ntot;  // n0: items of phase 0; ntot: items of all phases (this layer)
  int mtl[2], kst[2];      // tile pairs per chunk and k-stages per item, per phase
  int packed_chunks;       // chunk count of the packed list
  // position
  int layer, item, ks, phase, mt, ksteps, chunk;
  int4 ch;
  __device__ __forceinline__ void start(const TcParams& p, const ChainLayer* ly, int nl,
                                        const uint32_t* pk, int pk_chunks, int first_item,
                                        int stp, int layer0, bool span) {
    lay = ly;
    n_layers = nl;
    layer_end = span ? nl : layer0 + 1;
    packed = pk;
    packed_chunks = pk_chunks;
    step = stp;
    first = first_item;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mtl[i] = p.ph[i < kPhases ? i : 0].m_tiles;
      kst[i] = p.ph[i < kPhases ? i : 0].K / kBlockK;
    }
    chunks = p.chunks;
    layer = layer0;
    begin_layer(p.meta);
  }
  // items of the current layer; moves on past layers with none for this CTA
  __device__ __forceinline__ void begin_layer(const int32_t* meta0) {
    while (true) {
      int nch;
      if (packed) {
        nch = packed_chunks;
      } else if (lay) {
        chunks = lay[layer].chunks;
        nch = lay[layer].meta[0];
      } else {
        nch = meta0[0];
      }
      n0 = nch * mtl[0];
      ntot = n0 + (kPhases > 1 ? nch * mtl[1] : 0);
      item = first;
      ks = 0;
      phase = 0;
      mt = 0;
      ksteps = 1;
      chunk = 0;
      ch = make_int4(0, 0, 0, 0);
      if (item < ntot || layer + 1 >= layer_end) break;
      ++layer;
    }
    load();
  }
  __device__ __forceinline__ bool valid() const { return layer < layer_end && item < ntot; }
  __device__ __forceinline__ int seq() const { return item_seq(layer, item); }
  __device__ __forceinline__ void load() {
    if (item < ntot) {
      phase = (kPhases > 1 && item >= n0) ? 1 : 0;
      const int local = item - (phase ? n0 : 0);
      const int m = phase ? mtl[1] : mtl[0];
      chunk = local / m;
      mt = local % m;
      ch = packed ? unpack_chunk(packed[chunk]) : chunks[chunk];
      ksteps = phase ? kst[1] : kst[0];
    }
  }
  __device__ __forceinline__ void next() {
    if (++ks == ksteps) next_item();
  }
  __device__ __forceinline__ void next_item() {
    ks = 0;
    item += step;
    if (item >= ntot && layer + 1 < layer_end) {
      ++layer;
      begin_layer(nullptr);
    } else {
      load();
    }
  }
};

__device__ __forceinline__ int ld_acquire(const int* ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(int* ptr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_relaxed(const int* ptr) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void st_release_cta(int* ptr, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(ptx::smem_u32(ptr)), "r"(v)
               : "memory");
}

__device__ __forceinline__ int ld_acquire_cta(const int* ptr) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(ptx::smem_u32(ptr))
               : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// bounded wait until GEMM1 has published every tile pair of `chunk`
// (whole-layer launch: `tag` != 0, also gives up when another CTA has)
__device__ __forceinline__ bool wait_chunk_ready(const TcParams& p, int chunk, int target,
                                                 unsigned long long timeout_ns,
                                                 const volatile int* abort, uint64_t tag = 0) {
  const uint64_t deadline = ptx::globaltimer() + timeout_ns;
  uint32_t spins = 0;
  while (ld_acquire(p.gemm1_done + chunk) < target) {
    if (*abort || ptx::globaltimer() > deadline) return false;
    if (tag && (++spins & 15u) == 0 && grid_aborted(p.sync, tag)) return false;
  }
  return true;
}

// L2 priority of a weight tile copy.  Phase 0 of a launch (GEMM1 of the
// both-GEMMs launch; the one GEMM of either launch of the two-launch path)
// takes the normal class: when an expert's tokens fill several chunks, its
// tiles are read once per chunk, and evict-first lines tend to be gone by the
// second read (measured: the 256- and 1024-token layers ran about 1% faster,
// the 1024-token one 1% slower again with GEMM2's launch back at evict-first).
// GEMM2 of the both-GEMMs launch keeps evict-first.
__device__ __forceinline__ uint64_t weight_policy(int phase) {
  return phase == 0 ? ptx::policy_evict_normal() : ptx::policy_evict_first();
}

// The kernel body of every mode.  `lay`/`n_layers`: the layers of a chained
// whole-layer launch (lay null: one layer, described by p itself).
template <int kNMax, int kMode>
__device__ __forceinline__ void gemm_tc_body(const TcParams& p, const ChainLayer* lay,
                                             int n_layers) {
  using C = TcCfg<kNMax>;
  constexpr bool kLayer = kMode == kModeLayer;
  constexpr int kPhases = (kMode == kModeBoth || kLayer) ? 2 : 1;
  using Cursor = FillCursor<kPhases>;
  // whole-layer launch of one layer that also routes (T <= 32; narrow chunks)
  const bool route_in = kLayer && !lay && kNMax == kChunkNarrow && p.route.T > 0;
  // is this phase the SwiGLU GEMM1 / one whose inputs this launch writes?
  // GEMM2 reads GEMM1's h; in a chained launch, GEMM1 of every layer after the
  // first reads the act1 rows the previous layer's combine writes
  auto gated_phase = [](int phase) { return kMode == kModeGemm1 || (kPhases == 2 && phase == 0); };
  auto dep_phase = [&](int phase, int layer) {
    return kPhases == 2 && (phase == 1 || (lay != nullptr && layer > 0));
  };
  // are this phase's activation scales written during the launch (so they
  // need coherent loads)?  GEMM2's h; GEMM1's act1 rows when the launch writes them
  auto coherent_x = [&](int phase, int layer) { return dep_phase(phase, layer) || route_in; };
  // per-layer weights
  auto map_w = [&](int phase, int layer) -> const CUtensorMap* {
    return lay ? &lay[layer].map_w[phase] : &p.ph[phase].map_w;
  };
  auto w_sf = [&](int phase, int layer) -> const uint8_t* {
    return lay ? lay[layer].w_sf[phase] : p.ph[phase].w_sf;
  };
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // single-launch paths: the last work item (item_seq) whose inputs the
  // producer has seen published (a CTA's items only move forward); the scale
  // stagers read it instead of polling the global flags themselves
  int* dep_ready = reinterpret_cast<int*>(tmem_slot + 2);
  // whole-layer launch: the aux warps' agreed outcome of a barrier
  volatile int* aux_go = reinterpret_cast<volatile int*>(tmem_slot + 3);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1 + 4);  // TMA arrive.expect_tx + one arrival per scale warp
      ptx::mbar_init(&empty[s], 1);     // MMA commit
    }
    for (int b = 0; b < 2; ++b) {       // (only C::kAccBufs of the two are used)
      ptx::mbar_init(&acc_full[b], 1);   // MMA commit
      ptx::mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    *dep_ready = -1;
    *aux_go = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 2) {
    ptx::tmem_alloc(tmem_slot, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    for (int ph = 0; ph < kPhases; ++ph) {
      ptx::prefetch_tmap(map_w(ph, 0));
      ptx::prefetch_tmap(&p.ph[ph].map_x);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // Programmatic launch: the preceding kernel may still run.  Its outputs (the
  // activation tiles and scales, h for GEMM2) are read only after the wait
  // below; but in a single-GEMM launch with narrow chunks whose routing
  // finished before that kernel started (early_chunks: the preceding kernel is
  // the activation step or a chain's combine, or GEMM1 for GEMM2), the chunk
  // list is final, and the weights are inputs, so the producer already issues
  // the weight tiles of its first fills (each
  // stage's barrier expects both operands' bytes; the activation tiles follow
  // after the wait) — the weight stream starts while the preceding kernel
  // finishes, on the SMs it has left.
  uint32_t prefilled = 0;  // (producer) fills whose weight tiles are in flight
  if ((kMode == kModeGemm1 || kMode == kModeGemm2) && kNMax == kChunkNarrow && p.early_chunks &&
      warp == 0) {
    const int nch = p.meta[0];
    const int items0 = nch * p.ph[0].m_tiles;
    const int items_all = items0 + (kPhases > 1 ? nch * p.ph[kPhases - 1].m_tiles : 0);
    int it = blockIdx.x, ks = 0;
    while (prefilled < (uint32_t)C::kStages && it < items_all) {
      const int phase = (kPhases > 1 && it >= items0) ? 1 : 0;
      const TcPhase& ph = p.ph[phase];
      const int local = it - (phase ? items0 : 0);
      const int chunk = local / ph.m_tiles;
      const int4 ch = p.chunks[chunk];
      const int row0 = ch.x * ph.R + (local - chunk * ph.m_tiles) * ph.m_stride;
      const uint32_t tx = C::kA * C::kTxA + (uint32_t)((ch.z + 15) & ~15) * 128;
      uint8_t* st = smem + prefilled * C::kStageBytes;  // first use of every stage: free
      ptx::mbar_arrive_expect_tx_warp(&full[prefilled], tx);
      const uint64_t pol_w0 = weight_policy(phase);
      ptx::tma_load_2d_warp(st, map_w(phase, 0), &full[prefilled], ks * kBlockK, row0, pol_w0);
      ptx::tma_load_2d_warp(st + C::kATile, map_w(phase, 0), &full[prefilled], ks * kBlockK,
                            row0 + ph.half, pol_w0);
      ++prefilled;
      if (++ks == ph.K / kBlockK) {
        ks = 0;
        it += gridDim.x;
      }
    }
  }
  grid_dependency_wait();

  // whole-layer launch: this call's barrier tag, and for T <= 32 the routing
  // of the block, done by every CTA in its own shared memory (the stage
  // buffers serve as scratch before the first copy lands in them)
  LayerRouteState* rs =
      reinterpret_cast<LayerRouteState*>(smem + C::kStages * C::kStageBytes + C::kBarBytes);
  // step a4 reads token rows of x soon, while every CTA's first weight tiles
  // flood the memory system: CTA t brings row t into L2 now
  if (route_in && warp == 1 && lane == 0 && (int)blockIdx.x < p.route.T)
    ptx::bulk_prefetch_l2(p.route.x + (int64_t)blockIdx.x * p.ph[0].K,
                          (uint32_t)p.ph[0].K * 2u);
  const uint64_t tag = kLayer ? grid_sync_tag(p.sync) : 0;
  // the value a published (chunk, GEMM1 tile pair) flag of layer l holds in
  // this call (a kind never written when the debug flag forces the wait to
  // run out)
  auto flag_want = [&](int layer) {
    return tag | (p.ph[1].dep_target == INT_MAX ? kChunkFlagNever
                                                : kChunkFlagKind + (uint64_t)layer);
  };
  auto fail = [&](int code) {
    set_status(p.status, code);
    *abort_flag = 1;
    if (kLayer) grid_give_up(p.sync, tag);
  };
  if (route_in && p.route.w_router) {
    // the router in front: this CTA computes its experts' logits for the
    // block (the stage buffers as scratch), then every CTA waits for every
    // expert's (one barrier)
    layer_router_logits(p.route, p.ph[0].K, const_cast<float*>(p.route.logits),
                        reinterpret_cast<float*>(smem));
    if (threadIdx.x == 0) grid_arrive(p.sync, kSyncLogits, tag | kLogitsKind);
    if (warp == 0 &&
        !grid_wait(p.sync, kSyncLogits, tag | kLogitsKind, tag, p.timeout_ns, abort_flag) &&
        lane == 0)
      fail(kStatusTimeout);
    __syncthreads();
  }
  if (route_in) {
    layer_route_block(p.route, smem, rs, blockIdx.x == 0, p.status);
    ptx::fence_proxy_async_smem();  // generic scratch writes before TMA writes the stages
    __syncthreads();
  }
  const uint32_t* s_chunks = route_in ? rs->chunks : nullptr;
  const int s_nchunks = route_in ? rs->n_chunks : 0;
  // chunk i of layer l, and the layer's chunk count
  auto chunk_at = [&](int layer, int i) {
    return s_chunks ? unpack_chunk(s_chunks[i]) : lay ? lay[layer].chunks[i] : p.chunks[i];
  };
  auto n_chunks_of = [&](int layer) {
    return s_chunks ? s_nchunks : lay ? lay[layer].meta[0] : p.meta[0];
  };
  const int m1 = p.ph[0].m_tiles, m2 = kPhases > 1 ? p.ph[1].m_tiles : 0;

  // With the routing inside the launch: the producer first issues the weight
  // tiles of its first fills (each stage's barrier expects both operands'
  // bytes; the activation tiles follow once they exist), then every warp of
  // the CTA runs step a4 for the chunks of the CTA's GEMM1 items — a warp per
  // (slot row, run of 32 blocks of 32), two units' loads in flight — while
  // those tiles stream in.  Other CTAs multiplying the same chunk write the
  // same bytes, so only this CTA's own writes must precede its copies.
  if (route_in) {
    const int items0 = s_nchunks * m1, items_all = items0 + s_nchunks * m2;
    if (warp == 0) {
      int it = blockIdx.x, ks = 0;
      while (prefilled < (uint32_t)C::kStages && it < items_all) {
        const int phase = (kPhases > 1 && it >= items0) ? 1 : 0;
        const TcPhase& ph = p.ph[phase];
        const int local = it - (phase ? items0 : 0);
        const int chunk = local / ph.m_tiles;
        const int4 ch = chunk_at(0, chunk);
        const int row0 = ch.x * ph.R + (local - chunk * ph.m_tiles) * ph.m_stride;
        const uint32_t tx = C::kA * C::kTxA + (uint32_t)((ch.z + 15) & ~15) * 128;
        uint8_t* st = smem + prefilled * C::kStageBytes;  // first use of every stage: free
        ptx::mbar_arrive_expect_tx_warp(&full[prefilled], tx);
        const uint64_t pol_w0 = weight_policy(phase);
        ptx::tma_load_2d_warp(st, map_w(phase, 0), &full[prefilled], ks * kBlockK, row0, pol_w0);
        ptx::tma_load_2d_warp(st + C::kATile, map_w(phase, 0), &full[prefilled], ks * kBlockK,
                              row0 + ph.half, pol_w0);
        ++prefilled;
        if (++ks == ph.K / kBlockK) {
          ks = 0;
          it += gridDim.x;
        }
      }
    }
    const int64_t H = p.ph[0].K;
    const int segs = (int)((H / 32 + 31) / 32);
    constexpr int kWarps = kTcThreads / 32;
    int held_t = -1, held_slot = 0, held_sg = 0;
    uint4 held[4];
    auto load_unit = [&](int t, int sg, uint4 (&raw)[4]) {
      const int64_t b = (int64_t)sg * 32 + lane;
      if (b < H / 32) {
        const uint4* src = reinterpret_cast<const uint4*>(p.route.x + (int64_t)t * H + b * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) raw[i] = src[i];
      }
    };
    auto finish_unit = [&](int slot, int sg, const uint4 (&raw)[4]) {
      const int64_t b = (int64_t)sg * 32 + lane;
      if (b >= H / 32) return;
      float v[32];
      uint8_t c[32];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t wd[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * i + 2 * j] = __uint_as_float(wd[j] << 16);
          v[8 * i + 2 * j + 1] = __uint_as_float(wd[j] & 0xFFFF0000u);
        }
      }
      const int code = mxfp8_block(v, c);
      store_u8x32(p.route.xq + (int64_t)slot * H + b * 32, c);
      p.route.xs[(int64_t)slot * (H / 32) + b] = (uint8_t)code;
    };
    int u = 0;  // unit counter over this CTA's rows, dealt round-robin to the warps
    for (int item = blockIdx.x; item < items0; item += gridDim.x) {
      const int4 ch = chunk_at(0, item / m1);
      for (int r = 0; r < ch.z; ++r) {
        for (int sg = 0; sg < segs; ++sg, ++u) {
          if (u % kWarps != warp) continue;
          uint4 raw[4];
          load_unit(rs->perm[ch.y + r], sg, raw);
          if (held_t >= 0) finish_unit(held_slot, held_sg, held);
          held_t = 1;
          held_slot = ch.y + r;
          held_sg = sg;
#pragma unroll
          for (int i = 0; i < 4; ++i) held[i] = raw[i];
        }
      }
    }
    if (held_t >= 0) finish_unit(held_slot, held_sg, held);
    fence_proxy_async_global();  // generic writes before this CTA's TMA reads them
    __syncthreads();
  }
  auto deadline = [&]() { return ptx::globaltimer() + p.timeout_ns; };

  // Bounded wait whose outcome is the same in every lane of the warp: lanes can
  // see a timeout or the abort flag at different moments, and the warp-wide
  // tcgen05 / shuffle instructions after a wait need the whole warp.
  auto wait_all = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, deadline(), abort_flag));
  };

  // ---- whole-layer launch: work of the aux warps (1, 3 and the epilogue
  // warps; 192 threads, named barriers 1-3) after each layer's GEMM items
  constexpr int kAuxWarps = 6, kAuxThreads = kAuxWarps * 32;
  const int aux_w = warp == 1 ? 0 : warp == 3 ? 1 : warp - 6;  // valid for aux warps
  // Step a8 of layer l once every CTA's GEMM2 outputs of it are written: the
  // gate-weighted sum of each token's k slot rows in slot order (the combine
  // kernels' arithmetic), plus, in a chain, the residual, the layer's bf16
  // output and the next layer's act1 rows; then, in a chain, the arrival at
  // the next layer's act1 barrier.
  auto aux_combine = [&](int l) {
    named_barrier_sync(2, kAuxThreads);  // this CTA's epilogue stores are done
    const uint64_t out_v = tag | (kOutKind + (uint64_t)l);
    if (aux_w == 0) {
      if (lane == 0) grid_arrive(p.sync, kSyncOut + (l & 1), out_v);
      __syncwarp();
      const bool ok = grid_wait(p.sync, kSyncOut + (l & 1), out_v, tag, p.timeout_ns, abort_flag);
      if (lane == 0) {
        if (!ok) fail(kStatusTimeout);
        else if (blockIdx.x == 0 && l == n_layers - 1)
          grid_sync_retire(p.sync, tag);  // every CTA has read the counter by now
        *aux_go = ok ? 1 : 0;
      }
    }
    named_barrier_sync(3, kAuxThreads);
    if (!*aux_go) return;  // (the same in every aux warp: written once, before barrier 3)
    const int k = p.k;
    const int64_t H = p.H, total = (int64_t)p.T * (H / 4);
    const int32_t* pos = route_in ? rs->pos : lay ? lay[l].pos : p.pos;
    const float* gate = route_in ? rs->gate : lay ? lay[l].gate : p.gate;
    const uint16_t* x_res = lay ? lay[l].x_res : nullptr;
    uint16_t* x_out = lay ? lay[l].x_out : p.y;
    const int32_t* pos_next = lay ? lay[l].pos_next : nullptr;
    for (int64_t i = (int64_t)blockIdx.x * kAuxThreads + aux_w * 32 + lane; i < total;
         i += (int64_t)gridDim.x * kAuxThreads)
      combine_next_unit<true, true>(i, p.yp, pos, gate, p.T, H, k, x_res, x_out, pos_next,
                                    p.route.xq, p.route.xs, p.status);
    if (lay && l + 1 < n_layers) {
      fence_proxy_async_global();  // the next layer's TMA reads these act1 rows
      named_barrier_sync(1, kAuxThreads);
      if (aux_w == 0 && lane == 0)
        grid_arrive(p.sync, kSyncAct + ((l + 1) & 1), tag | (kActKind + (uint64_t)(l + 1)));
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Like the MMA issuer: a convergent warp walks the fills and one elected
    // lane issues each copy.
    const uint64_t pol_x = ptx::policy_evict_last();
    uint32_t fill = 0;
    uint32_t a_until = prefilled;  // fills below this have their weight tiles issued
    bool ok = true;
    for (int l = 0; ok && l < n_layers; ++l) {
      const int nch = n_chunks_of(l);
      const int items0 = nch * m1, items_all = items0 + nch * m2;
      if (lay && l > 0) {
        // A chained layer: its first weight tiles are issued as stages free up
        // (the previous layer's last items still run), then the layer waits
        // (bounded) until every CTA's combine has written its act1 rows.
        uint32_t f = fill;
        int it = blockIdx.x, ks = 0;
        while (f < fill + (uint32_t)C::kStages && it < items_all) {
          const int phase = (kPhases > 1 && it >= items0) ? 1 : 0;
          const TcPhase& ph = p.ph[phase];
          const int local = it - (phase ? items0 : 0);
          const int chunk = local / ph.m_tiles;
          const int4 ch = chunk_at(l, chunk);
          const int row0 = ch.x * ph.R + (local - chunk * ph.m_tiles) * ph.m_stride;
          const uint32_t tx = C::kA * C::kTxA + (uint32_t)((ch.z + 15) & ~15) * 128;
          const int s = (int)(f % C::kStages);
          if (!wait_all(&empty[s], ((f / C::kStages) & 1) ^ 1)) {
            if (lane == 0) fail(kStatusTimeout);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::kStageBytes;
          ptx::mbar_arrive_expect_tx_warp(&full[s], tx);
          const uint64_t pol_w = weight_policy(phase);
          ptx::tma_load_2d_warp(st, map_w(phase, l), &full[s], ks * kBlockK, row0, pol_w);
          ptx::tma_load_2d_warp(st + C::kATile, map_w(phase, l), &full[s], ks * kBlockK,
                                row0 + ph.half, pol_w);
          ++f;
          if (++ks == ph.K / kBlockK) {
            ks = 0;
            it += gridDim.x;
          }
        }
        if (!ok) break;
        a_until = f;
        const uint64_t act_v = tag | (kActKind + (uint64_t)l);
        if (!grid_wait(p.sync, kSyncAct + (l & 1), act_v, tag, p.timeout_ns, abort_flag)) {
          if (lane == 0) fail(kStatusTimeout);
          break;
        }
        fence_proxy_async_global();
      }
      for (int item = blockIdx.x; ok && item < items_all; item += gridDim.x) {
        const int phase = (kPhases > 1 && item >= items0) ? 1 : 0;
        const TcPhase& ph = p.ph[phase];
        const int local = item - (phase ? items0 : 0);
        const int chunk = local / ph.m_tiles;
        const int mt = local - chunk * ph.m_tiles;
        const int4 ch = chunk_at(l, chunk);
        // h of this chunk must be published by GEMM1 (unless the look-ahead of
        // the previous item already saw it complete); a chained layer's GEMM1
        // items are ready once the act1 barrier above is passed
        if (dep_phase(phase, l) && ld_acquire_cta(dep_ready) < item_seq(l, item)) {
          bool ready = true;
          if (phase == 1) {
            if (kLayer) {  // every GEMM1 tile pair of the chunk has set its flags
              const uint64_t until = deadline();
              uint32_t spins = 0;
              while (!chunk_tiles_published(p.sync, chunk * m1 * 4, m1 * 4, flag_want(l))) {
                bool stop = false;
                if ((++spins & 7u) == 0)
                  stop = *abort_flag || grid_aborted(p.sync, tag) || ptx::globaltimer() > until;
                if (__any_sync(0xffffffffu, stop)) {
                  ready = false;
                  break;
                }
              }
              if (ready) fence_acquire_gpu();
            } else {
              ready = wait_chunk_ready(p, chunk, ph.dep_target, p.timeout_ns, abort_flag);
            }
          }
          if (!__all_sync(0xffffffffu, ready)) {
            if (lane == 0) fail(kStatusTimeout);
            ok = false;
            break;
          }
          fence_proxy_async_global();
          if (lane == 0) st_release_cta(dep_ready, item_seq(l, item));
        }
        // Look-ahead (single-launch paths): read the next item's chunk flags
        // or counter now and look at them a few fills later, so the load's
        // latency hides behind this item's copies; if the chunk is complete,
        // publish the next item early so the scale stagers can load its h
        // scales ahead of time.  A chained layer's next GEMM1 item is ready
        // already.
        const int nxt = item + (int)gridDim.x;
        if (lay && l > 0 && nxt < items0 && lane == 0) st_release_cta(dep_ready, item_seq(l, nxt));
        bool look = kPhases > 1 && nxt < items_all && nxt >= items0;
        int look_cnt = 0;
        bool look_flags = true;  // (whole-layer launch) this lane's flags of the next chunk
        if (look) {
          const int nc = (nxt - items0) / (kPhases > 1 ? m2 : 1);
          if (kLayer) {
            for (int i = lane; i < m1 * 4; i += 32)
              look_flags &= ld_relaxed_u64(p.sync.chunk_flags + nc * m1 * 4 + i) == flag_want(l);
          } else {
            look_cnt = ld_relaxed(p.gemm1_done + nc);
          }
        }
        const int ksteps = ph.K / kBlockK;
        const int nrows = (ch.z + 15) & ~15;
        const int row0 = ch.x * ph.R + mt * ph.m_stride;
        const uint32_t tx = C::kA * C::kTxA + (uint32_t)nrows * 128;
        for (int ks = 0; ks < ksteps; ++ks, ++fill) {
          const int s = (int)(fill % C::kStages);
          const uint32_t use = fill / C::kStages;
          uint8_t* st = smem + s * C::kStageBytes;
          if (fill >= a_until) {  // (earlier fills have their weight tiles in flight)
            if (!wait_all(&empty[s], (use & 1) ^ 1)) {
              if (lane == 0) fail(kStatusTimeout);
              ok = false;
              break;
            }
            ptx::mbar_arrive_expect_tx_warp(&full[s], tx);
            const uint64_t pol_w = weight_policy(phase);
            ptx::tma_load_2d_warp(st, map_w(phase, l), &full[s], ks * kBlockK, row0, pol_w);
            ptx::tma_load_2d_warp(st + C::kATile, map_w(phase, l), &full[s], ks * kBlockK,
                                  row0 + ph.half, pol_w);
          }
          for (int r = 0; r < nrows; r += kBoxRowsB)
            ptx::tma_load_2d_warp(st + C::kA * C::kATile + r * 128, &ph.map_x, &full[s],
                                  ks * kBlockK, ch.y + r, pol_x);
          if (look && ks == min(3, ksteps - 1)) {
            if (__all_sync(0xffffffffu, kLayer ? look_flags : look_cnt >= p.ph[1].dep_target)) {
              fence_acq_rel_gpu();  // the relaxed load plus this fence: an acquire
              fence_proxy_async_global();
              if (lane == 0) st_release_cta(dep_ready, item_seq(l, nxt));
            }
            look = false;
          }
        }
      }
    }
    // a chained layer (one launch per layer): prefetch the first K steps of
    // the item this CTA takes first in the next layer's GEMM1 (items are
    // dealt round-robin over the same grid, so that is item blockIdx.x)
    if (ok && p.next.stages > 0 && (int)blockIdx.x < p.next.meta[0] * p.next.m_tiles) {
      const int4 ch = p.next.chunks[blockIdx.x / p.next.m_tiles];
      const int row0 = ch.x * p.next.R + ((int)blockIdx.x % p.next.m_tiles) * p.next.m_stride;
      if (ptx::elect_one()) {
        for (int ks = 0; ks < p.next.stages; ++ks) {
          ptx::tma_prefetch_2d(&p.next.map_w, ks * kBlockK, row0);
          ptx::tma_prefetch_2d(&p.next.map_w, ks * kBlockK, row0 + p.next.half);
        }
      }
      __syncwarp();
    }
    // every copy of this CTA is issued: the next kernel may be scheduled
    grid_launch_dependents();
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop on warp-uniform values and one elected lane
    // issues each tcgen05 instruction; wait outcomes are made warp-uniform.
    // A plain item loop: only N and the k-step count are needed here, and the
    // issuer's loop overhead is on the critical path of every stage.
    uint32_t fill = 0;
    bool ok = true;
    int j = 0;
    for (int l = 0; ok && l < n_layers; ++l) {
      const int nch = n_chunks_of(l);
      const int items0 = nch * m1, items_all = items0 + nch * m2;
      for (int item = blockIdx.x; ok && item < items_all; item += gridDim.x, ++j) {
        const int phase = (kPhases > 1 && item >= items0) ? 1 : 0;
        const int local = item - (phase ? items0 : 0);
        const int4 ch = chunk_at(l, local / p.ph[phase].m_tiles);
        const int ksteps = p.ph[phase].K / kBlockK;
        const uint32_t N = (uint32_t)((ch.z + 15) & ~15);
        const int b = j % C::kAccBufs;
        const uint32_t u = (uint32_t)(j / C::kAccBufs);
        if (!wait_all(&acc_empty[b], (u & 1) ^ 1)) {
          if (lane == 0) fail(kStatusTimeout);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t acc0 = tbase + b * C::kAccCols;
        const uint32_t acc1 = acc0 + kNMax;
        for (int ks = 0; ks < ksteps; ++ks, ++fill) {
          const int s = (int)(fill % C::kStages);
          const uint32_t use = fill / C::kStages;
          if (!wait_all(&full[s], use & 1)) {
            if (lane == 0) fail(kStatusTimeout);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t st = ptx::smem_u32(smem + s * C::kStageBytes);
          const uint32_t sa0 = st, sa1 = st + C::kATile, sb = st + C::kA * C::kATile;
          const uint32_t tsf = tbase + C::kSfBase + s * C::kSfStride;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t idesc = ptx::idesc_mxf8f6f4(N, kk, kk);
            const uint32_t accum = (ks | kk) ? 1u : 0u;
            ptx::mma_mxf8f6f4_warp(acc0, ptx::desc_kmajor_sw128(sa0 + 32 * kk),
                                   ptx::desc_kmajor_sw128(sb + 32 * kk), idesc, tsf,
                                   tsf + C::kSfbCol, accum);
            ptx::mma_mxf8f6f4_warp(acc1, ptx::desc_kmajor_sw128(sa1 + 32 * kk),
                                   ptx::desc_kmajor_sw128(sb + 32 * kk), idesc, tsf + 4,
                                   tsf + C::kSfbCol, accum);
          }
          ptx::mma_commit_warp(&empty[s]);  // frees the smem stage and its scale columns
        }
        if (!ok) break;
        ptx::mma_commit_warp(&acc_full[b]);
      }
    }
    ptx::mma_commit_warp(drain);
    if (!wait_all(drain, 0) && lane == 0) fail(kStatusTimeout);
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ scale stagers
    // When every phase's scale rows allow it (K a multiple of 512), scale
    // words are loaded a group of kSfGroup fills at a time, one group ahead of
    // the group being written into TMEM: one 16-byte load per row covers a
    // group (a quarter of the L2 requests of per-stage loads) and a group
    // never straddles two work items.  Scales of an item whose inputs are not
    // yet published are never loaded ahead: they are loaded at store time,
    // after the (bounded) wait, so a stager never blocks ahead of fills it
    // still has to stage.  Other K (small layers) take one fill at a time.
    // The cursor runs through every layer of the launch.  (The two loops are
    // kept apart: folding the second into the first's unrolled body slowed
    // the first by several percent at the full layer shape.)
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    bool vec = true;
    for (int ph = 0; ph < kPhases; ++ph) vec = vec && (p.ph[ph].K % (32 * 16)) == 0;
    Cursor ld, stc;
    ld.start(p, lay, n_layers, s_chunks, s_nchunks, blockIdx.x, gridDim.x, 0, true);
    stc = ld;
    uint32_t grp[2][kSfGroup][C::kWords];
    Cursor grp_at[2];
    auto words_of_fill = [&](uint32_t (&w)[C::kWords], const Cursor& c) {
      const TcPhase& ph = p.ph[c.phase];
      const uint8_t* wsf = w_sf(c.phase, c.layer);
      const int sf_row = ph.K / 32;
      const int64_t row = (int64_t)c.ch.x * ph.R + c.mt * ph.m_stride + q * 32 + lane;
#pragma unroll
      for (int a = 0; a < C::kA; ++a)
        if (row + a * ph.half < ph.rows_total)
          w[a] = __ldg(reinterpret_cast<const uint32_t*>(wsf + (row + a * ph.half) * sf_row +
                                                         c.ks * 4));
#pragma unroll
      for (int jb = 0; jb < kNMax / 32; ++jb) {
        const int n = jb * 32 + lane;
        if (n < c.ch.z) {
          const unsigned int* src = reinterpret_cast<const unsigned int*>(
              ph.x_sf + (int64_t)(c.ch.y + n) * sf_row + c.ks * 4);
          // scales written earlier in this launch need a coherent load
          w[C::kA + jb] = coherent_x(c.phase, c.layer) ? __ldcg(src) : __ldg(src);
        }
      }
    };
    auto words_of_group = [&](uint32_t (&g)[kSfGroup][C::kWords], const Cursor& c0) {
      // the group's fills are ks .. ks+3 of one work item (vector path)
      const TcPhase& ph = p.ph[c0.phase];
      const uint8_t* wsf = w_sf(c0.phase, c0.layer);
      const int sf_row = ph.K / 32;
      const int64_t row = (int64_t)c0.ch.x * ph.R + c0.mt * ph.m_stride + q * 32 + lane;
#pragma unroll
      for (int a = 0; a < C::kA; ++a) {
        if (row + a * ph.half < ph.rows_total) {
          const uint4 v = __ldg(
              reinterpret_cast<const uint4*>(wsf + (row + a * ph.half) * sf_row + c0.ks * 4));
          g[0][a] = v.x;
          g[1][a] = v.y;
          g[2][a] = v.z;
          g[3][a] = v.w;
        }
      }
#pragma unroll
      for (int jb = 0; jb < kNMax / 32; ++jb) {
        const int n = jb * 32 + lane;
        if (n < c0.ch.z) {
          const uint4* src = reinterpret_cast<const uint4*>(
              ph.x_sf + (int64_t)(c0.ch.y + n) * sf_row + c0.ks * 4);
          const uint4 v = coherent_x(c0.phase, c0.layer) ? __ldcg(src) : __ldg(src);
          g[0][C::kA + jb] = v.x;
          g[1][C::kA + jb] = v.y;
          g[2][C::kA + jb] = v.z;
          g[3][C::kA + jb] = v.w;
        }
      }
    };
    // bounded wait until the producer has published item `seq` (a
    // shared-memory read of dep_ready: the producer's acquire of the flags or
    // counter, then its release there, orders the writes of h or of the act1
    // rows before this warp's loads of their scales)
    auto wait_item_ready = [&](int seq) {
      const uint64_t until = deadline();
      while (ld_acquire_cta(dep_ready) < seq) {
        if (*abort_flag || ptx::globaltimer() > until) return false;
      }
      return true;
    };
    bool ok = true;
    uint32_t fill = 0;
    if (!vec) {
      // Scale rows of a K that is not a multiple of 512 (small layers): one
      // fill at a time, its words loaded right after its own item's (bounded)
      // wait, so a fill never waits for a later item's inputs.
      while (ok && stc.valid()) {
        uint32_t w[C::kWords];
#pragma unroll
        for (int x = 0; x < C::kWords; ++x) w[x] = 0;
        if (kPhases == 2 && dep_phase(stc.phase, stc.layer) &&
            !__all_sync(0xffffffffu, wait_item_ready(stc.seq()))) {
          if (lane == 0) fail(kStatusTimeout);
          ok = false;
          break;
        }
        words_of_fill(w, stc);
        const int s = (int)(fill % C::kStages);
        if (!wait_all(&empty[s], ((fill / C::kStages) & 1) ^ 1)) {
          if (lane == 0) fail(kStatusTimeout);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tsf = tbase + lane_off + C::kSfBase + s * C::kSfStride;
#pragma unroll
        for (int a = 0; a < C::kA; ++a) ptx::tmem_st_x1(tsf + 4 * a + q, w[a]);
#pragma unroll
        for (int jb = 0; jb < kNMax / 32; ++jb) ptx::tmem_st_x1(tsf + C::kSfbCol + jb, w[C::kA + jb]);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&full[s]);
        ++fill;
        stc.next();
      }
    } else {
      // Vector path: a group is four fills of one work item.  A group whose
      // item's inputs are not yet published is loaded at store time, after
      // the (bounded) wait.
      bool deferred[2] = {false, false};
      auto load_group = [&](int gi, uint32_t (&g)[kSfGroup][C::kWords]) {
#pragma unroll
        for (int i = 0; i < kSfGroup; ++i)
#pragma unroll
          for (int w = 0; w < C::kWords; ++w) g[i][w] = 0;
        grp_at[gi] = ld;
        if (kPhases == 2)
          deferred[gi] = __any_sync(0xffffffffu, dep_phase(ld.phase, ld.layer) &&
                                                     ld_acquire_cta(dep_ready) < ld.seq());
        if (!deferred[gi] && ld.valid()) words_of_group(g, ld);
#pragma unroll
        for (int i = 0; i < kSfGroup; ++i) ld.next();
      };
      load_group(0, grp[0]);
      load_group(1, grp[1]);
      while (ok && stc.valid()) {
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
          if (kPhases == 2 && ok && stc.valid() && deferred[gi]) {
            if (!__all_sync(0xffffffffu, wait_item_ready(grp_at[gi].seq()))) {
              if (lane == 0) fail(kStatusTimeout);
              ok = false;
            } else if (grp_at[gi].valid()) {
              words_of_group(grp[gi], grp_at[gi]);
            }
            deferred[gi] = false;
          }
#pragma unroll
          for (int i = 0; i < kSfGroup; ++i) {
            if (ok && stc.valid()) {
              const int s = (int)(fill % C::kStages);
              const uint32_t use = fill / C::kStages;
              if (!wait_all(&empty[s], (use & 1) ^ 1)) {
                if (lane == 0) fail(kStatusTimeout);
                ok = false;
              } else {
                ptx::tc_fence_after();
                const uint32_t tsf = tbase + lane_off + C::kSfBase + s * C::kSfStride;
#pragma unroll
                for (int a = 0; a < C::kA; ++a) ptx::tmem_st_x1(tsf + 4 * a + q, grp[gi][i][a]);
#pragma unroll
                for (int jb = 0; jb < kNMax / 32; ++jb)
                  ptx::tmem_st_x1(tsf + C::kSfbCol + jb, grp[gi][i][C::kA + jb]);
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&full[s]);
                ++fill;
                stc.next();
              }
            }
          }
          if (ok && stc.valid()) load_group(gi, grp[gi]);  // the group two ahead
        }
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int j = 0;
    for (int l = 0; l < n_layers; ++l) {
      Cursor c;
      c.start(p, lay, n_layers, s_chunks, s_nchunks, blockIdx.x, gridDim.x, l, false);
      for (; c.valid(); ++j) {
        const TcPhase& ph = p.ph[c.phase];
        const int4 ch = c.ch;
        const int mt = c.mt, chunk = c.chunk;
        const int b = j % C::kAccBufs;
        const uint32_t u = (uint32_t)(j / C::kAccBufs);
        if (!wait_all(&acc_full[b], u & 1)) {
          if (lane == 0) fail(kStatusTimeout);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t acc0 = tbase + lane_off + b * C::kAccCols;
        const int row = mt * ph.m_stride + q * 32 + lane;  // output row within the expert
        // eight tokens (accumulator columns) at a time, computed for all eight
        // (columns past the chunk exist and are ignored) so their arithmetic
        // and warp reductions interleave; only the stores are predicated
        for (int n0 = 0; n0 < ch.z; n0 += 8) {
          uint32_t v0[8], v1[8];
          ptx::tmem_ld_x8(acc0 + n0, v0);
          ptx::tmem_ld_x8(acc0 + kNMax + n0, v1);
          ptx::tmem_ld_wait();
          const int nv = min(8, ch.z - n0);  // warp-uniform
          const int64_t slot0 = ch.y + n0;
          if (gated_phase(c.phase)) {
            // h = silu(gate) * up, then MXFP8 along I: this warp's 32 rows are
            // one block of 32 of token n0 + t
            float h[8], amax[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const float g = __uint_as_float(v0[t]);
              h[t] = __fdividef(g, 1.0f + __expf(-g)) * __uint_as_float(v1[t]);
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) amax[t] = warp_max_abs(h[t]);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              if (t < nv) {
                const int code = block_scale_code(amax[t], 8);
                p.hq[(slot0 + t) * ph.out_dim + row] =
                    e4m3_encode_satfinite(h[t] * exp2_exact(127 - code));
                if (lane == 0) p.hs[(slot0 + t) * (ph.out_dim / 32) + row / 32] = (uint8_t)code;
              }
            }
          } else {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              if (t < nv) {
                p.yp[(slot0 + t) * ph.out_dim + row] = __uint_as_float(v0[t]);
                if (row + 128 < ph.out_dim)
                  p.yp[(slot0 + t) * ph.out_dim + row + 128] = __uint_as_float(v1[t]);
              }
            }
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&acc_empty[b]);
        if (kLayer && gated_phase(c.phase)) {
          // publish this warp's quarter of the tile pair of h: its generic
          // stores made visible to other CTAs' TMA reads (async proxy) and
          // loads, then its own flag (four per tile pair; no barrier among the
          // epilogue warps, which may leave their loops at different items
          // when a wait runs out)
          fence_proxy_async_global();
          __syncwarp();
          if (lane == 0)
            publish_chunk_tile(p.sync, (chunk * ph.m_tiles + mt) * 4 + q,
                               tag | (kChunkFlagKind + (uint64_t)l));
        } else if (kPhases == 2 && gated_phase(c.phase)) {
          // publish this warp's quarter of h: its generic stores made visible to
          // other CTAs' TMA reads (async proxy) and loads, then one release
          // increment per warp (four per tile pair)
          fence_proxy_async_global();
          __threadfence();
          __syncwarp();
          if (lane == 0) red_release_add(p.gemm1_done + chunk, 1);
        }
        c.next_item();
      }
      if (kLayer) aux_combine(l);
    }
  } else if (kLayer && (warp == 1 || warp == 3)) {
    // ------------------------------------------------------------ aux (whole-layer launch)
    for (int l = 0; l < n_layers; ++l) aux_combine(l);
  }

  if (*abort_flag) {  // let copies already in flight land before the CTA exits
    const uint64_t until = ptx::globaltimer() + 2000000ull;
    while (ptx::globaltimer() < until) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 2) ptx::tmem_dealloc(tbase, C::kTmemCols);
}

template <int kNMax, int kMode>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
  gemm_tc_body<kNMax, kMode>(p, nullptr, 1);
}

// A chain of layers in one persistent launch (whole layers, routed before it)
template <int kNMax>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_chain_kernel(
    const __grid_constant__ ChainParams cp) {
  gemm_tc_body<kNMax, kModeLayer>(cp.p, cp.lay, cp.n_layers);
}

}  // namespace moe
