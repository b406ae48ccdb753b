// Steps a1-a4 in one launch for small token blocks (T <= kSmallRouteTokens,
// e.g. one DFlash verification block of 8 positions per sequence: the case
// where each operator lasts microseconds and launch gaps dominate —
// dothoosh.com, section "TileRT").
//
// Every CTA recomputes the whole routing of the block in its own shared
// memory (at most 32 tokens: one warp per token for the top-k — the
// three-kernel path's device code — then histogram, scan, stable permutation
// and chunk list for at most 512 assignments, where each assignment's rank
// within its expert is a direct count of the earlier equal ones: the same
// arrays as the general permutation, bit for bit), CTA 0 publishes the
// routing arrays.  Step a4 runs token-major: the warps that the top-k leaves
// idle read and quantise (MXFP8, blocks of 32 along H) or read (bf16 mode)
// their share of the token rows while the routing runs, and write each to
// the token's k slot rows once the slots are known.
// Redundant routing costs a few microseconds of L2 reads of the [T, E]
// logits per CTA; it removes two launches and their dependency waits.
#pragma once

#include "common.cuh"
#include "quant.cuh"
#include "route.cuh"

namespace moe {

constexpr int kSmallRouteTokens = 32;  // one warp per token in a 1024-thread CTA

// Shared memory of route_act_small_kernel: the block scans' scratch (64 ints
// at offset 0), then this block's routing arrays.
struct SmallRouteSmem {
  size_t idx, gate, cnt, off, perm, pos, chunks, meta, total;
};

__host__ __device__ inline SmallRouteSmem small_route_smem(int T, int E, int k, int max_chunks) {
  auto up16 = [](size_t b) { return (b + 15) & ~size_t(15); };
  SmallRouteSmem L{};
  size_t o = 64 * sizeof(int);
  const size_t tk = (size_t)T * k;
  L.idx = o;
  o = up16(o + tk * 4);
  L.gate = o;
  o = up16(o + tk * 4);
  L.cnt = o;
  o = up16(o + (size_t)E * 4);
  L.off = o;
  o = up16(o + (size_t)(E + 1) * 4);
  L.perm = o;
  o = up16(o + tk * 4);
  L.pos = o;
  o = up16(o + tk * 4);
  L.chunks = o;
  o = up16(o + (size_t)max_chunks * 16);
  L.meta = o;
  o = up16(o + 2 * 4);
  L.total = o;
  return L;
}

// One token-major unit of step a4: token t's run of 32 blocks of 32 along H
// (a block per lane), read and quantised (MXFP8) or read (bf16) into
// registers, then written to each of the token's k slot rows.
template <bool kMxfp8>
struct SmallActUnit {
  uint32_t w[kMxfp8 ? 8 : 16];
  int code;
  int64_t t, b;
  bool live;
  __device__ __forceinline__ void load(const uint16_t* __restrict__ x, int64_t u, int64_t segs,
                                       int64_t H) {
    const int lane = threadIdx.x & 31;
    t = u / segs;
    b = (u - t * segs) * 32 + lane;
    live = b < H / 32;
    if (!live) return;
    if (kMxfp8) {
      float v[32];
      uint8_t c[32];
      load_bf16x32(x + t * H + b * 32, v);
      code = mxfp8_block(v, c);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = (uint32_t)c[4 * i] | ((uint32_t)c[4 * i + 1] << 8) |
               ((uint32_t)c[4 * i + 2] << 16) | ((uint32_t)c[4 * i + 3] << 24);
    } else {
      const uint4* a = reinterpret_cast<const uint4*>(x + t * H + b * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 q = a[i];
        w[4 * i] = q.x;
        w[4 * i + 1] = q.y;
        w[4 * i + 2] = q.z;
        w[4 * i + 3] = q.w;
      }
    }
  }
  __device__ __forceinline__ void store(const int32_t* s_pos, int k, int TK, int64_t H,
                                        uint8_t* __restrict__ q, uint8_t* __restrict__ s,
                                        int* status) const {
    if (!live) return;
    const int64_t nb = H / 32;
    for (int j = 0; j < k; ++j) {
      const int64_t slot = s_pos[t * k + j];
      if (slot < 0 || slot >= TK) {
        set_status(status, kStatusFault);
        continue;
      }
      uint4* o = reinterpret_cast<uint4*>(q + (slot * H + b * 32) * (kMxfp8 ? 1 : 2));
#pragma unroll
      for (int i = 0; i < (kMxfp8 ? 2 : 4); ++i)
        o[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
      if (kMxfp8) s[slot * nb + b] = (uint8_t)code;
    }
  }
};

// The routing of one block of T <= 32 tokens by one CTA (every CTA that calls
// it for the block computes the same arrays); `publish`: this CTA writes them
// out.  x == nullptr: no step a4; else CTA `cta` of the `ncta` that share the
// block's a4 units.
template <int MAXPL, bool kMxfp8>
__device__ __forceinline__ void route_small_block(
    const float* __restrict__ logits, const uint16_t* __restrict__ x, int T, int H, int E, int k,
    int max_chunks, int chunk_max, bool publish, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, int32_t* __restrict__ cnt, int32_t* __restrict__ off,
    int32_t* __restrict__ perm, int32_t* __restrict__ pos, int4* __restrict__ chunks,
    int32_t* __restrict__ meta, int32_t* __restrict__ done, uint8_t* __restrict__ q,
    uint8_t* __restrict__ s, int* status, int cta, int ncta) {
  extern __shared__ __align__(16) uint8_t sm[];
  const SmallRouteSmem L = small_route_smem(T, E, k, max_chunks);
  int* s_warp = reinterpret_cast<int*>(sm);  // 32 + 2 ints of block-scan scratch
  int* s_tot = s_warp + 32;
  int32_t* s_idx = reinterpret_cast<int32_t*>(sm + L.idx);
  float* s_gate = reinterpret_cast<float*>(sm + L.gate);
  int32_t* s_cnt = reinterpret_cast<int32_t*>(sm + L.cnt);
  int32_t* s_off = reinterpret_cast<int32_t*>(sm + L.off);
  int32_t* s_perm = reinterpret_cast<int32_t*>(sm + L.perm);
  int32_t* s_pos = reinterpret_cast<int32_t*>(sm + L.pos);
  int4* s_chunks = reinterpret_cast<int4*>(sm + L.chunks);
  int32_t* s_meta = reinterpret_cast<int32_t*>(sm + L.meta);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int TK = T * k;
  const int64_t segs = (H / 32 + 31) / 32, units = (int64_t)T * segs;
  // warps T..31 of every CTA take the first token-major units of a4 while
  // warps 0..T-1 route; the rest of the units follow the routing
  const int64_t early = (int64_t)ncta * (32 - T);

  SmallActUnit<kMxfp8> held;
  held.live = false;
  if (warp < T) {
    // (1) top-k + softmax: warp t takes token t
    route_topk_token<MAXPL>(logits, warp, E, k, s_idx, s_gate, status);
  } else if (x) {
    const int64_t u = cta + (int64_t)ncta * (warp - T);
    if (u < units) held.load(x, u, segs, H);
  }
  for (int e = tid; e < E; e += 1024) s_cnt[e] = 0;
  if (publish && done)
    for (int i = tid; i < max_chunks; i += 1024) done[i] = 0;  // per-call completion counters
  __syncthreads();
  // (2)-(4) for at most 32 * 16 assignments: counts, offsets, each assignment's
  // rank among the earlier ones of its expert (a direct count), chunk list —
  // route_permute_kernel's results exactly
  for (int f = tid; f < TK; f += 1024) {
    int e = s_idx[f];
    if ((unsigned)e >= (unsigned)E) {  // never from the top-k; kept as a guard
      set_status(status, kStatusFault);
      e = 0;
      s_idx[f] = 0;
    }
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  const int c = tid < E ? s_cnt[tid] : 0;
  const int excl = block_exclusive_scan_1024(c, s_warp, &s_tot[0]);
  if (tid < E) s_off[tid] = excl;
  if (tid == 0) s_off[E] = TK;
  __syncthreads();
  if (tid < TK) {
    const int e = s_idx[tid];
    const int4* v4 = reinterpret_cast<const int4*>(s_idx);
    int r = 0;
#pragma unroll 4
    for (int g = 0; g < (tid >> 2); ++g) {
      const int4 v = v4[g];
      r += (v.x == e) + (v.y == e) + (v.z == e) + (v.w == e);
    }
    for (int g = tid & ~3; g < tid; ++g) r += s_idx[g] == e;
    const int slot = s_off[e] + r;
    s_pos[tid] = slot;
    s_perm[slot] = tid / k;
  }
  route_chunk_list<true>(c, excl, E, chunk_max, s_chunks, max_chunks, s_meta, s_warp, s_tot,
                         status);
  __syncthreads();
  if (publish) {
    for (int i = tid; i < TK; i += 1024) {
      topk_idx[i] = s_idx[i];
      topk_w[i] = s_gate[i];
      perm[i] = s_perm[i];
      pos[i] = s_pos[i];
    }
    for (int e = tid; e <= E; e += 1024) {
      if (e < E) cnt[e] = s_cnt[e];
      off[e] = s_off[e];
    }
    for (int c = tid; c < s_meta[0]; c += 1024) chunks[c] = s_chunks[c];
    if (tid < 2) meta[tid] = s_meta[tid];
  }

  if (!x) return;
  // a4: the held unit, then the units past the early ones (a warp each)
  held.store(s_pos, k, TK, H, q, s, status);
  for (int64_t u = early + (int64_t)cta * 32 + warp; u < units; u += (int64_t)ncta * 32) {
    SmallActUnit<kMxfp8> a;
    a.load(x, u, segs, H);
    a.store(s_pos, k, TK, H, q, s, status);
  }
}

// Steps a1-a4 of one layer: every CTA routes, CTA 0 publishes, all quantise
template <int MAXPL, bool kMxfp8>
__global__ void __launch_bounds__(1024) route_act_small_kernel(
    const float* __restrict__ logits, const uint16_t* __restrict__ x, int T, int H, int E, int k,
    int max_chunks, int chunk_max, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
    int32_t* __restrict__ cnt, int32_t* __restrict__ off, int32_t* __restrict__ perm,
    int32_t* __restrict__ pos, int4* __restrict__ chunks, int32_t* __restrict__ meta,
    int32_t* __restrict__ done, uint8_t* __restrict__ q, uint8_t* __restrict__ s, int* status) {
  grid_dependency_wait();
  grid_launch_dependents();
  route_small_block<MAXPL, kMxfp8>(logits, x, T, H, E, k, max_chunks, chunk_max,
                                   blockIdx.x == 0, topk_idx, topk_w, cnt, off, perm, pos,
                                   chunks, meta, done, q, s, status, blockIdx.x, gridDim.x);
}

// A chain of layers over one small block, on a 1-D grid of g0 + n - 1 CTAs:
// CTAs 0..g0-1 route layer 0 as route_act_small_kernel does (every one routes
// it, CTA 0 publishes, all run its step a4 into q / s); CTA g0 + l - 1 routes
// and publishes layer l >= 1 alone (its activation rows come from the
// previous layer's combine).  Layer l's routing arrays start l * stride bytes
// after layer 0's.
template <int MAXPL, bool kMxfp8>
__global__ void __launch_bounds__(1024) route_act_small_layers_kernel(
    const __grid_constant__ LayerLogits lg, const uint16_t* __restrict__ x, int T, int H, int E,
    int k, int max_chunks, int chunk_max, int32_t* topk_idx0, float* topk_w0, int32_t* cnt0,
    int32_t* off0, int32_t* perm0, int32_t* pos0, int4* chunks0, int32_t* meta0, int32_t* done0,
    uint8_t* __restrict__ q, uint8_t* __restrict__ s, int64_t stride, int g0, int* status) {
  const int b = (int)blockIdx.x;
  const int l = b < g0 ? 0 : b - g0 + 1;
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t o = (int64_t)l * stride;
  auto at = [o](auto* p) {
    using P = decltype(p);
    return reinterpret_cast<P>(reinterpret_cast<char*>(p) + o);
  };
  route_small_block<MAXPL, kMxfp8>(lg.p[l], l == 0 ? x : nullptr, T, H, E, k, max_chunks,
                                   chunk_max, b == 0 || l > 0, at(topk_idx0), at(topk_w0),
                                   at(cnt0), at(off0), at(perm0), at(pos0), at(chunks0), at(meta0),
                                   done0 ? at(done0) : nullptr, q, s, status, l == 0 ? b : 0,
                                   l == 0 ? g0 : 1);
}

}  // namespace moe
