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
// routing arrays, and every CTA then gathers and quantises its share of the
// slot rows (MXFP8, blocks of 32 along H) or copies them (bf16 mode).
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

template <int MAXPL, bool kMxfp8>
__global__ void __launch_bounds__(1024) route_act_small_kernel(
    const float* __restrict__ logits, const uint16_t* __restrict__ x, int T, int H, int E, int k,
    int max_chunks, int chunk_max, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
    int32_t* __restrict__ cnt, int32_t* __restrict__ off, int32_t* __restrict__ perm,
    int32_t* __restrict__ pos, int4* __restrict__ chunks, int32_t* __restrict__ meta,
    int32_t* __restrict__ done, uint8_t* __restrict__ q, uint8_t* __restrict__ s, int* status) {
  extern __shared__ __align__(16) uint8_t sm[];
  const SmallRouteSmem L = small_route_smem(T, E, k, max_chunks);
  int32_t* s_idx = reinterpret_cast<int32_t*>(sm + L.idx);
  float* s_gate = reinterpret_cast<float*>(sm + L.gate);
  int32_t* s_cnt = reinterpret_cast<int32_t*>(sm + L.cnt);
  int32_t* s_off = reinterpret_cast<int32_t*>(sm + L.off);
  int32_t* s_perm = reinterpret_cast<int32_t*>(sm + L.perm);
  int32_t* s_pos = reinterpret_cast<int32_t*>(sm + L.pos);
  int4* s_chunks = reinterpret_cast<int4*>(sm + L.chunks);
  int32_t* s_meta = reinterpret_cast<int32_t*>(sm + L.meta);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int TK = T * k;
  grid_dependency_wait();
  grid_launch_dependents();

  // (1) top-k + softmax: warp t takes token t
  int* s_warp = reinterpret_cast<int*>(sm);  // 32 + 2 ints of block-scan scratch
  int* s_tot = s_warp + 32;
  if (warp < T) route_topk_token<MAXPL>(logits, warp, E, k, s_idx, s_gate, status);
  for (int e = tid; e < E; e += 1024) s_cnt[e] = 0;
  if (blockIdx.x == 0 && done)
    for (int i = tid; i < max_chunks; i += 1024) done[i] = 0;  // per-call completion counters
  __syncthreads();
  // (2)-(4) for at most 32 * 16 assignments: counts, offsets, each assignment's
  // rank among the earlier ones of its expert (a direct count: at most 511
  // broadcast reads), chunk list — route_permute_kernel's results exactly
  for (int f = tid; f < TK; f += 1024) {
    if ((unsigned)s_idx[f] >= (unsigned)E) {  // never from the top-k; kept as a guard
      set_status(status, kStatusFault);
      s_idx[f] = 0;
    }
  }
  __syncthreads();
  for (int f = tid; f < TK; f += 1024) atomicAdd(&s_cnt[s_idx[f]], 1);
  __syncthreads();
  const int c = tid < E ? s_cnt[tid] : 0;
  const int excl = block_exclusive_scan_1024(c, s_warp, &s_tot[0]);
  if (tid < E) s_off[tid] = excl;
  if (tid == 0) s_off[E] = TK;
  __syncthreads();
  if (tid < TK) {
    const int e = s_idx[tid];
    int r = 0;
    for (int g = 0; g < tid; ++g) r += s_idx[g] == e;
    const int slot = s_off[e] + r;
    s_pos[tid] = slot;
    s_perm[slot] = tid / k;
  }
  route_chunk_list(c, excl, E, chunk_max, s_chunks, max_chunks, s_meta, s_warp, s_tot, status);
  __syncthreads();
  if (blockIdx.x == 0) {  // publish the routing arrays
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

  // a4: this CTA's share of the slot rows; a warp per (slot, run of 32
  // blocks of 32), a block per lane (the standalone kernels' arithmetic)
  const int64_t nb = H / 32, segs = (nb + 31) / 32;
  const int64_t warps = (int64_t)gridDim.x * 32;
  for (int64_t u = (int64_t)blockIdx.x * 32 + warp; u < (int64_t)TK * segs; u += warps) {
    const int64_t r = u / segs;
    const int64_t b = (u - r * segs) * 32 + lane;
    int64_t src = s_perm[r];
    if (src < 0 || src >= T) {
      if (lane == 0) set_status(status, kStatusFault);
      src = 0;
    }
    if (b >= nb) continue;
    if (kMxfp8) {
      float v[32];
      uint8_t c[32];
      load_bf16x32(x + src * H + b * 32, v);
      const int code = mxfp8_block(v, c);
      store_u8x32(q + r * H + b * 32, c);
      s[r * nb + b] = (uint8_t)code;
    } else {
      const uint4* a = reinterpret_cast<const uint4*>(x + src * H + b * 32);
      uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(q) + r * H + b * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = a[i];
    }
  }
}

}  // namespace moe
