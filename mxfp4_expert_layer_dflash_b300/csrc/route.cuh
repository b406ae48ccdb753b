// Routing steps of the layer:
//  (1) top-k of each token's router logits (the lower expert index wins ties)
//      and the softmax renormalised over the k selected logits;
//  (2) per-expert histogram of the T*k assignments;
//  (3) exclusive prefix scan over experts and the list of work chunks;
//  (4) stable permutation: slot = off[e] + rank of (t, j) among expert e's
//      assignments in ascending t*k + j.
// Expert routing is part of the pipeline the runtime is co-designed with:
// techllm.github.io, "Xiaomi MiMo and TileRT ...", section "3. TileRT".
#pragma once

#include <float.h>

#include "common.cuh"

namespace moe {

// One warp per token.  MAXPL logits per lane (E <= 32 * MAXPL).
template <int MAXPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int32_t* __restrict__ idx,
                                                         float* __restrict__ w, int* status) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int t = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  float v[MAXPL];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < MAXPL; ++i) {
    int e = lane + 32 * i;
    v[i] = e < E ? l[e] : -FLT_MAX;
    if (e >= E) taken |= 1u << i;
  }
  float my_v = 0.0f;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < MAXPL; ++i) {
      int e = lane + 32 * i;
      if (!((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be >= E) {  // only possible with non-finite logits
      if (lane == 0) set_status(status, kStatusFault);
      be = 0;
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_v = bv;
      my_e = be;
    }
  }
  const float m = __shfl_sync(0xffffffffu, my_v, 0);  // first pick is the largest
  const float ex = lane < k ? expf(my_v - m) : 0.0f;
  const float s = warp_sum(ex);
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_e;
    w[(size_t)t * k + lane] = ex / s;
  }
}

__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int wv = s_warp[lane];
    int wx = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, wx, o);
      if (lane >= o) wx += y;
    }
    s_warp[lane] = wx - wv;  // exclusive prefix of warp totals
    if (lane == 31) *total = wx;
  }
  __syncthreads();
  int r = s_warp[warp] + x - v;
  __syncthreads();
  return r;
}

// Single CTA of 1024 threads: histogram, scan, stable permutation, chunk list.
// Dynamic shared memory: (35 * E + 1 + 34) ints.
__global__ void __launch_bounds__(1024) route_permute_kernel(
    const int32_t* __restrict__ idx, int T, int k, int E, int32_t* __restrict__ cnt_out,
    int32_t* __restrict__ off_out, int32_t* __restrict__ perm, int32_t* __restrict__ pos,
    int4* __restrict__ chunks, int max_chunks, int chunk_max, int32_t* __restrict__ meta,
    int32_t* __restrict__ done, int* status) {
  extern __shared__ int smem[];
  int* s_cnt = smem;          // E
  int* s_off = s_cnt + E;     // E + 1
  int* s_run = s_off + E + 1; // E
  int* s_w = s_run + E;       // 32 * E
  int* s_warp = s_w + 32 * E; // 32
  int* s_tot = s_warp + 32;   // 2
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int TK = T * k;
  grid_dependency_wait();
  grid_launch_dependents();

  for (int e = tid; e < E; e += 1024) {
    s_cnt[e] = 0;
    s_run[e] = 0;
  }
  if (done)
    for (int i = tid; i < max_chunks; i += 1024) done[i] = 0;  // per-call completion counters
  __syncthreads();
  for (int f = tid; f < TK; f += 1024) {
    int e = idx[f];
    if ((unsigned)e >= (unsigned)E) {
      set_status(status, kStatusFault);
      e = 0;
    }
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();

  const int c = tid < E ? s_cnt[tid] : 0;
  const int excl = block_exclusive_scan_1024(c, s_warp, &s_tot[0]);
  if (tid < E) {
    s_off[tid] = excl;
    cnt_out[tid] = c;
    off_out[tid] = excl;
  }
  if (tid == 0) {
    s_off[E] = TK;
    off_out[E] = TK;
  }
  __syncthreads();

  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < TK; base += 1024) {
    const int f = base + tid;
    const bool valid = f < TK;
    int e = valid ? idx[f] : -1;
    if (valid && (unsigned)e >= (unsigned)E) e = 0;
    for (int i = tid; i < 32 * E; i += 1024) s_w[i] = 0;
    __syncthreads();
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & lt_mask);
    if (valid && rank == 0) s_w[warp * E + e] = __popc(same);
    __syncthreads();
    for (int ee = tid; ee < E; ee += 1024) {
      int run = s_run[ee];
      for (int w = 0; w < 32; ++w) {
        int cw = s_w[w * E + ee];
        s_w[w * E + ee] = run;
        run += cw;
      }
      s_run[ee] = run;
    }
    __syncthreads();
    if (valid) {
      const int slot = s_off[e] + s_w[warp * E + e] + rank;
      perm[slot] = f / k;
      pos[f] = slot;
    }
    __syncthreads();
  }

  // chunk list: touched experts in ascending order, each split into
  // ceil(n / chunk_max) chunks of near-equal size
  const int nch = c > 0 ? (c + chunk_max - 1) / chunk_max : 0;
  const int cbase = block_exclusive_scan_1024(nch, s_warp, &s_tot[0]);
  const int touched = block_exclusive_scan_1024(c > 0 ? 1 : 0, s_warp, &s_tot[1]);
  (void)touched;
  if (tid < E && nch > 0) {
    const int q = (c + nch - 1) / nch;
    for (int i = 0; i < nch; ++i) {
      const int b = cbase + i;
      const int n = min(q, c - i * q);
      if (b < max_chunks) chunks[b] = make_int4(tid, excl + i * q, n, 0);
      else set_status(status, kStatusFault);
    }
  }
  if (tid == 0) {
    meta[0] = min(s_tot[0], max_chunks);
    meta[1] = s_tot[1];
  }
}

}  // namespace moe
