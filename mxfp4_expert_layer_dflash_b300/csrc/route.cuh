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

#include "common.cuh"

namespace moe {

// Order-preserving key of a logit: a larger value has a larger key, equal
// values (+0 and -0 included) have equal keys.  Non-finite logits are outside
// the supported inputs.
__device__ __forceinline__ uint32_t topk_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0) u = 0;  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float topk_key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

__device__ __forceinline__ uint32_t warp_redux_max(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

__device__ __forceinline__ uint32_t warp_redux_min(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// Step (1) for token t, by one warp.  MAXPL logits per lane (E <= 32 * MAXPL).
// Round j picks the largest remaining logit, the lowest expert index among
// equal ones: the warp's largest key (one reduction), then the lowest index
// among the lanes whose own best has that key (a second one).
// kL2: load the logits from L2 only (written by other CTAs of the same launch)
// `l`: token t's E logits (global or shared memory)
template <int MAXPL, bool kL2 = false>
__device__ __forceinline__ void route_topk_row(const float* __restrict__ l, int t, int E, int k,
                                               int32_t* __restrict__ idx, float* __restrict__ w,
                                               int* status) {
  const int lane = threadIdx.x & 31;
  uint32_t key[MAXPL];
#pragma unroll
  for (int i = 0; i < MAXPL; ++i) {
    const int e = lane + 32 * i;
    // 0: below every finite logit's key
    key[i] = e < E ? topk_key(kL2 ? __ldcg(l + e) : l[e]) : 0u;
  }
  float my_v = 0.0f;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < MAXPL; ++i) {  // strict >: the lowest i (index) among equal keys
      if (key[i] > bk) {
        bk = key[i];
        bi = i;
      }
    }
    const uint32_t wk = warp_redux_max(bk);
    uint32_t be = warp_redux_min(bi >= 0 && bk == wk ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu);
    if (be >= (uint32_t)E) {  // only possible with non-finite logits
      if (lane == 0) set_status(status, kStatusFault);
      be = 0;
    }
    if ((int)(be & 31) == lane) {
#pragma unroll
      for (int i = 0; i < MAXPL; ++i)
        if (i == (int)(be >> 5)) key[i] = 0u;  // taken
    }
    if (lane == j) {
      my_v = topk_key_value(wk);
      my_e = (int)be;
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

template <int MAXPL, bool kL2 = false>
__device__ __forceinline__ void route_topk_token(const float* __restrict__ logits, int t, int E,
                                                 int k, int32_t* __restrict__ idx,
                                                 float* __restrict__ w, int* status) {
  route_topk_row<MAXPL, kL2>(logits + (size_t)t * E, t, E, k, idx, w, status);
}

// The router's split-K partials part[ks][t][e] summed into logits, and step
// (1) on them, in one kernel: a CTA per token.  Each thread takes kVec
// consecutive experts (4 when E % 4 == 0, else 1) of one of kTopkGroups split
// groups (splits g, g + 8, ...): its loads (one per split) are all issued
// before they are added, then the groups' sums are added in group order
// through shared memory — a fixed order, so the logits are deterministic;
// `logits` (may be null) receives them.  Then one warp takes the top-k from
// shared memory.  k == 0: the logits alone.  k_splits <= kTopkMaxSplits.
constexpr int kTopkGroups = 8, kTopkLoads = 8;
constexpr int kTopkMaxSplits = kTopkGroups * kTopkLoads;
constexpr int kTopkThreads = 1024;
// kCtas = 2: two CTAs of at most kTopkThreads2 threads share an SM (fewer
// registers each), so one wave covers twice the tokens — for token counts
// above one CTA per SM; kCtas = 1 keeps every load of a thread in registers
constexpr int kTopkThreads2 = 768;
template <int MAXPL, int kVec, int kCtas>
__global__ void __launch_bounds__(kCtas == 2 ? kTopkThreads2 : kTopkThreads, kCtas)
    splitk_topk_kernel(const float* __restrict__ part, int k_splits, int T, int E, int k,
                       float* __restrict__ logits, int32_t* __restrict__ idx, float* __restrict__ w,
                       int* status) {
  static_assert(kVec == 1 || kVec == 4, "experts per thread");
  __shared__ __align__(16) float s_grp[kTopkGroups][32 * MAXPL];
  __shared__ __align__(16) float s_l[32 * MAXPL];
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t n = (int64_t)T * E;  // floats per split
  const int EV = E / kVec;
  auto load = [&](const float* p, float (&r)[kVec]) {
    if (kVec == 4) {
      const float4 q = __ldcg(reinterpret_cast<const float4*>(p));
      r[0] = q.x;
      r[kVec > 1 ? 1 : 0] = q.y;
      r[kVec > 2 ? 2 : 0] = q.z;
      r[kVec > 3 ? 3 : 0] = q.w;
    } else {
      r[0] = __ldcg(p);
    }
  };
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    for (int u = threadIdx.x; u < kTopkGroups * EV; u += blockDim.x) {
      const int g = u / EV, e0 = (u - g * EV) * kVec;
      const float* src = part + (int64_t)t * E + e0;
      float v[kTopkLoads][kVec];
#pragma unroll
      for (int i = 0; i < kTopkLoads; ++i) {
        const int ks = g + kTopkGroups * i;
        if (ks < k_splits) {
          load(src + ks * n, v[i]);
        } else {
#pragma unroll
          for (int c = 0; c < kVec; ++c) v[i][c] = 0.0f;
        }
      }
#pragma unroll
      for (int c = 0; c < kVec; ++c) {
        float a = v[0][c];
#pragma unroll
        for (int i = 1; i < kTopkLoads; ++i) a += v[i][c];
        s_grp[g][e0 + c] = a;
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      float a = s_grp[0][e];
#pragma unroll
      for (int g = 1; g < kTopkGroups; ++g) a += s_grp[g][e];
      s_l[e] = a;
      if (logits) logits[(int64_t)t * E + e] = a;
    }
    __syncthreads();
    if (k > 0 && threadIdx.x < 32) route_topk_row<MAXPL>(s_l, t, E, k, idx, w, status);
    __syncthreads();
  }
}

// one warp per token
template <int MAXPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T,
                                                         int E, int k, int32_t* __restrict__ idx,
                                                         float* __restrict__ w, int* status) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int t = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (t < T) route_topk_token<MAXPL>(logits, t, E, k, idx, w, status);
}

// Router logits of the layers of a chain (host array copied into the launch)
struct LayerLogits {
  const float* p[MOE_MAX_CHAIN];
};

// step (1) of every layer of a chain in one launch: blockIdx.y = layer, whose
// routing block starts `stride` bytes after the previous layer's
template <int MAXPL>
__global__ void __launch_bounds__(256) route_topk_layers_kernel(
    const __grid_constant__ LayerLogits lg, int T, int E, int k, int32_t* __restrict__ idx0,
    float* __restrict__ w0, int64_t stride, int* status) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int t = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int64_t off = (int64_t)blockIdx.y * stride;
  if (t < T)
    route_topk_token<MAXPL>(lg.p[blockIdx.y], t, E, k,
                            reinterpret_cast<int32_t*>(reinterpret_cast<char*>(idx0) + off),
                            reinterpret_cast<float*>(reinterpret_cast<char*>(w0) + off), status);
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

// Chunk list of a routed block, by one 1024-thread CTA whose thread e < E
// holds expert e's count c and first slot excl: touched experts in ascending
// order, each split into ceil(n / chunk_max) chunks of near-equal size;
// meta[0] = chunks, meta[1] = touched experts.  kPacked: both prefix sums in
// one scan of (chunks | touched << 16) — exact while the block has fewer than
// 65536 chunks (the small-block kernel: at most 512 assignments).
template <bool kPacked = false>
__device__ __forceinline__ void route_chunk_list(int c, int excl, int E, int chunk_max,
                                                 int4* __restrict__ chunks, int max_chunks,
                                                 int32_t* __restrict__ meta, int* s_warp,
                                                 int* s_tot, int* status) {
  const int tid = threadIdx.x;
  const int nch = c > 0 ? (c + chunk_max - 1) / chunk_max : 0;
  int cbase;
  if (kPacked) {
    cbase = block_exclusive_scan_1024(nch | (c > 0 ? 1 << 16 : 0), s_warp, &s_tot[0]) & 0xFFFF;
  } else {
    cbase = block_exclusive_scan_1024(nch, s_warp, &s_tot[0]);
    block_exclusive_scan_1024(c > 0 ? 1 : 0, s_warp, &s_tot[1]);
  }
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
    meta[0] = min(kPacked ? s_tot[0] & 0xFFFF : s_tot[0], max_chunks);
    meta[1] = kPacked ? s_tot[0] >> 16 : s_tot[1];
  }
}

// assignments from which step (4) walks warp segments instead of rounds
// (full shape, T = 1024: 20.0 -> 16.9 us; at T = 256 the rounds are faster)
constexpr int kSegmentedPermute = 4096;

// Steps (2)-(4) by one CTA of 1024 threads: histogram, scan, stable
// permutation, chunk list.  Dynamic shared memory: (35 * E + 1 + 34) ints.
__device__ __forceinline__ void route_permute_cta(
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
  if (TK >= kSegmentedPermute) {
    // Step (4) for many assignments: warp w takes the contiguous segment
    // [w * seg, (w + 1) * seg) of the flat order.  Pass 1 counts each expert in
    // the warp's segment (the warp's own row of s_w, 32 assignments at a time,
    // one match per group of equal experts); an exclusive scan over the 32 rows
    // gives, per expert, its assignments in the earlier segments; pass 2 walks
    // the segment again and places each assignment after those, after the
    // earlier ones of its own segment (a running base) and after the equal ones
    // of lower lanes — the stable order of the flat index t*k + j, with two
    // block barriers instead of three per 1024 assignments.
    const int seg = (TK + 32 * 32 - 1) / (32 * 32) * 32;  // a multiple of 32
    const int f0 = warp * seg, f1 = min(TK, f0 + seg);
    int* my_w = s_w + warp * E;
    for (int e = lane; e < E; e += 32) my_w[e] = 0;
    __syncwarp();
    auto expert_at = [&](int f) {
      int e = f < f1 ? idx[f] : -1;
      if (f < f1 && (unsigned)e >= (unsigned)E) e = 0;  // flagged by the histogram above
      return e;
    };
    for (int b = f0; b < f1; b += 32) {
      const int e = expert_at(b + lane);
      const unsigned same = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && __popc(same & lt_mask) == 0) my_w[e] += __popc(same);
      __syncwarp();
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += 1024) {
      int run = 0;
      for (int w = 0; w < 32; ++w) {
        const int cw = s_w[w * E + ee];
        s_w[w * E + ee] = run;
        run += cw;
      }
    }
    __syncthreads();
    for (int b = f0; b < f1; b += 32) {
      const int f = b + lane;
      const int e = expert_at(f);
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(same & lt_mask);
      if (e >= 0) {
        const int slot = s_off[e] + my_w[e] + rank;
        perm[slot] = f / k;
        pos[f] = slot;
      }
      __syncwarp();
      if (e >= 0 && rank == 0) my_w[e] += __popc(same);
      __syncwarp();
    }
    __syncthreads();
  } else {
    // Step (4) in rounds of 1024 assignments: a thread each, ranks within the
    // round from one match per warp and a scan over the 32 warps per expert,
    // carried across rounds in s_run.
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
  }

  route_chunk_list(c, excl, E, chunk_max, chunks, max_chunks, meta, s_warp, s_tot, status);
}

__global__ void __launch_bounds__(1024) route_permute_kernel(
    const int32_t* __restrict__ idx, int T, int k, int E, int32_t* __restrict__ cnt_out,
    int32_t* __restrict__ off_out, int32_t* __restrict__ perm, int32_t* __restrict__ pos,
    int4* __restrict__ chunks, int max_chunks, int chunk_max, int32_t* __restrict__ meta,
    int32_t* __restrict__ done, int* status) {
  grid_dependency_wait();
  grid_launch_dependents();
  route_permute_cta(idx, T, k, E, cnt_out, off_out, perm, pos, chunks, max_chunks, chunk_max,
                    meta, done, status);
}

// steps (2)-(4) of every layer of a chain: one CTA per layer; each of the
// layer's arrays starts `stride` bytes after the previous layer's
__global__ void __launch_bounds__(1024) route_permute_layers_kernel(
    const int32_t* idx0, int T, int k, int E, int32_t* cnt0, int32_t* off0, int32_t* perm0,
    int32_t* pos0, int4* chunks0, int max_chunks, int chunk_max, int32_t* meta0, int32_t* done0,
    int64_t stride, int* status) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t off = (int64_t)blockIdx.x * stride;
  auto at = [off](auto* p) {
    using P = decltype(p);
    return reinterpret_cast<P>(reinterpret_cast<char*>(const_cast<void*>(
                                   static_cast<const void*>(p))) + off);
  };
  route_permute_cta(at(idx0), T, k, E, at(cnt0), at(off0), at(perm0), at(pos0), at(chunks0),
                    max_chunks, chunk_max, at(meta0), at(done0), status);
}

}  // namespace moe
