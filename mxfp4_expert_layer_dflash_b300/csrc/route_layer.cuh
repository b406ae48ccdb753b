// Steps a1-a4 inside the persistent layer kernel, for a block of T <= 32
// tokens (one DFlash verification block of up to 8 positions for up to four
// sequences: techllm.github.io, "2. DFlash"), so that the whole layer is one
// launch — the resident engine kernel of dothoosh.com, section "TileRT", which
// removes the gaps between operators that each last microseconds.
//
// Every CTA of the launch routes the whole block in its own shared memory with
// its 384 threads (the same arrays, bit for bit, as the standalone routing
// kernels: the shared top-k device code, then counts, one scan over experts,
// each assignment's rank within its expert as a direct count of the earlier
// ones, and the chunk list), so no CTA waits for another to start streaming
// weights.  What the GEMM roles need afterwards stays in shared memory: the
// chunk list (packed in one word per chunk), each assignment's slot and gate,
// each slot's token.  CTA 0 also publishes the routing arrays to global
// memory, where the caller's workspace keeps them for inspection.
//
// Step a4 is done per CTA for the chunks of its own GEMM1 work items
// (layer_act1_rows): a chunk's slot rows are quantised by every CTA that
// multiplies them, each writing the same bytes, so a CTA only waits for its
// own writes before its copies read them — no grid-wide barrier.
#pragma once

#include "common.cuh"
#include "quant.cuh"
#include "route.cuh"
#include "route_small.cuh"

namespace moe {

constexpr int kLayerThreads = 384;  // = kTcThreads: the GEMM kernel's CTA
constexpr int kLayerMaxTK = kSmallRouteTokens * MOE_MAX_K;  // 512 assignments
// chunk list bound of a block (min(E, T*k) + T*k / 32 + 1)
constexpr int kLayerMaxChunks = kLayerMaxTK + kLayerMaxTK / 32 + 1;

// Packed chunk: expert (10 bits), first slot (9 bits), slot count (6 bits);
// exact for E <= 1024, T*k <= 512 and chunks of at most 32 slots.
__device__ __forceinline__ uint32_t pack_chunk(int e, int first, int n) {
  return (uint32_t)e | ((uint32_t)first << 10) | ((uint32_t)n << 19);
}
__device__ __forceinline__ int4 unpack_chunk(uint32_t v) {
  return make_int4((int)(v & 1023u), (int)((v >> 10) & 511u), (int)(v >> 19), 0);
}

// What the layer kernel keeps from its own routing (in its shared memory)
struct LayerRouteState {
  uint32_t chunks[kLayerMaxChunks];
  int32_t pos[kLayerMaxTK];   // (t*k + j) -> slot
  float gate[kLayerMaxTK];    // g[t, j]
  uint8_t perm[kLayerMaxTK];  // slot -> token (T <= 32)
  int n_chunks;
  int pad[3];
};

// Inputs and global outputs of the in-kernel routing
struct LayerRouteParams {
  const float* logits;  // [T, E] (written by the launch itself when w_router is given)
  const uint16_t* x;    // [T, H] bf16
  const uint16_t* w_router;  // [E, H] bf16 router weights, or null: logits are an input
  int T, E, k, chunk_max, max_chunks;  // T = 0: routing is not done in the kernel
  // published by CTA 0 (the forward's workspace)
  int32_t* topk_idx;
  float* topk_w;
  int32_t* cnt;
  int32_t* off;
  int32_t* perm;
  int32_t* pos;
  int4* chunks;
  int32_t* meta;
  uint8_t* xq;    // [T*k, H] act1 codes in slot order (E4M3)
  uint8_t* xs;    // [T*k, H/32] their E8M0 scales
};

// exclusive prefix sum over the 384 threads' values (all threads call it)
__device__ __forceinline__ int block_exclusive_scan_384(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kLayerThreads / 32;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int wv = lane < kWarps ? s_warp[lane] : 0;
    int wx = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wx, o);
      if (lane >= o) wx += y;
    }
    if (lane < kWarps) s_warp[lane] = wx - wv;
    if (lane == 31) *total = wx;
  }
  __syncthreads();
  const int r = s_warp[warp] + x - v;
  __syncthreads();
  return r;
}

// Routing of the block by this CTA (384 threads, all call it).  `scratch`:
// at least layer_route_scratch_bytes(E) bytes of shared memory that is free
// during the call (the GEMM's stage buffers, before their first copy).
__host__ __device__ inline size_t layer_route_scratch_bytes(int E) {
  return (size_t)(64 + 2 * kLayerMaxTK + kLayerMaxTK + 2 * (E + 1) + 8) * sizeof(int);
}

__device__ __forceinline__ void layer_route_block(const LayerRouteParams& r, uint8_t* scratch,
                                                  LayerRouteState* st, bool publish,
                                                  int* status) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int T = r.T, E = r.E, k = r.k, TK = T * k;
  int* s_warp = reinterpret_cast<int*>(scratch);  // 32 + 2 ints of scan scratch
  int* s_tot = s_warp + 32;
  int32_t* s_idx = s_warp + 64;                   // [kLayerMaxTK]
  float* s_w = reinterpret_cast<float*>(s_idx + kLayerMaxTK);
  int32_t* s_perm = s_idx + 2 * kLayerMaxTK;      // [kLayerMaxTK]
  int32_t* s_cnt = s_perm + kLayerMaxTK;          // [E]
  int32_t* s_off = s_cnt + E + 1;                 // [E + 1]

  // (1) top-k + softmax: warp w takes tokens w, w + 12, w + 24 (logits the
  // launch computed itself are read from L2)
  for (int t = warp; t < T; t += kLayerThreads / 32) {
    if (r.w_router) {
      if (E <= 128)
        route_topk_token<4, true>(r.logits, t, E, k, s_idx, s_w, status);
      else if (E <= 384)
        route_topk_token<12, true>(r.logits, t, E, k, s_idx, s_w, status);
      else
        route_topk_token<32, true>(r.logits, t, E, k, s_idx, s_w, status);
    } else {
      if (E <= 128)
        route_topk_token<4>(r.logits, t, E, k, s_idx, s_w, status);
      else if (E <= 384)
        route_topk_token<12>(r.logits, t, E, k, s_idx, s_w, status);
      else
        route_topk_token<32>(r.logits, t, E, k, s_idx, s_w, status);
    }
  }
  for (int e = tid; e < E; e += kLayerThreads) s_cnt[e] = 0;
  __syncthreads();
  // (2) counts
  for (int f = tid; f < TK; f += kLayerThreads) {
    int e = s_idx[f];
    if ((unsigned)e >= (unsigned)E) {  // never from the top-k; kept as a guard
      set_status(status, kStatusFault);
      e = 0;
      s_idx[f] = 0;
    }
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  // (3) offsets: thread i owns experts [i * per, (i + 1) * per)
  const int per = (E + kLayerThreads - 1) / kLayerThreads;  // <= 3
  const int e0 = tid * per;
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (e0 + i < E) local += s_cnt[e0 + i];
  int run = block_exclusive_scan_384(local, s_warp, &s_tot[0]);
  for (int i = 0; i < per; ++i) {
    if (e0 + i < E) {
      s_off[e0 + i] = run;
      run += s_cnt[e0 + i];
    }
  }
  if (tid == 0) s_off[E] = TK;
  __syncthreads();
  // (4) slot of each assignment: its expert's offset + the number of earlier
  // assignments to the same expert (ascending t*k + j within an expert)
  for (int f = tid; f < TK; f += kLayerThreads) {
    const int e = s_idx[f];
    const int4* v4 = reinterpret_cast<const int4*>(s_idx);
    int rk = 0;
#pragma unroll 4
    for (int g = 0; g < (f >> 2); ++g) {
      const int4 v = v4[g];
      rk += (v.x == e) + (v.y == e) + (v.z == e) + (v.w == e);
    }
    for (int g = f & ~3; g < f; ++g) rk += s_idx[g] == e;
    const int slot = s_off[e] + rk;
    st->pos[f] = slot;
    st->gate[f] = s_w[f];
    s_perm[slot] = f / k;
    st->perm[slot] = (uint8_t)(f / k);
  }
  // chunk list: touched experts in ascending order, each cut into
  // ceil(n / chunk_max) near-equal chunks (the standalone kernels' rule)
  int nch_local = 0, touched_local = 0;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    const int c = e < E ? s_cnt[e] : 0;
    nch_local += c > 0 ? (c + r.chunk_max - 1) / r.chunk_max : 0;
    touched_local += c > 0;
  }
  int cbase = block_exclusive_scan_384(nch_local | (touched_local << 16), s_warp, &s_tot[0]) &
              0xFFFF;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    const int c = e < E ? s_cnt[e] : 0;
    if (c == 0) continue;
    const int nch = (c + r.chunk_max - 1) / r.chunk_max;
    const int q = (c + nch - 1) / nch;
    for (int j = 0; j < nch; ++j) {
      const int b = cbase + j;
      if (b < kLayerMaxChunks && b < r.max_chunks)
        st->chunks[b] = pack_chunk(e, s_off[e] + j * q, min(q, c - j * q));
      else
        set_status(status, kStatusFault);
    }
    cbase += nch;
  }
  if (tid == 0) st->n_chunks = min(s_tot[0] & 0xFFFF, min(r.max_chunks, kLayerMaxChunks));
  __syncthreads();
  if (publish) {
    for (int i = tid; i < TK; i += kLayerThreads) {
      r.topk_idx[i] = s_idx[i];
      r.topk_w[i] = s_w[i];
      r.perm[i] = s_perm[i];
      r.pos[i] = st->pos[i];
    }
    for (int e = tid; e <= E; e += kLayerThreads) {
      if (e < E) r.cnt[e] = s_cnt[e];
      r.off[e] = s_off[e];
    }
    for (int c = tid; c < st->n_chunks; c += kLayerThreads) r.chunks[c] = unpack_chunk(st->chunks[c]);
    if (tid == 0) {
      r.meta[0] = st->n_chunks;
      r.meta[1] = s_tot[0] >> 16;
    }
  }
}

// The router in front of the routing (logits = x W_r^T with bf16 W_r, read as
// a plain linear layer; expert routing is part of the pipeline the runtime is
// built around: techllm.github.io, "3. TileRT").  CTA c takes experts
// [c E / G, (c + 1) E / G); its threads split H into runs of 16 elements,
// each thread multiplying its runs of the experts' weight rows with the same
// runs of up to 8 token rows at a time (exact bf16 products, fp32 sums in
// ascending element order, every load of a run independent of the others),
// then the threads' sums are added by a fixed butterfly within each warp and
// the warps' in warp order.  Deterministic; the order differs from the
// standalone router's tensor-core sums, within the same error bound.
// `s_part`: 12 x 8 x 4 floats of shared memory.  All threads call it.
constexpr int kRouterTok = 8, kRouterExp = 4;
__device__ __forceinline__ void layer_router_logits(const LayerRouteParams& r, int64_t H,
                                                    float* __restrict__ logits,
                                                    float* __restrict__ s_part) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kLayerThreads / 32;
  const int G = (int)gridDim.x, c = (int)blockIdx.x, E = r.E, T = r.T;
  const int e_begin = (int)((int64_t)c * E / G), e_end = (int)((int64_t)(c + 1) * E / G);
  const int runs = (int)(H / 16);
  for (int eg = e_begin; eg < e_end; eg += kRouterExp) {
    const int ne = min(kRouterExp, e_end - eg);
    for (int tg = 0; tg < T; tg += kRouterTok) {
      const int nt = min(kRouterTok, T - tg);
      float acc[kRouterTok][kRouterExp];
#pragma unroll
      for (int t = 0; t < kRouterTok; ++t)
#pragma unroll
        for (int e = 0; e < kRouterExp; ++e) acc[t][e] = 0.0f;
      for (int run = tid; run < runs; run += kLayerThreads) {
        uint4 wv[kRouterExp][2], xv[kRouterTok][2];
#pragma unroll
        for (int e = 0; e < kRouterExp; ++e) {
          if (e < ne) {
            const uint4* src = reinterpret_cast<const uint4*>(r.w_router + (int64_t)(eg + e) * H) +
                               2 * run;
            wv[e][0] = src[0];
            wv[e][1] = src[1];
          }
        }
#pragma unroll
        for (int t = 0; t < kRouterTok; ++t) {
          if (t < nt) {
            const uint4* src = reinterpret_cast<const uint4*>(r.x + (int64_t)(tg + t) * H) + 2 * run;
            xv[t][0] = src[0];
            xv[t][1] = src[1];
          }
        }
#pragma unroll
        for (int t = 0; t < kRouterTok; ++t) {
#pragma unroll
          for (int e = 0; e < kRouterExp; ++e) {
            if (t < nt && e < ne) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t ww[4] = {wv[e][h].x, wv[e][h].y, wv[e][h].z, wv[e][h].w};
                const uint32_t xx[4] = {xv[t][h].x, xv[t][h].y, xv[t][h].z, xv[t][h].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  acc[t][e] = fmaf(__uint_as_float(ww[j] << 16), __uint_as_float(xx[j] << 16),
                                   acc[t][e]);
                  acc[t][e] = fmaf(__uint_as_float(ww[j] & 0xFFFF0000u),
                                   __uint_as_float(xx[j] & 0xFFFF0000u), acc[t][e]);
                }
              }
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kRouterTok; ++t) {
#pragma unroll
        for (int e = 0; e < kRouterExp; ++e) {
          float v = acc[t][e];
#pragma unroll
          for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) s_part[(warp * kRouterTok + t) * kRouterExp + e] = v;
        }
      }
      __syncthreads();
      if (tid < nt * ne) {
        const int t = tid / ne, e = tid - t * ne;
        float v = 0.0f;
        for (int w = 0; w < kWarps; ++w) v += s_part[(w * kRouterTok + t) * kRouterExp + e];
        logits[(int64_t)(tg + t) * E + eg + e] = v;
      }
      __syncthreads();
    }
  }
}

// Step a4 for slot row `slot` of token t, blocks sg*32 .. sg*32+31 of 32
// along H (a block per lane): MXFP8 codes and scale into xq/xs, the rule of
// the standalone activation kernels.  One warp.
__device__ __forceinline__ void layer_act1_unit(const uint16_t* __restrict__ x, int t, int slot,
                                                int sg, int64_t H, uint8_t* __restrict__ xq,
                                                uint8_t* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = H / 32, b = (int64_t)sg * 32 + lane;
  if (b >= nb) return;
  float v[32];
  uint8_t c[32];
  load_bf16x32(x + (int64_t)t * H + b * 32, v);
  const int code = mxfp8_block(v, c);
  store_u8x32(xq + (int64_t)slot * H + b * 32, c);
  xs[(int64_t)slot * nb + b] = (uint8_t)code;
}

}  // namespace moe
