// Rejection-sampling verification of a block of drafted tokens per sequence,
// the step after the verify forward (lossless speculative decoding:
// techllm.github.io, "Xiaomi MiMo and TileRT ...", section "2. DFlash"; blocks
// of at most 8 positions: dothoosh.com, section "جزئیات پیاده‌سازی DFlash").
//
// For sequence s with drafted tokens d_0..d_{g-1}, draft distributions q_i and
// target distributions p_0..p_g:
//   d_i is accepted while u_i * q_i(d_i) < p_i(d_i) (the fp32 values compared
//   exactly, in fp64);
//   at the first rejection i a token is drawn from max(0, p_i - q_i), after g
//   acceptances from p_g (from p_i itself if the residual has no mass).
// Draws are inverse CDFs over fixed-point masses m(x) = floor(w(x) * 2^62):
// with M = sum m and the sequence's 64-bit uniform U, the token is the first x
// whose running sum exceeds floor(U * M / 2^64).  The masses are exact
// integers, so the result does not depend on the order of any sum.
//
// Two kernels.  verify_decide_kernel: one warp per sequence takes the accept
// decisions (a lane per position, a ballot finds the first rejection).
// verify_draw_kernel: the vocabulary of each sequence is cut into ranges of
// 2048 tokens, one CTA each; a CTA sums its range's masses and publishes the
// sum, and the last CTA of the sequence to arrive (an atomic counter, no
// waiting) finds the range that holds the threshold and scans only that range.
// Reads: the chosen row(s) once, plus one range again from L2.  No FP64
// arithmetic: the masses come from the fp32 bits.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kVerifyMaxChunks = 1024;  // ranges per sequence: V <= 2^21 tokens

struct VerifyParams {
  const float* p;       // [S, g+1, V]
  const float* q;       // [S, g, V]
  const int32_t* draft; // [S, g]
  const float* u;       // [S, g]
  const uint64_t* U;    // [S]
  int S, g;
  int64_t V;
  int chunks;           // vocabulary ranges per sequence
  int64_t chunk_len;
  uint64_t* part;       // [S, chunks] range mass sums
  uint32_t* count;      // [S] ranges done (cleared by the decision step)
  int32_t* n_acc;       // [S]
  int32_t* tokens;      // [S, g+1]
  int* status;
};

// First rejected position of sequence s (g when all drafts are accepted),
// evaluated by one warp: lane i tests position i (all loads in flight at
// once), a ballot finds the first failure.  A drafted token outside the
// vocabulary is a rejection (and a fault), checked before any read.
__device__ __forceinline__ int verify_decision_warp(const VerifyParams& P, int s) {
  const int lane = threadIdx.x & 31;
  for (int base = 0; base < P.g; base += 32) {
    const int i = base + lane;
    bool reject = false;
    if (i < P.g) {
      const int32_t d = P.draft[(int64_t)s * P.g + i];
      if (d < 0 || d >= P.V) {
        set_status(P.status, kStatusFault);
        reject = true;
      } else {
        const double lhs = (double)P.u[(int64_t)s * P.g + i] *
                           (double)P.q[((int64_t)s * P.g + i) * P.V + d];
        reject = !(lhs < (double)P.p[((int64_t)s * (P.g + 1) + i) * P.V + d]);
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, reject);
    if (m) return base + __ffs(m) - 1;
  }
  return P.g;
}

// floor(w * 2^62) of an fp32 w in [0, 2], from its bits in integer arithmetic
// (no FP64: the significand 1.m * 2^23 shifted by the exponent - 127 + 62 - 23;
// subnormals give 0).  Negative, NaN or larger inputs are clamped to [0, 2].
__device__ __forceinline__ uint64_t fixed_mass(float w) {
  w = fminf(fmaxf(w, 0.0f), 2.0f);
  const uint32_t bits = __float_as_uint(w);
  const int e = (int)(bits >> 23);
  if (e == 0) return 0;
  const uint64_t mant = (uint64_t)((bits & 0x7FFFFFu) | 0x800000u);
  const int sh = e - 88;
  return sh >= 0 ? mant << sh : (sh > -64 ? mant >> -sh : 0);
}

// weight of token x in the distribution drawn from: p(x), or the fp32
// difference max(0, p(x) - q(x)) (never contracted with anything)
__device__ __forceinline__ float verify_weight(float pv, float qv, bool residual) {
  if (!residual) return pv;
  const float diff = __fsub_rn(pv, qv);
  return diff > 0.0f ? diff : 0.0f;
}

__device__ __forceinline__ uint64_t verify_mass(const float* prow, const float* qrow, int64_t x) {
  return fixed_mass(verify_weight(prow[x], qrow ? qrow[x] : 0.0f, qrow != nullptr));
}

// Block-wide sum / exclusive prefix of one uint64 per thread (thread order).
template <int kThreads>
__device__ __forceinline__ uint64_t block_sum_u64(uint64_t v, uint64_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t t = 0;
    for (int w = 0; w < kThreads / 32; ++w) t += red[w];
    red[kThreads / 32] = t;
  }
  __syncthreads();
  const uint64_t t = red[kThreads / 32];
  __syncthreads();
  return t;
}

template <int kThreads>
__device__ __forceinline__ uint64_t block_excl_scan_u64(uint64_t v, uint64_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) red[warp] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t run = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      const uint64_t t = red[w];
      red[w] = run;
      run += t;
    }
  }
  __syncthreads();
  const uint64_t r = red[warp] + x - v;
  __syncthreads();
  return r;
}

// Step 1, one warp per sequence: the accept decisions.  Writes the first
// rejected position j (g if none) to jpos, n_acc = j, the accepted drafts to
// tokens[s, 0..j-1] and -1 past position j (tokens[s, j] comes from step 2),
// and clears the sequence's arrival counter for step 2.
__global__ void __launch_bounds__(256) verify_decide_kernel(const VerifyParams P,
                                                            int32_t* __restrict__ jpos) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int s = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (s >= P.S) return;
  const int j = verify_decision_warp(P, s);
  for (int i = lane; i <= P.g; i += 32) {
    if (i < j) P.tokens[(int64_t)s * (P.g + 1) + i] = P.draft[(int64_t)s * P.g + i];
    if (i > j) P.tokens[(int64_t)s * (P.g + 1) + i] = -1;
  }
  if (lane == 0) {
    jpos[s] = j;
    P.n_acc[s] = j;
    P.count[s] = 0;
  }
}

// Step 2: CTA (s, c) holds the masses of tokens [c*L, c*L + L) of sequence s's
// chosen distribution (L = kVerifyRange: 8 consecutive tokens per thread, from
// 16-byte loads when the rows allow), publishes their sum, and the last CTA of
// the sequence to arrive draws the token.
constexpr int kVerifyDrawThreads = 256;
constexpr int kVerifyPerThread = 8;
constexpr int kVerifyRange = kVerifyDrawThreads * kVerifyPerThread;

// masses of the 8 tokens x0 .. x0+7 (0 past the vocabulary)
__device__ __forceinline__ void verify_masses8(const float* prow, const float* qrow, int64_t x0,
                                               int64_t V, bool vec, uint64_t (&m)[8]) {
  float pv[8], qv[8];
  if (vec && x0 + 8 <= V) {
    const float4 a0 = *reinterpret_cast<const float4*>(prow + x0);
    const float4 a1 = *reinterpret_cast<const float4*>(prow + x0 + 4);
    pv[0] = a0.x; pv[1] = a0.y; pv[2] = a0.z; pv[3] = a0.w;
    pv[4] = a1.x; pv[5] = a1.y; pv[6] = a1.z; pv[7] = a1.w;
    if (qrow) {
      const float4 b0 = *reinterpret_cast<const float4*>(qrow + x0);
      const float4 b1 = *reinterpret_cast<const float4*>(qrow + x0 + 4);
      qv[0] = b0.x; qv[1] = b0.y; qv[2] = b0.z; qv[3] = b0.w;
      qv[4] = b1.x; qv[5] = b1.y; qv[6] = b1.z; qv[7] = b1.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      pv[e] = x0 + e < V ? prow[x0 + e] : 0.0f;
      qv[e] = (qrow && x0 + e < V) ? qrow[x0 + e] : 0.0f;
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e)
    m[e] = x0 + e < V ? fixed_mass(verify_weight(pv[e], qv[e], qrow != nullptr)) : 0;
}

__global__ void __launch_bounds__(kVerifyDrawThreads)
    verify_draw_kernel(const VerifyParams P, const int32_t* __restrict__ jpos) {
  __shared__ uint64_t red[kVerifyDrawThreads / 32 + 1];
  __shared__ uint64_t csum[kVerifyMaxChunks];
  __shared__ int s_last, s_chunk;
  __shared__ unsigned long long s_t;
  __shared__ int64_t s_x;
  grid_dependency_wait();
  grid_launch_dependents();
  const int s = blockIdx.x / P.chunks, c = blockIdx.x % P.chunks;
  const int tid = threadIdx.x;
  const int j = jpos[s];
  const float* prow = P.p + ((int64_t)s * (P.g + 1) + j) * P.V;
  const float* qrow = j < P.g ? P.q + ((int64_t)s * P.g + j) * P.V : nullptr;
  const bool vec = P.V % 4 == 0;

  uint64_t m[8];
  verify_masses8(prow, qrow, (int64_t)c * kVerifyRange + tid * kVerifyPerThread, P.V, vec, m);
  uint64_t mine = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) mine += m[e];
  const uint64_t total = block_sum_u64<kVerifyDrawThreads>(mine, red);
  if (tid == 0) {
    P.part[(int64_t)s * P.chunks + c] = total;
    __threadfence();
    s_last = atomicAdd(&P.count[s], 1u) == (uint32_t)(P.chunks - 1);
  }
  __syncthreads();
  if (!s_last) return;

  // the last range of sequence s to arrive: every range's sum is published
  __threadfence();
  for (int k = tid; k < P.chunks; k += kVerifyDrawThreads)
    csum[k] = *reinterpret_cast<volatile const uint64_t*>(P.part + (int64_t)s * P.chunks + k);
  __syncthreads();
  if (tid == 0) {
    uint64_t M = 0;
    for (int k = 0; k < P.chunks; ++k) M += csum[k];
    s_t = M;
  }
  __syncthreads();
  if (s_t == 0 && qrow) {
    // no residual mass (p_j <= q_j everywhere in fp32): draw from p_j itself
    qrow = nullptr;
    for (int k = 0; k < P.chunks; ++k) {
      uint64_t mk[8];
      verify_masses8(prow, nullptr, (int64_t)k * kVerifyRange + tid * kVerifyPerThread, P.V,
                     vec, mk);
      uint64_t v = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) v += mk[e];
      v = block_sum_u64<kVerifyDrawThreads>(v, red);
      if (tid == 0) csum[k] = v;
    }
    __syncthreads();
    if (tid == 0) {
      uint64_t M = 0;
      for (int k = 0; k < P.chunks; ++k) M += csum[k];
      s_t = M;
    }
    __syncthreads();
  }
  if (tid == 0) {
    const uint64_t M = s_t;
    const uint64_t t = __umul64hi(P.U[s], M);  // floor(U * M / 2^64) < M
    uint64_t run = 0;
    int k = 0;
    for (; k < P.chunks - 1; ++k) {
      if (run + csum[k] > t) break;
      run += csum[k];
    }
    s_chunk = M == 0 ? -1 : k;
    s_t = t - run;  // threshold inside range k
    s_x = 0;
  }
  __syncthreads();
  if (s_chunk >= 0) {
    const int64_t x0 = (int64_t)s_chunk * kVerifyRange + tid * kVerifyPerThread;
    if (s_chunk != c || qrow == nullptr) {
      verify_masses8(prow, qrow, x0, P.V, vec, m);  // range k from L2 (or the fallback rows)
      mine = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) mine += m[e];
    }
    const uint64_t before = block_excl_scan_u64<kVerifyDrawThreads>(mine, red);
    const uint64_t t = s_t;
    if (t >= before && t < before + mine) {
      uint64_t run = before;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        run += m[e];
        if (run > t) {
          s_x = x0 + e;
          break;
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) P.tokens[(int64_t)s * (P.g + 1) + j] = (int32_t)s_x;
}

}  // namespace moe
