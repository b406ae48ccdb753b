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
// Work split: the vocabulary of each sequence is cut into `chunks` ranges, one
// CTA each.  A CTA takes the (cheap, redundant) accept decision, sums its
// range's masses and publishes the sum; the last CTA of the sequence to arrive
// (an atomic counter, no waiting) finds the range that holds the threshold and
// scans only that range.  Reads: the chosen row(s) of the vocabulary once, plus
// one range again from L2.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kVerifyThreads = 512;
constexpr int kVerifyMaxChunks = 64;

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
  uint32_t* count;      // [S] ranges done (zero at the start of a call)
  int32_t* n_acc;       // [S]
  int32_t* tokens;      // [S, g+1]
  int* status;
};

// first rejected position of sequence s (g when all drafts are accepted); a
// drafted token outside the vocabulary is a rejection (and a fault)
__device__ __forceinline__ int verify_decision(const VerifyParams& P, int s) {
  for (int i = 0; i < P.g; ++i) {
    const int32_t d = P.draft[(int64_t)s * P.g + i];
    if (d < 0 || d >= P.V) {
      set_status(P.status, kStatusFault);
      return i;
    }
    const double lhs = (double)P.u[(int64_t)s * P.g + i] *
                       (double)P.q[((int64_t)s * P.g + i) * P.V + d];
    if (!(lhs < (double)P.p[((int64_t)s * (P.g + 1) + i) * P.V + d])) return i;
  }
  return P.g;
}

// fixed-point mass of token x in the distribution drawn from
__device__ __forceinline__ uint64_t verify_mass(const float* prow, const float* qrow, int64_t x) {
  float w = prow[x];
  if (qrow) {
    const float diff = __fsub_rn(w, qrow[x]);  // the fp32 difference, never contracted
    w = diff > 0.0f ? diff : 0.0f;
  }
  w = fminf(w, 2.0f);  // probabilities: keeps the conversion in range for any input
  return __double2ull_rz((double)w * 0x1p62);
}

__device__ __forceinline__ uint64_t block_sum_u64(uint64_t v, uint64_t* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  uint64_t t = 0;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kVerifyThreads / 32; ++w) t += red[w];
    red[0] = t;
  }
  __syncthreads();
  t = red[0];
  __syncthreads();
  return t;
}

// exclusive prefix of v over the block's threads (in thread order)
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
    for (int w = 0; w < kVerifyThreads / 32; ++w) {
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

__global__ void __launch_bounds__(kVerifyThreads) verify_kernel(const VerifyParams P) {
  __shared__ uint64_t red[kVerifyThreads / 32];
  __shared__ uint64_t csum[kVerifyMaxChunks];
  __shared__ int s_j, s_last, s_chunk;
  __shared__ unsigned long long s_t;
  __shared__ int64_t s_x;
  grid_dependency_wait();
  grid_launch_dependents();
  const int s = blockIdx.x / P.chunks, c = blockIdx.x % P.chunks;
  const int tid = threadIdx.x;
  if (tid == 0) s_j = verify_decision(P, s);
  __syncthreads();
  const int j = s_j;
  const float* prow = P.p + ((int64_t)s * (P.g + 1) + j) * P.V;
  const float* qrow = j < P.g ? P.q + ((int64_t)s * P.g + j) * P.V : nullptr;

  // this range's mass
  const int64_t x0 = (int64_t)c * P.chunk_len, x1 = min(P.V, x0 + P.chunk_len);
  uint64_t acc = 0;
  for (int64_t x = x0 + tid; x < x1; x += kVerifyThreads) acc += verify_mass(prow, qrow, x);
  acc = block_sum_u64(acc, red);
  if (tid == 0) {
    P.part[(int64_t)s * P.chunks + c] = acc;
    __threadfence();
    s_last = atomicAdd(&P.count[s], 1u) == (uint32_t)(P.chunks - 1);
  }
  __syncthreads();
  if (!s_last) return;

  // the last range of sequence s: every range's sum is published
  __threadfence();
  if (tid < P.chunks)
    csum[tid] = *reinterpret_cast<volatile const uint64_t*>(P.part + (int64_t)s * P.chunks + tid);
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
      const int64_t a = (int64_t)k * P.chunk_len, b = min(P.V, a + P.chunk_len);
      uint64_t v = 0;
      for (int64_t x = a + tid; x < b; x += kVerifyThreads) v += verify_mass(prow, nullptr, x);
      v = block_sum_u64(v, red);
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
    // scan range s_chunk: thread tid owns a contiguous piece of it
    const int64_t a = (int64_t)s_chunk * P.chunk_len, b = min(P.V, a + P.chunk_len);
    const int64_t piece = (b - a + kVerifyThreads - 1) / kVerifyThreads;
    const int64_t pa = min(b, a + tid * piece), pb = min(b, pa + piece);
    uint64_t mine = 0;
    for (int64_t x = pa; x < pb; ++x) mine += verify_mass(prow, qrow, x);
    const uint64_t before = block_excl_scan_u64(mine, red);
    const uint64_t t = s_t;
    if (t >= before && t < before + mine) {
      uint64_t run = before;
      for (int64_t x = pa; x < pb; ++x) {
        run += verify_mass(prow, qrow, x);
        if (run > t) {
          s_x = x;
          break;
        }
      }
    }
  }
  __syncthreads();
  if (tid <= P.g) {
    int32_t v = -1;
    if (tid < j) v = P.draft[(int64_t)s * P.g + tid];
    if (tid == j) v = (int32_t)s_x;
    P.tokens[(int64_t)s * (P.g + 1) + tid] = v;
  }
  if (tid == 0) P.n_acc[s] = j;
}

}  // namespace moe
