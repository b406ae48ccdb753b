// Deterministic gate-weighted combine back to token order:
//   y[t, :] = bf16_RNE( sum_{j=0..k-1} g[t, j] * yp[pos[t, j], :] ),
// accumulated in fp32 in the fixed slot order j = 0..k-1 (no atomics).
#pragma once

#include "common.cuh"
#include "fmt.cuh"

namespace moe {

// slot rows loaded per round trip of a combine thread
constexpr int kCombineBatch = 4;

// sum_j g[t, j] * yp[pos[t, j], h0 .. h0+3] in fp32, j = 0..k-1 in order (one
// fmaf per term from 0); kCombineBatch rows' loads are issued before their
// multiply-adds so a thread waits for k / kCombineBatch round trips, not k
// kL2: load yp from L2 only (rows written by other CTAs of the same launch)
template <bool kL2 = false>
__device__ __forceinline__ float4 combine4(const float* __restrict__ yp,
                                           const int32_t* __restrict__ pos,
                                           const float* __restrict__ gate, int64_t t, int64_t H,
                                           int k, int64_t h0) {
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int j0 = 0; j0 < k; j0 += kCombineBatch) {
    float4 v[kCombineBatch];
    float g[kCombineBatch];
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      if (j0 + u < k) {
        g[u] = gate[t * k + j0 + u];
        const float4* src =
            reinterpret_cast<const float4*>(yp + (int64_t)pos[t * k + j0 + u] * H + h0);
        v[u] = kL2 ? __ldcg(src) : *src;
      }
    }
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      if (j0 + u < k) {
        acc.x = fmaf(g[u], v[u].x, acc.x);
        acc.y = fmaf(g[u], v[u].y, acc.y);
        acc.z = fmaf(g[u], v[u].z, acc.z);
        acc.w = fmaf(g[u], v[u].w, acc.w);
      }
    }
  }
  return acc;
}

__device__ __forceinline__ uint2 bf16x4_bits(float4 a) {
  return make_uint2((uint32_t)float_to_bf16_bits(a.x) | ((uint32_t)float_to_bf16_bits(a.y) << 16),
                    (uint32_t)float_to_bf16_bits(a.z) | ((uint32_t)float_to_bf16_bits(a.w) << 16));
}

// one thread per 4 consecutive outputs of a token
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ yp,
                                                      const int32_t* __restrict__ pos,
                                                      const float* __restrict__ gate, int T, int H,
                                                      int k, uint16_t* __restrict__ y) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t per_tok = H / 4;
  const int64_t total = (int64_t)T * per_tok;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / per_tok, h0 = (i - t * per_tok) * 4;
    *reinterpret_cast<uint2*>(y + t * H + h0) = bf16x4_bits(combine4(yp, pos, gate, t, H, k, h0));
  }
}

// A chain of layers (several expert layers back to back over one token
// block, the pipeline kept resident instead of launched operator by operator:
// dothoosh.com, section "TileRT"): layer l's combine fused with layer l+1's
// activation step.  Per token t:
//   x' = bf16_RNE( sum_j g[t, j] * yp[pos[t, j], :]  (+ x_res[t, :]) )
// in the combine's fp32 order (the residual added last), written to x_out
// when given and, when pos_next is given, straight into layer l+1's slot rows
// pos_next[t, j'] (j' < k): MXFP8 codes + scales (kMxfp8) or bf16 copies.
// One thread per 4 outputs, so the 8 lanes 8m..8m+7 of a warp hold one block
// of 32 (H % 128 == 0: a warp never straddles tokens); the block's amax is a
// 3-step shuffle reduction and each lane encodes its own 4 values, the same
// scale and codes as the standalone MXFP8 step.  Unit i = 4 outputs of one
// token; all 32 lanes of a warp must call it (with 32 consecutive units).
// kL2: yp rows written by other CTAs of the same launch (loaded from L2).
template <bool kMxfp8, bool kL2 = false>
__device__ __forceinline__ void combine_next_unit(
    int64_t i, const float* __restrict__ yp, const int32_t* __restrict__ pos,
    const float* __restrict__ gate, int T, int64_t H, int k, const uint16_t* __restrict__ x_res,
    uint16_t* __restrict__ x_out, const int32_t* __restrict__ pos_next,
    uint8_t* __restrict__ q_next, uint8_t* __restrict__ s_next, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t per_tok = H / 4, nb = H / 32, slots = (int64_t)T * k;
  const int64_t t = i / per_tok, h0 = (i - t * per_tok) * 4;
  float4 a = combine4<kL2>(yp, pos, gate, t, H, k, h0);
  if (x_res) {
    const uint2 r = *reinterpret_cast<const uint2*>(x_res + t * H + h0);
    a.x += __uint_as_float(r.x << 16);
    a.y += __uint_as_float(r.x & 0xFFFF0000u);
    a.z += __uint_as_float(r.y << 16);
    a.w += __uint_as_float(r.y & 0xFFFF0000u);
  }
  const uint2 bits = bf16x4_bits(a);
  if (x_out) *reinterpret_cast<uint2*>(x_out + t * H + h0) = bits;
  if (!pos_next) return;
  uint32_t codes = 0;
  int code = 0;
  if (kMxfp8) {
    const float v[4] = {__uint_as_float(bits.x << 16), __uint_as_float(bits.x & 0xFFFF0000u),
                        __uint_as_float(bits.y << 16), __uint_as_float(bits.y & 0xFFFF0000u)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    code = block_scale_code(amax, 8);
    const float inv = exp2_exact(127 - code);
#pragma unroll
    for (int q = 0; q < 4; ++q) codes |= (uint32_t)e4m3_encode_satfinite(v[q] * inv) << (8 * q);
  }
  const int my_slot = lane < k ? pos_next[t * k + lane] : 0;  // one round trip for k slots
  for (int j = 0; j < k; ++j) {
    const int64_t slot = __shfl_sync(0xffffffffu, my_slot, j);
    if (slot < 0 || slot >= slots) {
      set_status(status, kStatusFault);
      continue;
    }
    if (kMxfp8) {
      *reinterpret_cast<uint32_t*>(q_next + slot * H + h0) = codes;
      if ((lane & 7) == 0) s_next[slot * nb + h0 / 32] = (uint8_t)code;
    } else {
      *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(q_next) + slot * H + h0) = bits;
    }
  }
}

template <bool kMxfp8>
__global__ void __launch_bounds__(256) combine_next_kernel(
    const float* __restrict__ yp, const int32_t* __restrict__ pos,
    const float* __restrict__ gate, int T, int H, int k, const uint16_t* __restrict__ x_res,
    uint16_t* __restrict__ x_out, const int32_t* __restrict__ pos_next,
    uint8_t* __restrict__ q_next, uint8_t* __restrict__ s_next, int* status) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t total = (int64_t)T * (H / 4);  // a multiple of 32: whole warps
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x)
    combine_next_unit<kMxfp8>(i, yp, pos, gate, T, H, k, x_res, x_out, pos_next, q_next, s_next,
                              status);
}

}  // namespace moe
