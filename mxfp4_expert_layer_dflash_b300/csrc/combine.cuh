// Deterministic gate-weighted combine back to token order:
//   y[t, :] = bf16_RNE( sum_{j=0..k-1} g[t, j] * yp[pos[t, j], :] ),
// accumulated in fp32 in the fixed slot order j = 0..k-1 (no atomics).
#pragma once

#include "common.cuh"
#include "fmt.cuh"

namespace moe {

// one thread per 8 consecutive outputs of a token
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ yp,
                                                      const int32_t* __restrict__ pos,
                                                      const float* __restrict__ gate, int T, int H,
                                                      int k, uint16_t* __restrict__ y) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t per_tok = H / 8;
  const int64_t total = (int64_t)T * per_tok;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / per_tok, h0 = (i % per_tok) * 8;
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
    for (int j = 0; j < k; ++j) {
      const int64_t p = pos[t * k + j];
      const float g = gate[t * k + j];
      const float4* src = reinterpret_cast<const float4*>(yp + p * H + h0);
      const float4 a = src[0], b = src[1];
      acc[0] = fmaf(g, a.x, acc[0]);
      acc[1] = fmaf(g, a.y, acc[1]);
      acc[2] = fmaf(g, a.z, acc[2]);
      acc[3] = fmaf(g, a.w, acc[3]);
      acc[4] = fmaf(g, b.x, acc[4]);
      acc[5] = fmaf(g, b.y, acc[5]);
      acc[6] = fmaf(g, b.z, acc[6]);
      acc[7] = fmaf(g, b.w, acc[7]);
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = (uint32_t)float_to_bf16_bits(acc[2 * q]) |
             ((uint32_t)float_to_bf16_bits(acc[2 * q + 1]) << 16);
    *reinterpret_cast<uint4*>(y + t * H + h0) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace moe
