// Grouped expert GEMMs on CUDA cores (first correct path).
//
// GEMM1: for each chunk of expert e's slots, gate/up = W13_e . x_slot, then
//        h = silu(gate) * up, requantized to MXFP8 along I (blocks of 32) or
//        rounded to bf16.
// GEMM2: yp[slot] = W2_e . h_slot (fp32).
// Weights are decoded on the fly from E2M1 + E8M0 (one 16-byte load = one
// block of 32 elements).
#pragma once

#include "common.cuh"
#include "fmt.cuh"

namespace moe {

constexpr int kSimtRows = 32;  // rows per work item (one MXFP8 block of h)
constexpr int kSimtTok = 8;    // tokens per register group

__device__ __forceinline__ void decode_fp4x32(uint4 q, uint32_t scale, float* out) {
  const float s = e8m0_decode(scale);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) out[8 * i + j] = e2m1_decode((w[i] >> (4 * j)) & 0xFu) * s;
}

// dot of 32 decoded weights with activation block b of slot row `row`
template <int ACT>
__device__ __forceinline__ float act_dot32(const float* wv, const uint8_t* act, const uint8_t* sc,
                                           int64_t row, int64_t K, int64_t b) {
  float acc = 0.0f;
  if (ACT == MOE_ACT_MXFP8) {
    const uint4* p = reinterpret_cast<const uint4*>(act + row * K + b * 32);
    uint4 q0 = p[0], q1 = p[1];
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc += wv[4 * i + j] * e4m3_decode((w[i] >> (8 * j)) & 0xFFu);
    acc *= e8m0_decode(sc[row * (K / 32) + b]);
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(act + (row * K + b * 32) * 2);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 q = p[i];
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc += wv[8 * i + 2 * j] * __uint_as_float(w[j] << 16);
        acc += wv[8 * i + 2 * j + 1] * __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
  }
  return acc;
}

template <int ACT>
__global__ void __launch_bounds__(128) gemm1_simt_kernel(
    const uint8_t* __restrict__ w13, const uint8_t* __restrict__ w13s,
    const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xs, const int4* __restrict__ chunks,
    const int32_t* __restrict__ meta, int H, int I, uint8_t* __restrict__ hq,
    uint8_t* __restrict__ hs) {
  __shared__ float hbuf[kSimtRows][kChunkNarrow];  // bf16 mode always uses narrow chunks
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int iblocks = I / kSimtRows;
  const int64_t items = (int64_t)meta[0] * iblocks;
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int4 ch = chunks[it / iblocks];
    const int ib = (int)(it % iblocks);
    const int e = ch.x, s0 = ch.y, n = ch.z;
    for (int r = warp * 8; r < warp * 8 + 8; ++r) {
      const int64_t gr = (int64_t)e * 2 * I + ib * kSimtRows + r, ur = gr + I;
      for (int g0 = 0; g0 < n; g0 += kSimtTok) {
        float ag[kSimtTok], au[kSimtTok];
#pragma unroll
        for (int t = 0; t < kSimtTok; ++t) ag[t] = au[t] = 0.0f;
        for (int b = lane; b < H / 32; b += 32) {
          float fg[32], fu[32];
          decode_fp4x32(*reinterpret_cast<const uint4*>(w13 + gr * (H / 2) + b * 16),
                        w13s[gr * (H / 32) + b], fg);
          decode_fp4x32(*reinterpret_cast<const uint4*>(w13 + ur * (H / 2) + b * 16),
                        w13s[ur * (H / 32) + b], fu);
#pragma unroll
          for (int t = 0; t < kSimtTok; ++t) {
            if (g0 + t < n) {
              ag[t] += act_dot32<ACT>(fg, xq, xs, s0 + g0 + t, H, b);
              au[t] += act_dot32<ACT>(fu, xq, xs, s0 + g0 + t, H, b);
            }
          }
        }
#pragma unroll
        for (int t = 0; t < kSimtTok; ++t) {
          const float g = warp_sum(ag[t]), u = warp_sum(au[t]);
          if (lane == 0 && g0 + t < n) hbuf[r][g0 + t] = g / (1.0f + expf(-g)) * u;
        }
      }
    }
    __syncthreads();
    for (int t = warp; t < n; t += 4) {
      const float v = hbuf[lane][t];
      const int64_t slot = s0 + t;
      if (ACT == MOE_ACT_MXFP8) {
        const int code = block_scale_code(warp_max(fabsf(v)), 8);
        hq[slot * I + ib * kSimtRows + lane] = e4m3_encode_satfinite(v * exp2_exact(127 - code));
        if (lane == 0) hs[slot * (I / 32) + ib] = (uint8_t)code;
      } else {
        reinterpret_cast<uint16_t*>(hq)[slot * I + ib * kSimtRows + lane] = float_to_bf16_bits(v);
      }
    }
    __syncthreads();
  }
}

template <int ACT>
__global__ void __launch_bounds__(128) gemm2_simt_kernel(
    const uint8_t* __restrict__ w2, const uint8_t* __restrict__ w2s,
    const uint8_t* __restrict__ hq, const uint8_t* __restrict__ hs, const int4* __restrict__ chunks,
    const int32_t* __restrict__ meta, int H, int I, float* __restrict__ yp) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int oblocks = H / kSimtRows;
  const int64_t items = (int64_t)meta[0] * oblocks;
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int4 ch = chunks[it / oblocks];
    const int ob = (int)(it % oblocks);
    const int e = ch.x, s0 = ch.y, n = ch.z;
    for (int r = warp * 8; r < warp * 8 + 8; ++r) {
      const int64_t orow = (int64_t)e * H + ob * kSimtRows + r;
      for (int g0 = 0; g0 < n; g0 += kSimtTok) {
        float acc[kSimtTok];
#pragma unroll
        for (int t = 0; t < kSimtTok; ++t) acc[t] = 0.0f;
        for (int b = lane; b < I / 32; b += 32) {
          float f[32];
          decode_fp4x32(*reinterpret_cast<const uint4*>(w2 + orow * (I / 2) + b * 16),
                        w2s[orow * (I / 32) + b], f);
#pragma unroll
          for (int t = 0; t < kSimtTok; ++t)
            if (g0 + t < n) acc[t] += act_dot32<ACT>(f, hq, hs, s0 + g0 + t, I, b);
        }
#pragma unroll
        for (int t = 0; t < kSimtTok; ++t) {
          const float v = warp_sum(acc[t]);
          if (lane == 0 && g0 + t < n)
            yp[(int64_t)(s0 + g0 + t) * H + ob * kSimtRows + r] = v;
        }
      }
    }
  }
}

}  // namespace moe
