// Quantization kernels:
//  - MXFP4 packing of fp32 weights (offline): per block of 32, scale code
//    clamp(floor(log2(amax)) - 2 + 127, 0, 254), elements on the E2M1 grid
//    (block size 32: ai.appwright.xyz, "投機的デコード", "第1層：FP4量子化");
//  - the activation step a4: gather x rows into expert-major slot order and
//    quantize them to MXFP8-E4M3 (blocks of 32 along H), or copy them as bf16.
#pragma once

#include "common.cuh"
#include "fmt.cuh"

namespace moe {

// one thread per block of 32 fp32 elements; blocks are contiguous in memory
__global__ void __launch_bounds__(256) mxfp4_quantize_kernel(const float* __restrict__ w,
                                                             int64_t nblocks,
                                                             uint8_t* __restrict__ fp4,
                                                             uint8_t* __restrict__ e8m0) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
    const float4* src = reinterpret_cast<const float4*>(w + b * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 q = __ldcs(src + i);  // streamed once
      v[4 * i] = q.x;
      v[4 * i + 1] = q.y;
      v[4 * i + 2] = q.z;
      v[4 * i + 3] = q.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int code = block_scale_code(amax, 2);
    const float inv = exp2_exact(127 - code);  // exact power of two
    uint32_t words[4];
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
      uint32_t x = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) x |= e2m1_encode(v[wd * 8 + i] * inv) << (4 * i);
      words[wd] = x;
    }
    *reinterpret_cast<uint4*>(fp4 + b * 16) = make_uint4(words[0], words[1], words[2], words[3]);
    e8m0[b] = (uint8_t)code;
  }
}

// load 32 bf16 (64 bytes, 16-byte aligned) as floats
__device__ __forceinline__ void load_bf16x32(const uint16_t* p, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 q = s[i];
    uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

__device__ __forceinline__ void store_u8x32(uint8_t* p, const uint8_t* c) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = (uint32_t)c[4 * i] | ((uint32_t)c[4 * i + 1] << 8) | ((uint32_t)c[4 * i + 2] << 16) |
           ((uint32_t)c[4 * i + 3] << 24);
  reinterpret_cast<uint4*>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
  reinterpret_cast<uint4*>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// MXFP8 rows: one warp per (row, segment of 32 blocks of 32), a block per
// lane.  row_map selects the source row (identity when null, or the
// permutation slot -> token).
__global__ void __launch_bounds__(256) mxfp8_rows_kernel(const uint16_t* __restrict__ x,
                                                         const int32_t* __restrict__ row_map,
                                                         int64_t rows, int64_t K, int64_t src_rows,
                                                         uint8_t* __restrict__ q,
                                                         uint8_t* __restrict__ s, int* status) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t nb = K / 32;
  const int64_t segs = (nb + 31) / 32;
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < rows * segs;
       u += warps) {
    const int64_t r = u / segs;
    const int64_t b = (u - r * segs) * 32 + lane;
    int64_t src = row_map ? row_map[r] : r;
    if (src < 0 || src >= src_rows) {
      if (lane == 0) set_status(status, kStatusFault);
      src = 0;
    }
    if (b < nb) {
      float v[32];
      uint8_t c[32];
      load_bf16x32(x + src * K + b * 32, v);
      const int code = mxfp8_block(v, c);
      store_u8x32(q + r * K + b * 32, c);
      s[r * nb + b] = (uint8_t)code;
    }
  }
}

// MXFP8 packing of fp32 rows [rows, K] (weights of a dense FP8 layer): one
// warp per row, lane-strided blocks of 32, the same rule as the activations
__global__ void __launch_bounds__(256) mxfp8_rows_f32_kernel(const float* __restrict__ w,
                                                             int64_t rows, int64_t K,
                                                             uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ s) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t nb = K / 32;
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    for (int64_t b = lane; b < nb; b += 32) {
      float v[32];
      uint8_t c[32];
      const float4* src = reinterpret_cast<const float4*>(w + r * K + b * 32);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 f = src[i];
        v[4 * i] = f.x;
        v[4 * i + 1] = f.y;
        v[4 * i + 2] = f.z;
        v[4 * i + 3] = f.w;
      }
      const int code = mxfp8_block(v, c);
      store_u8x32(q + r * K + b * 32, c);
      s[r * nb + b] = (uint8_t)code;
    }
  }
}

// Step a4 per token: a warp per (token, run of 32 blocks of 32), a block per
// lane; each token's row is quantised (MXFP8) or read (bf16) once and written
// to its k slot rows pos[t*k + j] — the same bytes as the per-slot kernels
// with k times fewer loads.
template <bool kMxfp8>
__global__ void __launch_bounds__(256) act_tokens_kernel(const uint16_t* __restrict__ x,
                                                         const int32_t* __restrict__ pos, int T,
                                                         int k, int64_t K, uint8_t* __restrict__ q,
                                                         uint8_t* __restrict__ s, int* status) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t nb = K / 32, segs = (nb + 31) / 32, slots = (int64_t)T * k;
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       u < (int64_t)T * segs; u += warps) {
    const int64_t t = u / segs;
    const int64_t b = (u - t * segs) * 32 + lane;
    const bool live = b < nb;  // lanes past the row still take part in the shuffles
    // the token's k slots in one round trip: lane j loads slot j
    const int my_slot = lane < k ? pos[t * k + lane] : 0;
    uint8_t c[32];
    int code = 0;
    uint4 raw[4];
    if (live) {
      if (kMxfp8) {
        float v[32];
        load_bf16x32(x + t * K + b * 32, v);
        code = mxfp8_block(v, c);
      } else {
        const uint4* a = reinterpret_cast<const uint4*>(x + t * K + b * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) raw[i] = a[i];
      }
    }
    for (int j = 0; j < k; ++j) {
      const int64_t slot = __shfl_sync(0xffffffffu, my_slot, j);
      if (!live) continue;
      if (slot < 0 || slot >= slots) {
        set_status(status, kStatusFault);
        continue;
      }
      if (kMxfp8) {
        store_u8x32(q + slot * K + b * 32, c);
        s[slot * nb + b] = (uint8_t)code;
      } else {
        uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(q) + slot * K + b * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = raw[i];
      }
    }
  }
}

}  // namespace moe
