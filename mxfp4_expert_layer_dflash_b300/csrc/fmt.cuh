// Device-side number formats of the layer: E2M1 (FP4 weight elements), E8M0
// (block scales), E4M3 (MXFP8 activations) and bf16.
//
// MXFP4 = E2M1 elements in blocks of 32 sharing one E8M0 scale (block size 32:
// ai.appwright.xyz, "投機的デコード", section "第1層：FP4量子化").  Grid
// {0, .5, 1, 1.5, 2, 3, 4, 6} with a sign bit; scale 2^(c - 127).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

// exact floor(log2(a)) of a positive finite fp32, from its bits
__device__ __forceinline__ int floor_log2_bits(float a) {
  uint32_t u = __float_as_uint(a);
  int ex = (int)((u >> 23) & 0xFFu);
  if (ex > 0) return ex - 127;
  uint32_t m = u & 0x7FFFFFu;  // subnormal: m * 2^-149
  return (31 - __clz((int)m)) - 149;
}

// 2^n as an exact fp32, n in [-127, 127]
__device__ __forceinline__ float exp2_exact(int n) {
  return n >= -126 ? __uint_as_float((uint32_t)(n + 127) << 23)
                   : __uint_as_float(0x00400000u);  // 2^-127, subnormal
}

// scale code of a block: clamp(floor(log2(amax)) - emax + 127, 0, 254); 0 if amax == 0
__device__ __forceinline__ int block_scale_code(float amax, int emax) {
  if (!(amax > 0.0f)) return 0;
  int c = floor_log2_bits(amax) - emax + 127;
  return c < 0 ? 0 : (c > 254 ? 254 : c);
}

// E2M1 code of a scaled value: nearest grid point, ties to the even code,
// saturating at 6; the sign comes from the sign bit (so -0 gives code 8).
__device__ __forceinline__ uint32_t e2m1_encode(float q) {
  float a = fabsf(q);
  uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
               (a >= 3.5f) + (a > 5.0f);
  return ((__float_as_uint(q) >> 28) & 8u) | m;
}

// E2M1 magnitude of code bits 2..0: exponent field 0 is subnormal (0, 0.5)
__device__ __forceinline__ float e2m1_decode(uint32_t code) {
  uint32_t ex = (code >> 1) & 3u, m = code & 1u;
  float mag = ex == 0 ? 0.5f * (float)m : (1.0f + 0.5f * (float)m) * (float)(1u << (ex - 1));
  return (code & 8u) ? -mag : mag;
}

__device__ __forceinline__ float e8m0_decode(uint32_t c) { return exp2_exact((int)c - 127); }

__device__ __forceinline__ uint8_t e4m3_encode_satfinite(float q) {
  return (uint8_t)__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_decode(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float((uint32_t)b << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// MXFP8-E4M3 quantization of one block of 32 values (emax of E4M3 is 8)
__device__ __forceinline__ int mxfp8_block(const float* v, uint8_t* out) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int code = block_scale_code(amax, 8);
  float inv = exp2_exact(127 - code);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {  // two values per conversion instruction
    const __nv_fp8x2_storage_t pr =
        __nv_cvt_float2_to_fp8x2(make_float2(v[i] * inv, v[i + 1] * inv), __NV_SATFINITE, __NV_E4M3);
    out[i] = (uint8_t)(pr & 0xFFu);
    out[i + 1] = (uint8_t)(pr >> 8);
  }
  return code;
}

}  // namespace moe
