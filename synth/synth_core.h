/*
 * Counter-based synthetic input generator: the element arithmetic shared by
 * the host build (synth.c) and the device build (synth_dev.cu) of this module.
 *
 * Test and benchmark infrastructure only.  It holds none of the MoE layer's
 * arithmetic (no quantization, routing or GEMM): it only turns (seed, tensor
 * id, flat element index) into a number.  Everything is integer arithmetic
 * plus exact conversions and one correctly rounded fp32 multiply, so the host
 * and the device produce the same bits for every element.
 *
 * Definitions
 *   mix64(z)        SplitMix64 output function (Steele, Lea & Flood, "Fast
 *                   splittable pseudorandom number generators", OOPSLA 2014;
 *                   constants as published with the Java SplittableRandom /
 *                   Vigna's splitmix64.c):
 *                     z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *                     z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *                     return z ^ (z >> 31)
 *   splitmix(s, n)  n-th output (n >= 1) of SplitMix64 seeded with s:
 *                     mix64(s + n * 0x9E3779B97F4A7C15)   (mod 2^64)
 *   key(seed, id)   splitmix(seed, id + 1)
 *   z(key, i)       Irwin-Hall sum of twelve 16-bit uniforms, centred and
 *                   scaled to unit variance: the twelve uniforms are the four
 *                   16-bit fields (low field first) of splitmix(key, 3i+1),
 *                   splitmix(key, 3i+2), splitmix(key, 3i+3);
 *                     S = sum of the twelve, z = (S - 393210) * 2^-16.
 *                   S - 393210 lies in [-393210, 393210] and is exact in
 *                   fp32, so z is exact.  Mean 0, variance 1 - 2^-32,
 *                   support [-6, 6]: the stand-in for a N(0,1) draw.
 *   normal(key,i,s) fp32 product s * z(key, i), rounded once (RN).
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_FN static __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

/* tensor ids */
#define SYNTH_ID_X 0u
#define SYNTH_ID_LOGITS 1u
#define SYNTH_ID_W13 2u
#define SYNTH_ID_W2 3u
#define SYNTH_ID_WROUTER 4u
#define SYNTH_ID_WDENSE 5u
#define SYNTH_ID_VERIFY_Z 6u
#define SYNTH_ID_VERIFY_N 7u
#define SYNTH_ID_VERIFY_D 8u
#define SYNTH_ID_VERIFY_U 9u
#define SYNTH_ID_VERIFY_R 10u

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

SYNTH_FN uint64_t synth_splitmix(uint64_t s, uint64_t n) {
  return synth_mix64(s + n * SYNTH_GAMMA);
}

SYNTH_FN uint64_t synth_key(uint64_t seed, uint32_t tensor_id) {
  return synth_splitmix(seed, (uint64_t)tensor_id + 1u);
}

/* integer numerator of z: S - 393210, in [-393210, 393210] */
SYNTH_FN int32_t synth_z_num(uint64_t key, uint64_t i) {
  uint32_t s = 0;
  for (uint64_t r = 1; r <= 3; ++r) {
    uint64_t u = synth_splitmix(key, 3u * i + r);
    s += (uint32_t)(u & 0xFFFFu) + (uint32_t)((u >> 16) & 0xFFFFu) +
         (uint32_t)((u >> 32) & 0xFFFFu) + (uint32_t)(u >> 48);
  }
  return (int32_t)s - 393210;
}

#endif
