/*
 * Counter-based synthetic input generator: the element arithmetic shared by
 * the host build (synth.c) and the device build (synth_dev.cu) of this module.
 *
 * Test and benchmark infrastructure only.  It holds none of the MoE layer's
 * arithmetic (no quantization, routing or GEMM): it only turns (seed, tensor
 * id, flat element index) into a number.  Integer hashing, exact conversions
 * and a fixed sequence of correctly rounded fp32 operations, so the host and
 * the device produce the same bits for every element.
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
 *   normal(key, i)  standard normal draw i of the stream, by Marsaglia's
 *                   polar method (G. Marsaglia & T. A. Bray, "A convenient
 *                   method for generating normal variables", SIAM Review
 *                   6(3), 1964): attempt a = 0, 1, ... takes
 *                   r = splitmix(key, 64i + a + 1); its bit fields 41..63
 *                   and 18..40 are 23-bit integers u1, u2, and
 *                   v = (2u + 1 - 2^23) 2^-23 lies in (-1, 1), never 0, exact;
 *                   the first attempt with s = v1^2 + v2^2 < 1 returns
 *                   v1 sqrt(-2 ln(s) / s) (after 40 rejections, a chance
 *                   below 1e-26, it returns 0).
 *   ln(s)           s = m 2^e with m in [sqrt(1/2), sqrt(2)] (bit fields,
 *                   exact), ln s = e ln 2 + 2 (y + y^3/3 + ... + y^11/11),
 *                   y = (m - 1)/(m + 1), |y| < 0.172 (the series of atanh:
 *                   truncation below 1e-10 relative).
 *   fill(key,i,s)   fp32 product s * normal(key, i), rounded once (RN).
 *   Every floating-point step above is one IEEE operation (+, -, *, /,
 *   sqrt) in fp32, rounded to nearest even, in the order written: CUDA's
 *   _rn intrinsics on the device, plain C operators on the host (compiled
 *   without contraction), so both produce the same bits.
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>
#if !defined(__CUDACC__)
#include <math.h>
#endif

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

/* fp32 operations with one round-to-nearest-even each and no contraction */
#if defined(__CUDA_ARCH__)
#define SYNTH_ADD(a, b) __fadd_rn((a), (b))
#define SYNTH_SUB(a, b) __fsub_rn((a), (b))
#define SYNTH_MUL(a, b) __fmul_rn((a), (b))
#define SYNTH_DIV(a, b) __fdiv_rn((a), (b))
#define SYNTH_SQRT(a) __fsqrt_rn((a))
#else
#define SYNTH_ADD(a, b) ((a) + (b))
#define SYNTH_SUB(a, b) ((a) - (b))
#define SYNTH_MUL(a, b) ((a) * (b))
#define SYNTH_DIV(a, b) ((a) / (b))
#define SYNTH_SQRT(a) sqrtf((a))
#endif

#define SYNTH_POLAR_TRIES 40u

/* ln(s) of a positive normal fp32 s (see the definitions above) */
SYNTH_FN float synth_ln(float s) {
  union {
    float f;
    uint32_t u;
  } v;
  v.f = s;
  int32_t e = (int32_t)(v.u >> 23) - 127;
  v.u = (v.u & 0x007FFFFFu) | 0x3F800000u; /* m in [1, 2) */
  if (v.u > 0x3FB504F3u) {                  /* m > sqrt(2): halve it */
    v.u -= 0x00800000u;
    e += 1;
  }
  const float m = v.f;
  const float y = SYNTH_DIV(SYNTH_SUB(m, 1.0f), SYNTH_ADD(m, 1.0f));
  const float y2 = SYNTH_MUL(y, y);
  float p = 0x1.745d18p-4f;                     /* 1/11 */
  p = SYNTH_ADD(SYNTH_MUL(p, y2), 0x1.c71c72p-4f); /* 1/9 */
  p = SYNTH_ADD(SYNTH_MUL(p, y2), 0x1.24924ap-3f); /* 1/7 */
  p = SYNTH_ADD(SYNTH_MUL(p, y2), 0x1.99999ap-3f); /* 1/5 */
  p = SYNTH_ADD(SYNTH_MUL(p, y2), 0x1.555556p-2f); /* 1/3 */
  const float lm = SYNTH_MUL(2.0f, SYNTH_ADD(y, SYNTH_MUL(SYNTH_MUL(y, y2), p)));
  return SYNTH_ADD(SYNTH_MUL((float)e, 0x1.62e430p-1f), lm); /* e ln 2 + ln m */
}

/* normal(key, i) (see the definitions above) */
SYNTH_FN float synth_normal(uint64_t key, uint64_t i) {
  for (uint32_t a = 0; a < SYNTH_POLAR_TRIES; ++a) {
    const uint64_t r = synth_splitmix(key, 64u * i + a + 1u);
    const int32_t n1 = (int32_t)((uint32_t)(r >> 41) << 1) + 1 - (1 << 23);
    const int32_t n2 = (int32_t)((uint32_t)((r >> 18) & 0x7FFFFFu) << 1) + 1 - (1 << 23);
    const float v1 = SYNTH_MUL((float)n1, 0x1p-23f), v2 = SYNTH_MUL((float)n2, 0x1p-23f);
    const float s = SYNTH_ADD(SYNTH_MUL(v1, v1), SYNTH_MUL(v2, v2));
    if (s < 1.0f) {
      const float q = SYNTH_DIV(SYNTH_MUL(-2.0f, synth_ln(s)), s);
      return SYNTH_MUL(v1, SYNTH_SQRT(q));
    }
  }
  return 0.0f;
}

#endif
