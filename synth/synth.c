/*
 * Host build of the counter-based synthetic input generator (definitions in
 * synth_core.h).  Test and benchmark infrastructure: it fills the inputs of
 * the MoE layer (x, router logits, fp32 expert weights before packing, bf16
 * router weights, fp32 dense-projection weights) and holds none of the
 * layer's arithmetic.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (see synth.py).
 * -ffp-contract=off keeps the single fp32 multiply a separate rounding, the
 * same one the device build performs with __fmul_rn.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "synth_core.h"

static float z_as_float(int32_t num) {
  /* num is an integer of magnitude <= 393210 < 2^24: exact in fp32, and the
   * power-of-two scaling keeps it exact */
  return (float)num * 0x1p-16f;
}

uint64_t synth_splitmix_out(uint64_t s, uint64_t n) { return synth_splitmix(s, n); }

int32_t synth_z_numerator(uint64_t seed, uint32_t tensor_id, uint64_t i) {
  return synth_z_num(synth_key(seed, tensor_id), i);
}

/* out[j] = sigma * z(key(seed, id), start + j), fp32, j in [0, n) */
void synth_fill_normal_f32(uint64_t seed, uint32_t tensor_id, uint64_t start,
                           uint64_t n, float sigma, float* out) {
  const uint64_t key = synth_key(seed, tensor_id);
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nn; ++j) {
    float z = z_as_float(synth_z_num(key, start + (uint64_t)j));
    volatile float p = sigma * z; /* one RN multiply, never fused */
    out[j] = p;
  }
}

/* fp32 -> bf16 bits, round to nearest even (finite inputs) */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* out[j] = bf16_RNE(sigma * z(key(seed, id), start + j)), j in [0, n) */
void synth_fill_bf16(uint64_t seed, uint32_t tensor_id, uint64_t start, uint64_t n,
                     float sigma, uint16_t* out) {
  const uint64_t key = synth_key(seed, tensor_id);
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nn; ++j) {
    volatile float p = sigma * z_as_float(synth_z_num(key, start + (uint64_t)j));
    out[j] = f32_to_bf16_rne(p);
  }
}

/* x[t, h] = bf16_RNE(z(key(seed, X), t*H + h)), unit variance */
void synth_fill_x_bf16(uint64_t seed, int64_t T, int64_t H, uint16_t* out) {
  const uint64_t key = synth_key(seed, SYNTH_ID_X);
  int64_t n = T * H;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) {
    out[j] = f32_to_bf16_rne(z_as_float(synth_z_num(key, (uint64_t)j)));
  }
}

/* logits[t, e] = z(key(seed, LOGITS), t*E + e); with zipf_bias != 0 a per-expert
 * bias 3*ln(1/rank), rank = e + 1, is added in double and the sum rounded to
 * fp32 (expert 0 is the most popular). */
void synth_fill_logits(uint64_t seed, int64_t T, int64_t E, int zipf_bias, float* out) {
  const uint64_t key = synth_key(seed, SYNTH_ID_LOGITS);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      float z = z_as_float(synth_z_num(key, (uint64_t)(t * E + e)));
      if (zipf_bias) {
        double b = 3.0 * log(1.0 / (double)(e + 1));
        out[t * E + e] = (float)((double)z + b);
      } else {
        out[t * E + e] = z;
      }
    }
  }
}
