/*
 * Host build of the counter-based synthetic input generator (definitions in
 * synth_core.h).  Test and benchmark infrastructure: it fills the inputs of
 * the MoE layer (x, router logits, fp32 expert weights before packing, bf16
 * router weights, fp32 dense-projection weights, the probabilities and
 * uniforms of a speculative verification) and holds none of the arithmetic
 * of the steps they feed.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (see synth.py).
 * -ffp-contract=off keeps the single fp32 multiply a separate rounding, the
 * same one the device build performs with __fmul_rn.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "synth_core.h"

uint64_t synth_splitmix_out(uint64_t s, uint64_t n) { return synth_splitmix(s, n); }

/* normal(key(seed, id), i): one draw, for tests */
float synth_std_normal(uint64_t seed, uint32_t tensor_id, uint64_t i) {
  return synth_normal(synth_key(seed, tensor_id), i);
}

/* the generator's logarithm, for tests */
float synth_ln_f32(float s) { return synth_ln(s); }

/* out[j] = sigma * normal(key(seed, id), start + j), fp32, j in [0, n) */
void synth_fill_normal_f32(uint64_t seed, uint32_t tensor_id, uint64_t start,
                           uint64_t n, float sigma, float* out) {
  const uint64_t key = synth_key(seed, tensor_id);
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nn; ++j) {
    float z = synth_normal(key, start + (uint64_t)j);
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

/* out[j] = bf16_RNE(sigma * normal(key(seed, id), start + j)), j in [0, n) */
void synth_fill_bf16(uint64_t seed, uint32_t tensor_id, uint64_t start, uint64_t n,
                     float sigma, uint16_t* out) {
  const uint64_t key = synth_key(seed, tensor_id);
  int64_t nn = (int64_t)n;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < nn; ++j) {
    volatile float p = sigma * synth_normal(key, start + (uint64_t)j);
    out[j] = f32_to_bf16_rne(p);
  }
}

/* x[t, h] = bf16_RNE(normal(key(seed, X), t*H + h)) */
void synth_fill_x_bf16(uint64_t seed, int64_t T, int64_t H, uint16_t* out) {
  const uint64_t key = synth_key(seed, SYNTH_ID_X);
  int64_t n = T * H;
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) {
    out[j] = f32_to_bf16_rne(synth_normal(key, (uint64_t)j));
  }
}

/* logits[t, e] = normal(key(seed, LOGITS), t*E + e); with zipf_bias != 0 a per-expert
 * bias 3*ln(1/rank), rank = e + 1, is added in double and the sum rounded to
 * fp32 (expert 0 is the most popular). */
void synth_fill_logits(uint64_t seed, int64_t T, int64_t E, int zipf_bias, float* out) {
  const uint64_t key = synth_key(seed, SYNTH_ID_LOGITS);
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      float z = synth_normal(key, (uint64_t)(t * E + e));
      if (zipf_bias) {
        double b = 3.0 * log(1.0 / (double)(e + 1));
        out[t * E + e] = (float)((double)z + b);
      } else {
        out[t * E + e] = z;
      }
    }
  }
}

/* softmax of row[0..V) in double, written as fp32 probabilities */
static void softmax_row_f32(const double* z, int64_t V, float* out) {
  double m = z[0];
  for (int64_t v = 1; v < V; ++v) m = z[v] > m ? z[v] : m;
  double s = 0.0;
  for (int64_t v = 0; v < V; ++v) s += exp(z[v] - m);
  for (int64_t v = 0; v < V; ++v) out[v] = (float)(exp(z[v] - m) / s);
}

/* Inputs of the speculative verification of a drafted block, for S sequences
 * of g drafted tokens over a vocabulary of V:
 *   p [S, g+1, V]  target probabilities, softmax(sigma_t * z)          (id 6)
 *   q [S, g, V]    draft probabilities, softmax(sigma_t * z + sigma_n * z'),
 *                  z' a second stream (id 7): a correlated, imperfect drafter
 *   d [S, g]       drafted tokens, drawn from q by inverse CDF in double with a
 *                  53-bit uniform from splitmix(key(seed, 8), s*g + i)
 *   u [S, g]       accept uniforms k / 2^24, k the top 24 bits of
 *                  splitmix(key(seed, 9), s*g + i)
 *   U [S]          64-bit resample uniforms splitmix(key(seed, 10), s) */
void synth_fill_verify(uint64_t seed, int64_t S, int g, int64_t V, float sigma_t, float sigma_n,
                       float* p, float* q, int32_t* d, float* u, uint64_t* U) {
  const uint64_t kz = synth_key(seed, SYNTH_ID_VERIFY_Z), kn = synth_key(seed, SYNTH_ID_VERIFY_N);
  const uint64_t kd = synth_key(seed, SYNTH_ID_VERIFY_D), ku = synth_key(seed, SYNTH_ID_VERIFY_U);
  const uint64_t kU = synth_key(seed, SYNTH_ID_VERIFY_R);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t row = 0; row < S * (g + 1); ++row) {
    const int64_t s = row / (g + 1), i = row % (g + 1);
    double* z = (double*)malloc(sizeof(double) * (size_t)V);
    for (int64_t v = 0; v < V; ++v)
      z[v] = (double)sigma_t * (double)synth_normal(kz, (uint64_t)(row * V + v));
    softmax_row_f32(z, V, p + row * V);
    if (i < g) {
      const int64_t qrow = s * g + i;
      for (int64_t v = 0; v < V; ++v)
        z[v] += (double)sigma_n * (double)synth_normal(kn, (uint64_t)(qrow * V + v));
      float* qr = q + qrow * V;
      softmax_row_f32(z, V, qr);
      const double r = (double)(synth_splitmix(kd, (uint64_t)qrow) >> 11) * 0x1p-53;
      double c = 0.0;
      int64_t pick = V - 1;
      for (int64_t v = 0; v < V; ++v) {
        c += (double)qr[v];
        if (c > r) {
          pick = v;
          break;
        }
      }
      d[qrow] = (int32_t)pick;
      u[qrow] = (float)(synth_splitmix(ku, (uint64_t)qrow) >> 40) * 0x1p-24f;
    }
    free(z);
  }
  for (int64_t s = 0; s < S; ++s) U[s] = synth_splitmix(kU, (uint64_t)s);
}
