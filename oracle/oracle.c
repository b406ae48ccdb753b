/*
 * CPU oracle for the MXFP4 Mixture-of-Experts expert layer (fp64, plain C).
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the CUDA library, with which it
 * shares no code.
 *
 * Sources of the definitions:
 *  - Only the MoE expert weights are FP4, in the MXFP4 format with a block
 *    size of 32 and a shared scale: ai.appwright.xyz, tag page "投機的デコード",
 *    section "第1層：FP4量子化"; techllm.github.io, "Xiaomi MiMo and TileRT ...
 *    1000 tokens per second", section "세 층의 속도 최적화 / 1. MXFP4".
 *  - The layer runs on T = sequences x 8 tokens because DFlash verifies a
 *    masked block of up to 8 positions in one forward: techllm.github.io,
 *    section "2. DFlash"; dothoosh.com, section "جزئیات پیاده‌سازی DFlash".
 *  - The parts the pages leave open are fixed by the layer specification this
 *    repository implements: E2M1 grid {0,.5,1,1.5,2,3,4,6} with sign, E8M0
 *    scale 2^(c-127) chosen as 2^(floor(log2(amax)) - 2), round to nearest
 *    even with saturation at +-6; top-k with the lower expert index winning
 *    ties; softmax renormalised over the k selected logits; SwiGLU
 *    silu(gate) * up; bf16 output; MXFP8-E4M3 activations.
 */
#include "oracle.h"

#include <math.h>
#include <omp.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ formats */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * exponent 0 is subnormal: m * 0.5; otherwise (1 + m/2) * 2^(exp-1). */
double oracle_e2m1_value(int code) {
  int s = (code >> 3) & 1, ex = (code >> 1) & 3, m = code & 1;
  double mag = (ex == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, ex - 1);
  return s ? -mag : mag;
}

/* E8M0: unsigned exponent, value 2^(code-127); 0xFF is NaN */
double oracle_e8m0_value(int code) {
  if (code == 255) return NAN;
  return ldexp(1.0, code - 127);
}

/* E4M3 (finite-only variant): bit 7 sign, bits 6..3 exponent (bias 7),
 * bits 2..0 mantissa; exponent 0 subnormal m/8 * 2^-6; S.1111.111 is NaN. */
double oracle_e4m3_value(int code) {
  int s = (code >> 7) & 1, ex = (code >> 3) & 15, m = code & 7;
  if (ex == 15 && m == 7) return NAN;
  double mag = (ex == 0) ? (m / 8.0) * ldexp(1.0, -6) : (1.0 + m / 8.0) * ldexp(1.0, ex - 7);
  return s ? -mag : mag;
}

/* bf16: the upper 16 bits of an IEEE binary32 */
double oracle_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

int oracle_floor_log2_f32(float a) {
  uint32_t u;
  memcpy(&u, &a, 4);
  int ex = (int)((u >> 23) & 0xFF);
  if (ex > 0) return ex - 127;
  uint32_t m = u & 0x7FFFFF; /* subnormal: m * 2^-149 */
  int p = 0;
  while ((m >> (p + 1)) != 0) ++p;
  return p - 149;
}

/* nearest of the non-negative codes [0, n) whose decoded magnitudes are mag[];
 * ties to the even code */
static int nearest_code(double a, int n, const double* mag) {
  int best = 0;
  double bd = fabs(a - mag[0]);
  for (int c = 1; c < n; ++c) {
    double d = fabs(a - mag[c]);
    if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      bd = d;
    }
  }
  return best;
}

/* decoded non-negative magnitudes, memoized once (same values as the decoders) */
static double g_e2m1_mag[8], g_e4m3_mag[0x7F];
static void init_mags(void) {
  static int ready = 0;
  if (ready) return;
#pragma omp critical(oracle_init_mags)
  if (!ready) {
    for (int c = 0; c < 8; ++c) g_e2m1_mag[c] = oracle_e2m1_value(c);
    for (int c = 0; c < 0x7F; ++c) g_e4m3_mag[c] = oracle_e4m3_value(c);
#pragma omp flush
    ready = 1;
  }
}

/* sign copied from the input's sign bit, so -0 and small negatives give code 8 */
int oracle_e2m1_encode(double q) {
  init_mags();
  int neg = signbit(q) ? 1 : 0;
  double a = fabs(q);
  if (a >= 6.0) return (neg << 3) | 7; /* saturate */
  return (neg << 3) | nearest_code(a, 8, g_e2m1_mag);
}

int oracle_e4m3_encode(double q) {
  init_mags();
  int neg = signbit(q) ? 1 : 0;
  double a = fabs(q);
  if (a >= 448.0) return (neg << 7) | 0x7E; /* satfinite */
  return (neg << 7) | nearest_code(a, 0x7F, g_e4m3_mag);
}

uint16_t oracle_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int ex2;
  frexp(a, &ex2);
  int e = ex2 - 1; /* floor(log2(a)) */
  if (e < -126) e = -126;
  double ulp = ldexp(1.0, e - 7); /* 8 significant bits */
  double n = a / ulp;             /* exact */
  double r = floor(n);
  double fr = n - r;
  if (fr > 0.5 || (fr == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  double rv = r * ulp;
  if (rv >= 0x1p128) return sign | 0x7F80;
  float f = (float)rv; /* exact: rv has <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return sign | (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------ quantization */

static int clamp_scale_code(int e) {
  int c = e + 127;
  return c < 0 ? 0 : (c > 254 ? 254 : c);
}

/* MXFP4: per block of 32 along K, scale code = clamp(floor(log2(amax)) - 2 + 127),
 * elements q = w / 2^(code-127) rounded to the E2M1 grid.  amax == 0 gives
 * scale code 0.  Element 2i sits in the low nibble of byte i. */
void oracle_mxfp4_quantize(const float* w, int64_t R, int64_t K, uint8_t* out_fp4,
                           uint8_t* out_e8m0) {
  const int64_t nb = K / 32;
  init_mags();
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = w + r * K + b * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) {
        float a = fabsf(blk[i]);
        if (a > amax) amax = a;
      }
      int code = (amax == 0.0f) ? 0 : clamp_scale_code(oracle_floor_log2_f32(amax) - 2);
      out_e8m0[r * nb + b] = (uint8_t)code;
      double X = oracle_e8m0_value(code);
      for (int i = 0; i < 32; i += 2) {
        int lo = oracle_e2m1_encode((double)blk[i] / X);
        int hi = oracle_e2m1_encode((double)blk[i + 1] / X);
        out_fp4[(r * K + b * 32 + i) / 2] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
}

/* MXFP8-E4M3: per block of 32, scale code = clamp(floor(log2(amax)) - 8 + 127)
 * (8 = exponent of the largest power of two in E4M3), elements rounded to
 * nearest even E4M3 with saturation at +-448.  amax == 0 gives scale code 0. */
void oracle_mxfp8_quantize_row(const double* v, int64_t K, uint8_t* codes, uint8_t* scales) {
  for (int64_t b = 0; b < K / 32; ++b) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
      double a = fabs(v[b * 32 + i]);
      if (a > amax) amax = a;
    }
    int code = 0;
    if (amax > 0.0) {
      int ex2;
      frexp(amax, &ex2);
      code = clamp_scale_code((ex2 - 1) - 8);
    }
    scales[b] = (uint8_t)code;
    double X = oracle_e8m0_value(code);
    for (int i = 0; i < 32; ++i) codes[b * 32 + i] = (uint8_t)oracle_e4m3_encode(v[b * 32 + i] / X);
  }
}

/* act step of the given mode applied in place to a row of K doubles */
static void apply_act(double* v, int64_t K, int act_mode, uint8_t* tmp_codes, uint8_t* tmp_sc) {
  if (act_mode == ORACLE_ACT_MXFP8) {
    oracle_mxfp8_quantize_row(v, K, tmp_codes, tmp_sc);
    for (int64_t i = 0; i < K; ++i)
      v[i] = oracle_e4m3_value(tmp_codes[i]) * oracle_e8m0_value(tmp_sc[i / 32]);
  } else if (act_mode == ORACLE_ACT_BF16) {
    for (int64_t i = 0; i < K; ++i) v[i] = oracle_bf16_value(oracle_bf16_from_double(v[i]));
  }
}

/* ------------------------------------------------------------------ routing */

void oracle_route(const float* logits, int64_t T, int64_t E, int k, int32_t* idx,
                  double* gate) {
  char* taken = (char*)malloc((size_t)E);
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict: lower index keeps ties */
      }
      taken[best] = 1;
      idx[t * k + j] = (int32_t)best;
    }
    double m = (double)l[idx[t * k]];
    double s = 0.0;
    for (int j = 0; j < k; ++j) s += exp((double)l[idx[t * k + j]] - m);
    for (int j = 0; j < k; ++j) gate[t * k + j] = exp((double)l[idx[t * k + j]] - m) / s;
  }
  free(taken);
}

void oracle_route_arrays(const int32_t* idx, int64_t T, int k, int64_t E, int32_t* cnt,
                         int32_t* off, int32_t* perm, int32_t* pos) {
  for (int64_t e = 0; e < E; ++e) cnt[e] = 0;
  for (int64_t f = 0; f < T * k; ++f) cnt[idx[f]]++;
  off[0] = 0;
  for (int64_t e = 0; e < E; ++e) off[e + 1] = off[e] + cnt[e];
  int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
  for (int64_t f = 0; f < T * k; ++f) { /* ascending flat index t*k + j */
    int32_t e = idx[f];
    int32_t p = off[e] + fill[e]++;
    perm[p] = (int32_t)(f / k);
    pos[f] = p;
  }
  free(fill);
}

/* ------------------------------------------------------------------ forward */

static double g_e2m1[16];
static double g_e8m0[256];
static int g_tables_ready = 0;

static void init_tables(void) {
  if (g_tables_ready) return;
  for (int c = 0; c < 16; ++c) g_e2m1[c] = oracle_e2m1_value(c);
  for (int c = 0; c < 256; ++c) g_e8m0[c] = oracle_e8m0_value(c);
  g_tables_ready = 1;
}

/* decoded weight element (row r, column c) of a packed matrix with K columns */
static inline double wval(const uint8_t* fp4, const uint8_t* e8m0, int64_t K, int64_t r,
                          int64_t c) {
  uint8_t byte = fp4[(r * K + c) >> 1];
  int nib = (c & 1) ? (byte >> 4) : (byte & 0xF);
  return g_e2m1[nib] * g_e8m0[e8m0[r * (K / 32) + c / 32]];
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

int oracle_moe_forward(const uint16_t* x_bf16, const float* router_logits,
                       const uint8_t* w13_fp4, const uint8_t* w13_e8m0,
                       const uint8_t* w2_fp4, const uint8_t* w2_e8m0, int64_t T, int64_t H,
                       int64_t I, int64_t E, int k, int act_mode, const int64_t* tokens,
                       int64_t n_tokens, double* y_f64, uint16_t* y_bf16, double* h_out,
                       int n_threads) {
  if (T < 0 || H <= 0 || I <= 0 || E <= 0 || k < 1 || k > E || H % 32 || I % 32) return -1;
  if (act_mode < 0 || act_mode > 2) return -1;
  if (!tokens) n_tokens = T;
  init_tables();
  init_mags();
  const int nt = n_threads > 0 ? n_threads : omp_get_max_threads();

  /* per token: act1(x) and the routing decision */
  double* a = (double*)malloc(sizeof(double) * (size_t)(n_tokens * H));
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_tokens * k));
  double* g = (double*)malloc(sizeof(double) * (size_t)(n_tokens * k));
  /* per (token, slot): the expert's output W2 act2(h) */
  double* d = (double*)malloc(sizeof(double) * (size_t)(n_tokens * k * H));

#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
  for (int64_t n = 0; n < n_tokens; ++n) {
    int64_t t = tokens ? tokens[n] : n;
    uint8_t* tc = (uint8_t*)malloc((size_t)H);
    uint8_t* ts = (uint8_t*)malloc((size_t)H / 32);
    double* an = a + n * H;
    for (int64_t h = 0; h < H; ++h) an[h] = oracle_bf16_value(x_bf16[t * H + h]);
    apply_act(an, H, act_mode == ORACLE_ACT_MXFP8 ? ORACLE_ACT_MXFP8 : ORACLE_ACT_EXACT, tc, ts);
    oracle_route(router_logits + t * E, 1, E, k, idx + n * k, g + n * k);
    free(tc);
    free(ts);
  }

#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
  for (int64_t task = 0; task < n_tokens * k; ++task) {
    const int64_t n = task / k;
    const int j = (int)(task % k);
    const int64_t e = idx[n * k + j];
    const double* an = a + n * H;
    double* hv = (double*)malloc(sizeof(double) * (size_t)I);
    uint8_t* tc = (uint8_t*)malloc((size_t)I);
    uint8_t* ts = (uint8_t*)malloc((size_t)I / 32);
    const int64_t r0 = e * 2 * I; /* first w13 row of expert e */
    for (int64_t i = 0; i < I; ++i) {
      double gate = 0.0, up = 0.0;
      for (int64_t h = 0; h < H; ++h) {
        gate += wval(w13_fp4, w13_e8m0, H, r0 + i, h) * an[h];
        up += wval(w13_fp4, w13_e8m0, H, r0 + I + i, h) * an[h];
      }
      hv[i] = silu(gate) * up;
    }
    apply_act(hv, I, act_mode, tc, ts);
    if (h_out)
      for (int64_t i = 0; i < I; ++i) h_out[(n * k + j) * I + i] = hv[i];
    double* dn = d + task * H;
    for (int64_t o = 0; o < H; ++o) {
      double acc = 0.0;
      for (int64_t i = 0; i < I; ++i) acc += wval(w2_fp4, w2_e8m0, I, e * H + o, i) * hv[i];
      dn[o] = acc;
    }
    free(hv);
    free(tc);
    free(ts);
  }

  /* gate-weighted sum in slot order j = 0..k-1, then bf16 rounding */
  for (int64_t n = 0; n < n_tokens; ++n) {
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += g[n * k + j] * d[(n * k + j) * H + h];
      if (y_f64) y_f64[n * H + h] = acc;
      if (y_bf16) y_bf16[n * H + h] = oracle_bf16_from_double(acc);
    }
  }
  free(a);
  free(idx);
  free(g);
  free(d);
  return 0;
}

/* --------------------------------------------------- a chain of layers
 *
 * Several expert layers run back to back over the same block of tokens: the
 * whole pipeline kept resident on the GPU rather than one operator at a time
 * (dothoosh.com, section "TileRT"; techllm.github.io, "Xiaomi MiMo and TileRT
 * ...", section "3. TileRT").  The pages give no formula for what flows
 * between the layers; read plainly, layer l's output is layer l+1's input,
 * optionally added to a residual stream before the one bf16 rounding:
 *   x_0 = x,  x_{l+1} = bf16_RNE( y_l + r * x_l ),  output x_L,
 * where y_l is layer l's fp64 output before its final rounding (each layer as
 * oracle_moe_forward, with its own router logits and weights) and r is 0 or 1.
 * With r = 0 each step is exactly oracle_moe_forward's bf16 output. */
int oracle_moe_chain(int n_layers, const uint16_t* x_bf16, const float* const* router_logits,
                     const uint8_t* const* w13_fp4, const uint8_t* const* w13_e8m0,
                     const uint8_t* const* w2_fp4, const uint8_t* const* w2_e8m0, int64_t T,
                     int64_t H, int64_t I, int64_t E, int k, int act_mode, int residual,
                     uint16_t* y_bf16, int n_threads) {
  if (n_layers < 1 || T < 0 || H <= 0 || (residual != 0 && residual != 1)) return -1;
  uint16_t* cur = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(T * H + 1));
  double* y = (double*)malloc(sizeof(double) * (size_t)(T * H + 1));
  for (int64_t i = 0; i < T * H; ++i) cur[i] = x_bf16[i];
  int rc = 0;
  for (int l = 0; l < n_layers && rc == 0; ++l) {
    rc = oracle_moe_forward(cur, router_logits[l], w13_fp4[l], w13_e8m0[l], w2_fp4[l],
                            w2_e8m0[l], T, H, I, E, k, act_mode, NULL, T, y, NULL, NULL,
                            n_threads);
    for (int64_t i = 0; rc == 0 && i < T * H; ++i)
      cur[i] = oracle_bf16_from_double(y[i] + (residual ? oracle_bf16_value(cur[i]) : 0.0));
  }
  if (rc == 0)
    for (int64_t i = 0; i < T * H; ++i) y_bf16[i] = cur[i];
  free(cur);
  free(y);
  return rc;
}

/* --------------------------------------------------- the router and a dense
 * FP8 projection (the steps beside the expert layer) */

/* Router: one logit per expert from the token's hidden state.  The pages name
 * expert routing as part of the pipeline the runtime is built around
 * (techllm.github.io, "Xiaomi MiMo and TileRT ...", section "3. TileRT") but
 * give no formula; read as the usual linear layer, logits = x W_r^T, with bf16
 * weights W_r [E, H].  Exact fp64 dot products of the decoded bf16 values. */
void oracle_router_logits(const uint16_t* x_bf16, const uint16_t* w_bf16, int64_t T,
                          int64_t H, int64_t E, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t e = 0; e < E; ++e) {
      double s = 0.0;
      for (int64_t h = 0; h < H; ++h)
        s += oracle_bf16_value(x_bf16[t * H + h]) * oracle_bf16_value(w_bf16[e * H + h]);
      out[t * E + e] = s;
    }
  }
}

/* MXFP8 packing of fp32 rows [R, K] (K % 32 == 0), the rule of
 * oracle_mxfp8_quantize_row applied to each row */
void oracle_mxfp8_quantize(const float* w, int64_t R, int64_t K, uint8_t* codes,
                           uint8_t* scales) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    double* v = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t i = 0; i < K; ++i) v[i] = (double)w[r * K + i];
    oracle_mxfp8_quantize_row(v, K, codes + r * K, scales + r * (K / 32));
    free(v);
  }
}

/* Dense FP8 projection, a layer outside the experts: the pages keep every
 * module but the MoE experts at FP8 (techllm.github.io, "Xiaomi MiMo and
 * TileRT ...", section "1. MXFP4 — MoE에만 걸린 양자화"; ai.appwright.xyz, tag
 * page "投機的デコード", section "第1層：FP4量子化": o_proj stays out of FP4).
 * Read as MXFP8 weights (E4M3 codes [N, K], E8M0 scales [N, K/32], decoded
 * exactly as e4m3(code) * 2^(scale - 127)) and
 *   y[t, n] = bf16_RNE( sum_k act(x[t, k]) * w[n, k] ),
 * act = MXFP8 of x along K (the same rule as the experts' inputs) or the
 * identity (exact mode).  y_f64 / y_bf16 [T, N] may each be NULL. */
int oracle_dense_forward(const uint16_t* x_bf16, const uint8_t* w_e4m3, const uint8_t* w_e8m0,
                         int64_t T, int64_t K, int64_t N, int act_mode, double* y_f64,
                         uint16_t* y_bf16) {
  if (T < 0 || K <= 0 || N <= 0 || K % 32) return -1;
  if (act_mode != ORACLE_ACT_EXACT && act_mode != ORACLE_ACT_MXFP8) return -1;
  init_mags();
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    double* a = (double*)malloc(sizeof(double) * (size_t)K);
    uint8_t* tc = (uint8_t*)malloc((size_t)K);
    uint8_t* ts = (uint8_t*)malloc((size_t)K / 32);
    for (int64_t i = 0; i < K; ++i) a[i] = oracle_bf16_value(x_bf16[t * K + i]);
    apply_act(a, K, act_mode, tc, ts);
    for (int64_t n = 0; n < N; ++n) {
      double s = 0.0;
      for (int64_t i = 0; i < K; ++i)
        s += a[i] * oracle_e4m3_value(w_e4m3[n * K + i]) *
             oracle_e8m0_value(w_e8m0[n * (K / 32) + i / 32]);
      if (y_f64) y_f64[t * N + n] = s;
      if (y_bf16) y_bf16[t * N + n] = oracle_bf16_from_double(s);
    }
    free(a);
    free(tc);
    free(ts);
  }
  return 0;
}

/* ------------------------------------------------ speculative verification */

/* Inverse-CDF draw over masses m[x] = floor(w[x] * 2^62) (w = fp32 weights in
 * [0, 1], the scaling exact): with M = sum m, the drawn index is the first x
 * whose running sum exceeds floor(U * M / 2^64).  Returns -1 when M == 0. */
static int64_t draw_fixed_point(const float* w, int64_t V, uint64_t U) {
  uint64_t M = 0;
  for (int64_t x = 0; x < V; ++x) M += (uint64_t)floor((double)w[x] * 0x1p62);
  if (M == 0) return -1;
  const unsigned __int128 prod = (unsigned __int128)U * (unsigned __int128)M;
  const uint64_t t = (uint64_t)(prod >> 64);
  uint64_t run = 0;
  for (int64_t x = 0; x < V; ++x) {
    run += (uint64_t)floor((double)w[x] * 0x1p62);
    if (run > t) return x;
  }
  return V - 1; /* not reached: t < M */
}

/* Rejection-sampling verification of one block of drafted tokens per
 * sequence (lossless speculative decoding: techllm.github.io, "Xiaomi MiMo and
 * TileRT ...", section "2. DFlash"; the block is at most 8 positions:
 * dothoosh.com, section "جزئیات پیاده‌سازی DFlash").  For sequence s, drafted
 * tokens d_0..d_{g-1} with draft distributions q_i and target distributions
 * p_0..p_g (p_g for the position after the block):
 *   accept d_i while u_i * q_i(d_i) < p_i(d_i) (exact: fp32 values compared
 *   in fp64; for u uniform on [0, 1) this happens with probability
 *   min(1, p_i(d_i) / q_i(d_i)), and a token with p_i(d_i) = 0 is never
 *   accepted);
 *   at the first rejection i, emit a token drawn from max(0, p_i - q_i) (the
 *   fp32 difference), else after g acceptances emit one drawn from p_g; draws
 *   use draw_fixed_point with the sequence's 64-bit uniform U[s] (from p_i
 *   itself if the residual mass is 0).
 * Outputs: n_acc[s] in [0, g]; tokens[s, 0..n_acc] = accepted drafts then the
 * emitted token (tokens [S, g+1]; entries past n_acc are -1).
 * p [S, g+1, V], q [S, g, V] fp32; draft [S, g] int32; u [S, g] fp32 in [0, 1). */
int oracle_verify(const float* p, const float* q, const int32_t* draft, const float* u,
                  const uint64_t* U, int64_t S, int g, int64_t V, int32_t* n_acc,
                  int32_t* tokens) {
  if (S < 0 || g < 1 || V < 1) return -1;
  float* r = (float*)malloc(sizeof(float) * (size_t)V);
  for (int64_t s = 0; s < S; ++s) {
    const float* ps = p + s * (int64_t)(g + 1) * V;
    const float* qs = q + s * (int64_t)g * V;
    int32_t* out = tokens + s * (int64_t)(g + 1);
    for (int i = 0; i <= g; ++i) out[i] = -1;
    int i = 0;
    for (; i < g; ++i) {
      const int32_t d = draft[s * g + i];
      if (d < 0 || d >= V) { free(r); return -1; }
      const double lhs = (double)u[s * g + i] * (double)qs[i * V + d];
      if (lhs < (double)ps[i * V + d]) {
        out[i] = d;
      } else {
        break;
      }
    }
    n_acc[s] = i;
    int64_t x;
    if (i < g) {
      for (int64_t v = 0; v < V; ++v) {
        const float diff = ps[i * V + v] - qs[i * V + v];
        r[v] = diff > 0.0f ? diff : 0.0f;
      }
      x = draw_fixed_point(r, V, U[s]);
      if (x < 0) x = draw_fixed_point(ps + i * V, V, U[s]);
    } else {
      x = draw_fixed_point(ps + (int64_t)g * V, V, U[s]);
    }
    out[i] = (int32_t)(x < 0 ? 0 : x);
  }
  free(r);
  return 0;
}
