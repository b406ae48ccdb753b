/*
 * CPU oracle for the MXFP4 Mixture-of-Experts expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, slow, fp64 C that states the layer's
 * definition directly.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the CUDA library never does, and the two
 * share no code, header, table or helper.
 *
 * What the layer computes (per token t, with W1 = rows [0,I) of w13 and
 * W3 = rows [I,2I) of w13, every weight decoded exactly as
 * e2m1(code) * 2^(scale - 127)):
 *
 *   (e_j, g_j)_{j<k} = top-k of router_logits[t] (ties: lower expert index
 *                      first), g = softmax over the k selected logits
 *   y[t] = bf16_RNE( sum_j g_j * W2_{e_j} act2( silu(W1_{e_j} act1(x_t))
 *                                               * (W3_{e_j} act1(x_t)) ) )
 *
 * act1/act2 are the identity in exact mode, MXFP8 (E4M3 elements, E8M0 scale
 * per 32 along the reduction dimension) in MXFP8-emulation mode, and bf16
 * rounding of the intermediate in bf16-emulation mode.
 *
 * A chain of layers runs them back to back over one token block, each
 * layer's output (optionally plus a residual) feeding the next.
 *
 * Beside the layer: the router logits that feed its top-k (a linear layer
 * with bf16 weights), a dense projection with MXFP8 weights (a layer outside
 * the experts, kept at FP8), and the rejection-sampling verification of a
 * block of drafted tokens (the step after the verify forward).
 *
 * Parity pins: every function below is checked by the CPU test-suite against
 * closed forms, format tables, library routines or brute force (see the
 * tests named test_oracle_*).  No function here is unpinned.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_ACT_EXACT 0
#define ORACLE_ACT_MXFP8 1
#define ORACLE_ACT_BF16 2

/* format decoders: exact values */
double oracle_e2m1_value(int code);   /* code in [0,16) */
double oracle_e8m0_value(int code);   /* code in [0,255): 2^(code-127); 255 -> NaN */
double oracle_e4m3_value(int code);   /* code in [0,256); 0x7F/0xFF -> NaN */
double oracle_bf16_value(uint16_t bits);

/* exact floor(log2(a)) of a positive finite fp32, read from its bits */
int oracle_floor_log2_f32(float a);

/* encoders: round to nearest, ties to the even code, saturating */
int oracle_e2m1_encode(double q);
int oracle_e4m3_encode(double q);
uint16_t oracle_bf16_from_double(double v);

/* MXFP4 packing of fp32 rows [R, K] (K % 32 == 0) */
void oracle_mxfp4_quantize(const float* w, int64_t R, int64_t K, uint8_t* out_fp4,
                           uint8_t* out_e8m0);

/* MXFP8 (E4M3) quantization of one row of K doubles (K % 32 == 0) */
void oracle_mxfp8_quantize_row(const double* v, int64_t K, uint8_t* codes, uint8_t* scales);

/* routing: top-k + renormalised softmax; idx [T,k] int32, gate [T,k] fp64 */
void oracle_route(const float* logits, int64_t T, int64_t E, int k, int32_t* idx,
                  double* gate);

/* stable counting sort of the (t, j) assignments by expert:
 * cnt[E], off[E+1], perm[T*k] (slot -> token), pos[T*k] (t*k+j -> slot) */
void oracle_route_arrays(const int32_t* idx, int64_t T, int k, int64_t E, int32_t* cnt,
                         int32_t* off, int32_t* perm, int32_t* pos);

/* The layer.  tokens (n_tokens entries) selects which rows of y to compute;
 * NULL means all T rows in order.  y_f64 [n_tokens, H] (before the final
 * bf16 rounding), y_bf16 [n_tokens, H], h_out [n_tokens, k, I] (act2 output)
 * may each be NULL.  n_threads <= 0 uses the OpenMP default.
 * Returns 0, or -1 on invalid arguments. */
int oracle_moe_forward(const uint16_t* x_bf16, const float* router_logits,
                       const uint8_t* w13_fp4, const uint8_t* w13_e8m0,
                       const uint8_t* w2_fp4, const uint8_t* w2_e8m0, int64_t T, int64_t H,
                       int64_t I, int64_t E, int k, int act_mode, const int64_t* tokens,
                       int64_t n_tokens, double* y_f64, uint16_t* y_bf16, double* h_out,
                       int n_threads);

/* A chain of n_layers layers over one token block: x_0 = x,
 * x_{l+1} = bf16_RNE(y_l + residual * x_l) with y_l layer l's fp64 output
 * (its own logits and weights, host arrays of n_layers pointers); writes x_L
 * to y_bf16 [T, H].  Returns 0, or -1 on invalid arguments. */
int oracle_moe_chain(int n_layers, const uint16_t* x_bf16, const float* const* router_logits,
                     const uint8_t* const* w13_fp4, const uint8_t* const* w13_e8m0,
                     const uint8_t* const* w2_fp4, const uint8_t* const* w2_e8m0, int64_t T,
                     int64_t H, int64_t I, int64_t E, int k, int act_mode, int residual,
                     uint16_t* y_bf16, int n_threads);

/* router logits [T, E] = x [T, H] (bf16) times W_r^T (W_r [E, H] bf16), exact fp64 */
void oracle_router_logits(const uint16_t* x_bf16, const uint16_t* w_bf16, int64_t T,
                          int64_t H, int64_t E, double* out);

/* MXFP8 packing of fp32 rows [R, K] (K % 32 == 0): E4M3 codes [R, K], E8M0 [R, K/32] */
void oracle_mxfp8_quantize(const float* w, int64_t R, int64_t K, uint8_t* codes,
                           uint8_t* scales);

/* dense FP8 projection y [T, N] = act(x [T, K]) W^T with MXFP8 weights W [N, K];
 * act_mode ORACLE_ACT_EXACT or ORACLE_ACT_MXFP8; y_f64 / y_bf16 may be NULL.
 * Returns 0, or -1 on invalid arguments. */
int oracle_dense_forward(const uint16_t* x_bf16, const uint8_t* w_e4m3, const uint8_t* w_e8m0,
                         int64_t T, int64_t K, int64_t N, int act_mode, double* y_f64,
                         uint16_t* y_bf16);

/* Rejection-sampling verification of a block of g drafted tokens per sequence
 * (see oracle.c): p [S, g+1, V], q [S, g, V] fp32 probabilities, draft [S, g],
 * u [S, g] fp32 uniforms in [0, 1), U [S] 64-bit uniforms; outputs n_acc [S]
 * and tokens [S, g+1] (-1 past the emitted token).  Returns 0, or -1 on
 * invalid arguments. */
int oracle_verify(const float* p, const float* q, const int32_t* draft, const float* u,
                  const uint64_t* U, int64_t S, int g, int64_t V, int32_t* n_acc,
                  int32_t* tokens);

#ifdef __cplusplus
}
#endif

#endif
