/*
 * moe_mxfp4.h — C ABI of libmoe_mxfp4.so: the MXFP4-weight Mixture-of-Experts
 * expert layer, run at DFlash verification token counts, on one B300
 * (sm_103a).
 *
 * What the layer is (sources):
 *  - MoE expert weights in MXFP4 (FP4 elements, block size 32, shared
 *    scale); everything outside the experts stays at higher precision:
 *    ai.appwright.xyz, tag page "投機的デコード", section "第1層：FP4量子化";
 *    techllm.github.io, "Xiaomi MiMo and TileRT push a 1-trillion-parameter
 *    model past 1000 tokens per second", section "1. MXFP4 — MoE에만 걸린
 *    양자화"; dothoosh.com, section "موتور فنی: کوانتیزاسیون و DFlash".
 *  - Token count: DFlash fills a masked block of up to 8 positions in one
 *    forward and the main model verifies the block, so each MoE layer sees
 *    T = sequences x 8 tokens: techllm.github.io, section "2. DFlash";
 *    dothoosh.com, section "جزئیات پیاده‌سازی DFlash" (block size capped at 8).
 *  - Decode is bound by weight bandwidth: ai.appwright.xyz, "第1層".
 *  - The layer definition the pages leave open (E2M1 grid, E8M0 scale rule,
 *    routing rule, SwiGLU, output type) is the layer specification this
 *    library implements, restated at each entry point below.
 *
 * Conventions for every entry point:
 *  - All tensors are caller-owned, row-major, contiguous device memory unless
 *    stated.  The library never frees caller memory and writes only the
 *    outputs named below.
 *  - Calls are stream-ordered and asynchronous; none synchronizes except
 *    moe_mxfp4_get_status.
 *  - Argument errors are detected on the host and returned before anything
 *    is launched.  Device-side faults (a bounded wait that expired, an index
 *    out of range) never trap: they set a device status word that
 *    moe_mxfp4_get_status returns.
 *  - Inputs must be finite; NaN/Inf give unspecified values (never a hang).
 *  - The library requires a device of compute capability 10.3 (B300).
 */
#ifndef MOE_MXFP4_H
#define MOE_MXFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* the CUDA runtime's stream and event handles (identical typedefs to driver_types.h) */
typedef struct CUstream_st* cudaStream_t;
typedef struct CUevent_st* cudaEvent_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,      /* null pointer, negative size, k out of range */
  MOE_ERR_UNSUPPORTED_SHAPE = -2, /* H or I not a multiple of 32, E or k too large */
  MOE_ERR_ALIGNMENT = -3,        /* a pointer is not aligned as documented */
  MOE_ERR_CUDA = -4,             /* a CUDA runtime call failed (launch, alloc, ...) */
  MOE_ERR_NO_MEMORY = -5,        /* workspace could not be allocated / is too small */
  MOE_ERR_DEVICE_TIMEOUT = -6,   /* a bounded device-side wait expired */
  MOE_ERR_DEVICE_FAULT = -7,     /* a device-side bounds/consistency check failed */
  MOE_ERR_NO_DEVICE = -8         /* no device of compute capability 10.3 is current */
} moe_status;

#define MOE_MAX_K 16     /* largest top-k */
#define MOE_MAX_E 1024   /* largest expert count */
#define MOE_MAX_CHAIN 256 /* most layers of one moe_mxfp4_forward_chain call */

/* activation modes of moe_opts.act_mode */
#define MOE_ACT_MXFP8 0  /* x and h quantized to MXFP8-E4M3 (blocks of 32) */
#define MOE_ACT_BF16 1   /* x used as bf16, h rounded to bf16 */

/* execution paths of moe_opts.path (the bf16 mode always runs the multi path) */
#define MOE_PATH_AUTO 0       /* moe_mxfp4_select_path decides (MULTI or GEMMS) */
#define MOE_PATH_MULTI 1      /* routing kernels, GEMM1, GEMM2, combine */
#define MOE_PATH_PERSISTENT 2 /* the whole layer in one launch for T <= 32 (routing,
                                 activation step, both GEMMs, combine; for the routed
                                 layer the router too); above that the routing kernels,
                                 then one launch for both GEMMs and the combine */
#define MOE_PATH_GEMMS 3      /* routing kernels, one launch for both GEMMs, combine */

/*
 * moe_mxfp4_forward — the MoE expert layer.
 *
 *   y[t] = bf16_RNE( sum_{j<k} g[t,j] * W2_{e_j} act2( silu(W1_{e_j} act1(x[t]))
 *                                                   * (W3_{e_j} act1(x[t])) ) )
 *
 * Routing: (e_j) are the k largest router_logits[t] in descending order, the
 * lower expert index first among equal logits; g[t,:] is the softmax of the
 * k selected logits.  W1 = rows [0, I) and W3 = rows [I, 2I) of the expert's
 * w13; each weight is e2m1(code) * 2^(scale - 127).  act1/act2 quantize to
 * MXFP8-E4M3 along the reduction dimension (the default) — see
 * moe_mxfp4_forward_ex for the bf16 mode.  silu(z) = z / (1 + e^-z).  The
 * gate-weighted sum is accumulated in fp32 in slot order j = 0..k-1 (the
 * result is deterministic run to run).
 *
 * Arguments (all device pointers):
 *  x_bf16         [T, H]       bf16 activations
 *  router_logits  [T, E]       fp32
 *  w13_fp4        [E, 2I, H/2] packed E2M1, element 2i in the low nibble of
 *                              byte i
 *  w13_e8m0       [E, 2I, H/32] one E8M0 scale per 32 elements along H
 *  w2_fp4         [E, H, I/2]  packed E2M1
 *  w2_e8m0        [E, H, I/32]
 *  T >= 0 (T = 0 returns MOE_OK and launches nothing), H and I multiples of
 *  32, 1 <= E <= MOE_MAX_E, 1 <= k <= min(E, MOE_MAX_K)
 *  y_bf16         [T, H]       bf16 output, overwritten
 *  stream         CUDA stream the work is ordered on (0 = legacy default)
 * Every pointer must be 16-byte aligned.  The GEMMs load FP4 weight rows 128
 * elements at a time by TMA (the 16U4_ALIGN16B operand form), so they take
 * H and I multiples of 128 and FP4 weights 32-byte aligned directly; any other
 * layer (H or I a multiple of 32 only, or FP4 weights 16-byte aligned only)
 * runs on zero-padded copies made in the scratch on every call — H and I
 * rounded up to multiples of 128, the copies' extra weights, scales and
 * activations zero — which gives the same y (zero terms add nothing to any
 * sum, and the padding is whole blocks of 32) at the cost of copying the
 * weights each call.  Scratch space comes from a
 * library-owned per-device cache that grows on first use of a larger shape
 * (a cudaMalloc outside any stream capture).
 * Sharing: every call on a device that is not given its own workspace
 * (moe_mxfp4_forward, and the other entry points that say they use the
 * library's scratch) uses that one cache.  Such calls must be ordered on the
 * GPU (one stream, or events between streams) — calls that overlap there race
 * on the scratch and give wrong results — and must not run at the same time
 * on the host either: growing the cache frees the previous buffer, which a
 * call on another host thread may still be enqueueing work on.  Callers that
 * run layers concurrently give each stream its own workspace through
 * moe_mxfp4_forward_ex (or moe_mxfp4_forward_chain's options).
 * Returns MOE_OK or an moe_status error (host-detected errors launch nothing).
 */
int moe_mxfp4_forward(const void* x_bf16, const float* router_logits, const uint8_t* w13_fp4,
                      const uint8_t* w13_e8m0, const uint8_t* w2_fp4, const uint8_t* w2_e8m0,
                      int T, int H, int I, int E, int k, void* y_bf16, cudaStream_t stream);

typedef struct {
  int act_mode;           /* MOE_ACT_MXFP8 (0) or MOE_ACT_BF16 (1) */
  int path;               /* MOE_PATH_* */
  void* workspace;        /* optional caller scratch (device, 256-byte aligned) */
  size_t workspace_bytes; /* >= moe_mxfp4_workspace_size(...) when workspace != NULL */
  uint32_t debug_flags;   /* 0 in normal use; see MOE_DEBUG_* */
  /* optional step markers: caller-created events; the library records
   * step_events[i] on `stream` just before the i-th kernel of the call and one
   * more after the last (i < n_step_events).  Kernel order: multi path —
   * route_topk, route_permute, act_quant, gemm1, gemm2, combine (for
   * T <= 32 the first three are one kernel, route_act, unless
   * MOE_DEBUG_SPLIT_ROUTING); persistent path — for T <= 32 one kernel, the
   * whole layer (with the router too for moe_mxfp4_forward_routed), else
   * route_topk, route_permute, act_quant, gemm1+gemm2+combine.
   * moe_mxfp4_forward_routed otherwise puts router_gemm, router_sum first;
   * router_sum adds the split partials into the logits and, where route_topk
   * would follow (the split routing kernels), already takes the top-k, so
   * route_topk is left out there. */
  cudaEvent_t* step_events;
  int n_step_events;
} moe_opts;

/* debug_flags: cap every bounded device wait at ~1 ms instead of ~2 s; used
 * to exercise the timeout path without faulting anything */
#define MOE_DEBUG_SHORT_TIMEOUT 1u
/* debug_flags: on the paths that run both GEMMs in one launch
 * (MOE_PATH_PERSISTENT, MOE_PATH_GEMMS; MXFP8 mode), make GEMM2 wait for a
 * GEMM1 publication that never comes, so the
 * cross-CTA dependency wait runs out (after ~1 ms with MOE_DEBUG_SHORT_TIMEOUT):
 * the call then reports MOE_ERR_DEVICE_TIMEOUT through moe_mxfp4_get_status and
 * y is unspecified.  Exercises the device timeout path without any fault;
 * ignored by the other paths. */
#define MOE_DEBUG_FORCE_DEP_TIMEOUT 2u
/* debug_flags: run routing and the activation step as three kernels even for
 * T <= 32 (where they are normally one kernel, for one layer and for a chain);
 * the results are identical — used by the tests to compare the two */
#define MOE_DEBUG_SPLIT_ROUTING 4u
/* debug_flags: in the bf16 mode, GEMM1's MMA warp never hands decoded weight
 * buffers back to the decoders, so their bounded wait runs out (~1 ms with
 * MOE_DEBUG_SHORT_TIMEOUT): the call reports MOE_ERR_DEVICE_TIMEOUT and y is
 * unspecified.  Exercises that kernel's timeout path without any fault. */
#define MOE_DEBUG_STALL_DECODE 8u

/*
 * moe_mxfp4_forward_ex — moe_mxfp4_forward with options (NULL opts = defaults).
 * With a caller workspace the call allocates nothing.
 *
 * act_mode = MOE_ACT_BF16 ("bf16 after dequant": the expert weights dequantised
 * and the activations kept in bf16 — an alternative to MXFP8 activations in
 * the problem statement): act1 is the identity on the bf16 x, every weight is
 * decoded exactly to bf16 (e2m1 * 2^(code - 127); exact for every E8M0 code up
 * to 252 — the largest a quantiser of fp32 weights emits — while 253 and 254
 * can overflow bf16), act2 rounds h = silu(gate) * up to bf16 (nearest even),
 * and the GEMMs accumulate in fp32 (tcgen05 kind::f16, the weights decoded
 * into tensor memory).  Bar: rel-Frobenius <= 5e-3 against the exact layer.
 */
int moe_mxfp4_forward_ex(const void* x_bf16, const float* router_logits, const uint8_t* w13_fp4,
                         const uint8_t* w13_e8m0, const uint8_t* w2_fp4, const uint8_t* w2_e8m0,
                         int T, int H, int I, int E, int k, void* y_bf16, cudaStream_t stream,
                         const moe_opts* opts);

/*
 * moe_mxfp4_forward_chain — n_layers expert layers back to back over one block
 * of T tokens, the pipeline kept on the GPU instead of one call per layer
 * (dothoosh.com, section "TileRT": the whole computational pipeline resident
 * and prefetched; techllm.github.io, "Xiaomi MiMo and TileRT ...", section
 * "3. TileRT").  The pages give no formula for the hand-off between layers;
 * it is read as composition with an optional residual stream:
 *
 *   x_0 = x,  x_{l+1} = bf16_RNE( y_l + residual * x_l ),  y_bf16 = x_{n_layers}
 *
 * where y_l is layer l's gate-weighted sum (moe_mxfp4_forward before its
 * final rounding, with layer l's own logits and weights; the residual is added
 * in fp32 after the sum).  With residual = 0 the result is bit-identical to
 * n_layers successive moe_mxfp4_forward_ex calls with the same options.
 *
 * All layers are routed first (routing reads only the given logits); each
 * layer's combine then writes the next layer's activation rows directly.
 *
 * Arguments: router_logits, w13_fp4, w13_e8m0, w2_fp4, w2_e8m0 are HOST
 * arrays of n_layers device pointers, each as in moe_mxfp4_forward (one
 * layer's tensors); the shape (T, H, I, E, k) is shared by all layers.
 * Chains take only the widths the GEMMs read directly: H and I multiples of
 * 128 and FP4 weights 32-byte aligned (MOE_ERR_UNSUPPORTED_SHAPE /
 * MOE_ERR_ALIGNMENT otherwise; no padded copies).
 * 1 <= n_layers <= MOE_MAX_CHAIN; residual is 0 or 1; y_bf16 [T, H] may equal
 * x_bf16.  opts as moe_mxfp4_forward_ex (act_mode, path, workspace of at least
 * moe_mxfp4_workspace_size_chain bytes, debug flags); step markers follow the
 * kernel order: route_topk (every layer), route_permute (every layer),
 * act_quant (layer 0), then per layer its GEMM kernel(s) and combine; for
 * T <= 32 the first three are one kernel, route_act (unless
 * MOE_DEBUG_SPLIT_ROUTING), with the same results.
 * Returns MOE_OK or an moe_status error (host-detected errors launch nothing).
 */
int moe_mxfp4_forward_chain(int n_layers, const void* x_bf16, const float* const* router_logits,
                            const uint8_t* const* w13_fp4, const uint8_t* const* w13_e8m0,
                            const uint8_t* const* w2_fp4, const uint8_t* const* w2_e8m0, int T,
                            int H, int I, int E, int k, int residual, void* y_bf16,
                            cudaStream_t stream, const moe_opts* opts);

/* scratch bytes moe_mxfp4_forward_chain needs (0 for an invalid shape) */
size_t moe_mxfp4_workspace_size_chain(int n_layers, int T, int H, int I, int E, int k,
                                      int act_mode);

/*
 * moe_mxfp4_select_path — the path MOE_PATH_AUTO takes for this shape on the
 * current device: MOE_PATH_GEMMS when a bound on the GEMM work items
 * (min(T*k, E) + T*k / chunk) * (I/128 + ceil(H/256)) is at most 110 per SM,
 * else MOE_PATH_MULTI (always MOE_PATH_MULTI in the bf16 mode).  One launch
 * for both GEMMs saves the gap between them and fills GEMM1's last wave with
 * GEMM2 items; with many items per SM two launches stream weights faster.  The automatic choice never takes
 * MOE_PATH_PERSISTENT: on this part its serial start (routing and the
 * activation step inside the launch) costs more than the launches it saves,
 * which overlap one another.  Every path gives bitwise equal results.
 * Returns a negative moe_status on invalid arguments.  No counterpart in the
 * papers: a support call.
 */
int moe_mxfp4_select_path(int T, int H, int I, int E, int k, int act_mode);

/* bytes of scratch a forward of this shape needs (0 on invalid arguments) */
size_t moe_mxfp4_workspace_size(int T, int H, int I, int E, int k, int act_mode);

/*
 * moe_mxfp4_workspace_size_padded — scratch bytes of a layer call that runs on
 * zero-padded copies (see moe_mxfp4_forward): what a caller workspace must
 * hold when the FP4 weight pointers are 16- but not 32-byte aligned (for H or
 * I not multiples of 128, moe_mxfp4_workspace_size already returns this).
 * routed = 1 for moe_mxfp4_forward_routed (the router weights are copied
 * too), 0 otherwise.  Returns 0 for unsupported arguments.
 */
size_t moe_mxfp4_workspace_size_padded(int T, int H, int I, int E, int k, int act_mode,
                                       int routed);

/*
 * moe_mxfp4_workspace_layout — where a forward leaves its intermediate arrays
 * inside a caller workspace (moe_opts.workspace of moe_mxfp4_forward_ex), so
 * that the routing, the permutation and the quantised activations the layer
 * actually used can be read back and checked after the call (the routing
 * arrays must equal the routing rule's bit for bit).  Byte offsets from the
 * workspace's start; after a call on that workspace completes:
 *  topk_idx [T, k] int32 and topk_w [T, k] fp32   step (1)
 *  cnt [E] int32, off [E+1] int32                 steps (2)-(3)
 *  perm [T*k] int32 (slot -> token),
 *  pos [T*k] int32 ((t*k + j) -> slot)            step (4): expert-major
 *                                                 slots, ascending t*k + j
 *                                                 within an expert
 *  xq [T*k, H], xs [T*k, H/32]                    act1(x) in slot order: E4M3
 *                                                 codes + E8M0 scales (MXFP8
 *                                                 mode) or bf16 copies (xs
 *                                                 unused)
 *  hq [T*k, I], hs [T*k, I/32]                    act2(h) in slot order, same
 *                                                 forms
 *  yp [T*k, H] fp32                               W2 act2(h) per slot
 *  logits [T, E] fp32                             the router's logits (the
 *                                                 routed layer's layout only;
 *                                                 SIZE_MAX otherwise)
 *  x_stream[2] [T, H] bf16                        SIZE_MAX here (chain only)
 *  total                                          moe_mxfp4_workspace_size
 * The layout depends only on the arguments.  A layer that runs on zero-padded
 * copies (H or I not a multiple of 128; see moe_mxfp4_forward) has the
 * padded shape's arrays at these offsets: rows of Hp = H rounded up to 128
 * (xq, xs, yp) and Ip (hq, hs) elements.  Returns MOE_OK or an error for
 * invalid arguments.  No counterpart in the papers: a support call for
 * checking the layer's steps one by one.
 */
typedef struct {
  size_t topk_idx, topk_w, cnt, off, perm, pos;
  size_t xq, xs, hq, hs, yp;
  size_t logits;
  size_t x_stream[2];
  size_t total;
} moe_workspace_layout;
int moe_mxfp4_workspace_layout(int T, int H, int I, int E, int k, int act_mode,
                               moe_workspace_layout* out);

/* the same for a workspace of moe_mxfp4_forward_routed (total =
 * moe_mxfp4_workspace_size_routed); logits holds the router's logits */
int moe_mxfp4_workspace_layout_routed(int T, int H, int I, int E, int k, int act_mode,
                                      moe_workspace_layout* out);

/*
 * moe_mxfp4_workspace_layout_chain — the same for layer `layer` (0 <= layer <
 * n_layers) of a moe_mxfp4_forward_chain workspace.  Every layer keeps its own
 * routing arrays (topk_idx .. pos, all valid after the call).  xq/xs, hq/hs
 * and yp are shared by the layers in turn: after the call xq/xs hold the last
 * layer's act1 input (written by the previous layer's combine, or by the
 * activation step when n_layers = 1), hq/hs and yp the last layer's.  With
 * residual = 1, x_stream[(n_layers - 1) & 1] holds x_{n_layers-1}, the last
 * layer's bf16 input (n_layers >= 2).
 */
int moe_mxfp4_workspace_layout_chain(int n_layers, int layer, int T, int H, int I, int E, int k,
                                     int act_mode, moe_workspace_layout* out);

/*
 * mxfp4_quantize — pack fp32 weights to MXFP4 with the layer's rule (offline).
 *  w        [rows, K] fp32 device, K a multiple of 32, 16-byte aligned
 *  out_fp4  [rows, K/2] packed E2M1 (element 2i in the low nibble of byte i)
 *  out_e8m0 [rows, K/32] E8M0 scale codes
 * Per block of 32 along K: amax = max |w|; scale code c = clamp(floor(log2(amax))
 * - 2 + 127, 0, 254) with floor(log2) read exactly from the fp32 bits (c = 0
 * when amax = 0); each element is q = w / 2^(c-127) rounded to the nearest of
 * {0, .5, 1, 1.5, 2, 3, 4, 6} (ties to the even code), saturated at 6, sign
 * from the input's sign bit.  Block size 32: ai.appwright.xyz, "第1層：FP4量子化".
 */
int mxfp4_quantize(const float* w, int64_t rows, int64_t K, uint8_t* out_fp4,
                   uint8_t* out_e8m0, cudaStream_t stream);

/*
 * moe_mxfp4_route — the routing steps alone (top-k + softmax, per-expert
 * histogram, prefix scan, stable permutation), for bit-exact checks.
 *  router_logits [T, E] fp32 device;  outputs (device):
 *  topk_idx [T, k] int32, topk_w [T, k] fp32, cnt [E] int32, off [E+1] int32,
 *  perm [T*k] int32 (slot -> token), pos [T*k] int32 ((t*k + j) -> slot).
 * Slots are expert-major; within an expert, ascending t*k + j.  The kernels
 * are those the forward runs for the same T: one launch of the small-block
 * routing kernel for T <= 32, the top-k and permutation kernels above.
 * Scratch (the chunk list) from the library-owned cache (shared: see the
 * ordering rules under moe_mxfp4_forward).
 */
int moe_mxfp4_route(const float* router_logits, int T, int E, int k, int32_t* topk_idx,
                    float* topk_w, int32_t* cnt, int32_t* off, int32_t* perm, int32_t* pos,
                    cudaStream_t stream);

/*
 * moe_mxfp8_quantize_rows — the MXFP8-E4M3 activation quantizer alone.
 *  x_bf16 [rows, K] device (K a multiple of 32) -> codes [rows, K] E4M3,
 *  scales [rows, K/32] E8M0.  Per block of 32: c = clamp(floor(log2(amax)) - 8
 *  + 127, 0, 254) (c = 0 when amax = 0); elements round to nearest even E4M3 of
 *  x / 2^(c-127), saturating at +-448.
 */
int moe_mxfp8_quantize_rows(const void* x_bf16, int64_t rows, int64_t K, uint8_t* codes,
                            uint8_t* scales, cudaStream_t stream);

/*
 * moe_mxfp4_forward_noalloc — moe_mxfp4_forward (same arguments, same result,
 * MXFP8 activations) for callers that cannot allocate device memory.  The
 * pages describe no such entry point; it exists for deployments where the
 * code that runs the layer is not allowed to call cudaMalloc and has no
 * workspace to hand over: plugin interfaces that give an operator only its
 * input and output buffers and plan all memory up front, runtimes whose
 * memory belongs to another allocator (a caching pool that direct cudaMalloc
 * calls would fragment or bypass), and real-time services that allocate
 * everything at start-up and forbid allocation on the serving path.
 *
 * Scratch: a file-scope device array of MOE_NOALLOC_SCRATCH_BYTES (80 MiB)
 * inside this library.  Every device that loads the library holds that array
 * until the process exits, whether or not this entry point is used.  The
 * first call on each device looks up the array's device address (and does the
 * library's other one-time set-up); make that first call before any stream
 * capture.  The call allocates nothing: no cudaMalloc, cudaFree or allocating
 * library routine.
 *
 * Limits and sharing:
 *  - Shapes whose scratch (moe_mxfp4_workspace_size(T, H, I, E, k, 0), or
 *    moe_mxfp4_workspace_size_padded(T, H, I, E, k, 0, 0) when the FP4
 *    weights are only 16-byte aligned) exceeds MOE_NOALLOC_SCRATCH_BYTES
 *    return MOE_ERR_NO_MEMORY before anything is launched; at H = 6144,
 *    I = 2048, E = 384, k = 8 the largest T is 317.
 *  - All calls share the one array and it keeps the last call's contents;
 *    nothing in it needs to start at zero (every scratch byte a call reads is
 *    written earlier in the same call).  Calls that overlap on the GPU (on
 *    different streams, or from different threads, without ordering between
 *    them) race on the array and give wrong results: order them.
 * Other arguments, alignment rules and errors: as moe_mxfp4_forward.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (80u * 1024u * 1024u)
int moe_mxfp4_forward_noalloc(const void* x_bf16, const float* router_logits,
                              const uint8_t* w13_fp4, const uint8_t* w13_e8m0,
                              const uint8_t* w2_fp4, const uint8_t* w2_e8m0, int T, int H, int I,
                              int E, int k, void* y_bf16, cudaStream_t stream);

/*
 * moe_router_topk — the router in front of the layer: logits = x W_r^T, then
 * the layer's top-k and softmax (step (1) of moe_mxfp4_forward).  The pages
 * name expert routing as part of the pipeline the runtime is built around
 * (techllm.github.io, "Xiaomi MiMo and TileRT ...", section "3. TileRT") but
 * give no formula; read as a linear layer with bf16 weights.
 *
 *  x_bf16         [T, H] bf16, device
 *  w_router_bf16  [E, H] bf16, device (one row of weights per expert)
 *  logits_out     [T, E] fp32, device, or NULL: the fp32 logits the top-k used
 *  topk_idx       [T, k] int32, device: experts in descending logit order,
 *                 the lower index first among equal logits
 *  topk_w         [T, k] fp32, device: softmax over the k selected logits
 * Shapes as moe_mxfp4_forward (H a multiple of 128, 1 <= E <= MOE_MAX_E,
 * 1 <= k <= min(E, MOE_MAX_K)); pointers 16-byte aligned.  The logits are
 * fp32 sums of exact bf16 products, accumulated on the tensor cores in K
 * ranges whose partial sums are added in a fixed order: deterministic run to
 * run.  Scratch from the library-owned cache (shared: see the ordering
 * rules under moe_mxfp4_forward).  Returns MOE_OK or an error.
 * No counterpart in the papers beyond the routing step itself.
 */
int moe_router_topk(const void* x_bf16, const void* w_router_bf16, int T, int H, int E, int k,
                    float* logits_out, int32_t* topk_idx, float* topk_w, cudaStream_t stream);

/*
 * moe_mxfp4_forward_routed — moe_mxfp4_forward_ex with the router fused in
 * front: router weights instead of router logits (see moe_router_topk); the
 * logits never leave the call.  opts as moe_mxfp4_forward_ex (NULL =
 * defaults); a caller workspace must hold moe_mxfp4_workspace_size_routed
 * bytes.  On the single-launch path (MXFP8 mode) with T <= 32 the router
 * runs inside the layer's one launch: each warp multiplies one expert's
 * weight row with every token row (exact bf16 products, fp32 sums in a fixed
 * order), one grid-wide barrier, then the routing; otherwise it is a
 * tensor-core GEMM in front (moe_router_topk's arithmetic).  Both orders stay
 * within the same error bound of the exact logits; each is deterministic.
 */
int moe_mxfp4_forward_routed(const void* x_bf16, const void* w_router_bf16,
                             const uint8_t* w13_fp4, const uint8_t* w13_e8m0,
                             const uint8_t* w2_fp4, const uint8_t* w2_e8m0, int T, int H, int I,
                             int E, int k, void* y_bf16, cudaStream_t stream,
                             const moe_opts* opts);

/* scratch bytes of moe_mxfp4_forward_routed (0 on invalid arguments) */
size_t moe_mxfp4_workspace_size_routed(int T, int H, int I, int E, int k, int act_mode);

/*
 * mxfp8_quantize — MXFP8 packing of fp32 rows (weights of a dense FP8 layer):
 * per block of 32 along K, scale code = clamp(floor(log2(amax)) - 8 + 127,
 * 0, 254) (amax = 0 gives code 0), elements = E4M3(w / 2^(code - 127)),
 * round to nearest even, saturating at +-448 — the rule of the layer's
 * activations.
 *  w         [rows, K] fp32, device, 16-byte aligned; K a multiple of 32
 *  out_e4m3  [rows, K] uint8, device, 16-byte aligned
 *  out_e8m0  [rows, K/32] uint8, device
 */
int mxfp8_quantize(const float* w, int64_t rows, int64_t K, uint8_t* out_e4m3, uint8_t* out_e8m0,
                   cudaStream_t stream);

/*
 * moe_fp8_dense_forward — a dense projection with MXFP8 weights, the
 * precision the pages keep outside the experts (techllm.github.io, "Xiaomi
 * MiMo and TileRT ...", section "1. MXFP4 — MoE에만 걸린 양자화";
 * ai.appwright.xyz, tag page "投機的デコード", section "第1層：FP4量子化": o_proj
 * stays out of FP4):
 *   y[t, n] = bf16_RNE( sum_k mxfp8(x)[t, k] * w[n, k] ),
 * w = e4m3(code) * 2^(scale - 127), x quantized to MXFP8 along K exactly as
 * the layer's activations.
 *  x_bf16    [T, K] bf16, device
 *  w_e4m3    [N, K] uint8 E4M3 codes, device (see mxfp8_quantize)
 *  w_e8m0    [N, K/32] uint8 scale codes, device
 *  y_bf16    [T, N] bf16, device, overwritten
 * K a multiple of 128, N a multiple of 4, T >= 0 (0 = no-op); pointers
 * 16-byte aligned.  The MMA accumulates in fp32 over K ranges whose partial
 * sums are added in a fixed order (deterministic).  Scratch from the
 * library-owned cache (shared: see the ordering rules under
 * moe_mxfp4_forward).  Returns MOE_OK or an error (host-detected errors
 * launch nothing).
 */
int moe_fp8_dense_forward(const void* x_bf16, const uint8_t* w_e4m3, const uint8_t* w_e8m0,
                          int T, int K, int N, void* y_bf16, cudaStream_t stream);

/*
 * moe_verify_block — rejection-sampling verification of a block of drafted
 * tokens per sequence, the step after the verify forward (lossless
 * speculative decoding: techllm.github.io, "Xiaomi MiMo and TileRT ...",
 * section "2. DFlash"; blocks of at most 8 positions: dothoosh.com, section
 * "جزئیات پیاده‌سازی DFlash").  For sequence s:
 *   drafted token d_i (i = 0..g-1) is accepted while u_i * q_i(d_i) < p_i(d_i),
 *   the fp32 values compared exactly (in fp64);
 *   at the first rejection i one token is drawn from max(0, p_i - q_i) (fp32
 *   difference), after g acceptances from p_g; if the residual has no mass,
 *   from p_i.  A draw is the first token x whose running sum of fixed-point
 *   masses floor(w * 2^62) exceeds floor(U[s] * M / 2^64), M the total mass:
 *   bit-reproducible, independent of any summation order.
 *  p       [S, g+1, V] fp32 target probabilities (rows of at most 2 total mass)
 *  q       [S, g, V]   fp32 draft probabilities
 *  draft   [S, g]      int32 drafted tokens (outside [0, V): a rejection and
 *                      MOE_ERR_DEVICE_FAULT in the status word)
 *  u       [S, g]      fp32 uniforms in [0, 1) for the accept tests
 *  U       [S]         64-bit uniforms for the draw
 *  n_acc   [S]         int32 out: accepted drafts, 0..g
 *  tokens  [S, g+1]    int32 out: the accepted drafts, then the drawn token,
 *                      then -1
 * All device pointers, 4-byte aligned (U 8-byte); 1 <= g <= MOE_VERIFY_MAX_DRAFT,
 * 1 <= V <= 2^21 (MOE_ERR_UNSUPPORTED_SHAPE above), S >= 0 (0 = no-op).
 * Scratch from the library-owned cache (shared: see the ordering rules under
 * moe_mxfp4_forward).
 * The random numbers are inputs: the call is deterministic.
 */
#define MOE_VERIFY_MAX_DRAFT 64
int moe_verify_block(const float* p, const float* q, const int32_t* draft, const float* u,
                     const uint64_t* U, int S, int g, int64_t V, int32_t* n_acc, int32_t* tokens,
                     cudaStream_t stream);

/*
 * moe_mxfp4_get_status — synchronizes `stream`, returns the first device-side
 * error recorded since the last call (MOE_OK if none) and clears it.  A CUDA
 * error seen while synchronizing returns MOE_ERR_CUDA.
 */
int moe_mxfp4_get_status(cudaStream_t stream);

/* number of kernels this library has launched in this process (all devices,
 * all entry points); a diagnostic for counting launches in a timed region */
uint64_t moe_mxfp4_launch_count(void);

/* number of device allocations (cudaMalloc) this library has made in this
 * process (all devices): its scratch cache growing.  A diagnostic: a call
 * that must not allocate leaves it unchanged. */
uint64_t moe_mxfp4_alloc_count(void);

/* human-readable name of an moe_status value (static string) */
const char* moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif
