// Shared definitions of the MXFP4 MoE layer library: status word, workspace
// layout, small device helpers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_mxfp4.h"

namespace moe {

// Assignments of one expert are processed in chunks of at most this many
// slots (tokens); a chunk is the N dimension of one GEMM work item.  Narrow
// chunks keep the GEMM pipeline deep (small activation tiles: six stages in
// flight); wide chunks cut the MMA instructions per token when experts
// receive many tokens.
#ifndef MOE_CHUNK_NARROW
#define MOE_CHUNK_NARROW 32
#endif
constexpr int kChunkNarrow = MOE_CHUNK_NARROW;
#ifndef MOE_CHUNK_WIDE
#define MOE_CHUNK_WIDE 96
#endif
constexpr int kChunkWide = MOE_CHUNK_WIDE;
// layers with at least this many tokens use wide chunks (MXFP8 mode)
#ifndef MOE_WIDE_MIN_TOKENS
#define MOE_WIDE_MIN_TOKENS 512
#endif
constexpr int kWideMinTokens = MOE_WIDE_MIN_TOKENS;
constexpr int kStatusTimeout = MOE_ERR_DEVICE_TIMEOUT;
constexpr int kStatusFault = MOE_ERR_DEVICE_FAULT;

// Per-call device scratch.  Offsets are computed on the host by
// workspace_layout(); every sub-buffer starts on a 256-byte boundary.
struct Work {
  int32_t* topk_idx;  // [T*k]
  float* topk_w;      // [T*k]
  int32_t* cnt;       // [E]
  int32_t* off;       // [E+1]
  int32_t* perm;      // [T*k] slot -> token
  int32_t* pos;       // [T*k] (t*k+j) -> slot
  int4* chunks;       // [max_chunks] {expert, first slot, n slots, 0}
  int32_t* done;      // [max_chunks] GEMM1 publications per chunk (persistent path)
  int32_t* meta;      // [0] chunk count, [1] touched experts, [2..] step counters
  uint8_t* xq;        // [T*k, H] E4M3 (MXFP8) or [T*k, H] bf16 (bf16 mode)
  uint8_t* xs;        // [T*k, H/32] E8M0
  uint8_t* hq;        // [T*k, I] E4M3 or bf16
  uint8_t* hs;        // [T*k, I/32]
  float* yp;          // [T*k, H] per-slot expert outputs (fp32)
  float* part;        // router split-K partials [splits][T][E] (routed forward only)
  float* rlogits;     // router logits [T, E] (routed forward only)
  uint8_t* sync;      // grid-wide barrier words of the whole-layer launch
  int max_chunks;
};

// Programmatic dependent launch.  The kernels of a forward after the first
// are launched with the programmatic stream-serialization attribute, so one
// may start while the previous kernel still runs.  Such a kernel calls
// grid_dependency_wait() before touching any global memory that an earlier
// kernel of the call reads or writes: the wait returns once the preceding
// grid has completed and its writes are visible (at once when the kernel was
// launched without the attribute).  grid_launch_dependents() lets the next
// kernel be scheduled before this one ends.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void set_status(int* status, int code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// largest |v| over the warp in one instruction: non-negative floats order
// like their bit patterns, so an unsigned max of |v|'s bits is the exact
// float max for finite values (all 32 lanes must take part)
__device__ __forceinline__ float warp_max_abs(float v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(__float_as_uint(fabsf(v))));
  return __uint_as_float(r);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace moe
