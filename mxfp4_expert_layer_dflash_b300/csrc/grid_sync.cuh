// Grid-wide barriers of a persistent launch whose CTAs are all resident at
// once (a cooperative launch), built on memory that need not start at zero:
// the scratch they live in is reused by every call and may hold anything.
//
// Each CTA owns one 64-bit flag per barrier kind and arrives by storing the
// call's tag into it (release); a barrier is passed once every CTA's flag
// equals the tag (acquire).  The tag is (call number << 32 | host salt << 8 |
// kind): the call number is one more than the counter word in the scratch,
// which every CTA reads at its start and CTA 0 writes back once it has passed
// the launch's last barrier (every CTA has read it by then), so consecutive
// calls on one scratch never share a tag — also when a call is replayed from
// a CUDA graph, where the host's salt is frozen.  The salt (the host's count
// of calls) separates eager calls even after a call that gave up before
// writing the counter back.  A CTA that gives up stores the tag with kind
// 0xFF into the abort word, so the others stop waiting at once.
// Stale flags never match; arbitrary contents match only by chance (2^-64
// per word).
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kMaxGridSync = 256;  // most CTAs a synchronised launch may have
// barrier slots (one flag per CTA each).  Consecutive layers of a launch use
// alternate slots for the same barrier: a CTA with no work in a layer reaches
// that layer's barrier right after the previous one, and must not overwrite a
// flag another CTA still waits on.
constexpr int kSyncOut = 0;     // (+ layer % 2) every CTA's GEMM2 outputs of a layer are written
constexpr int kSyncLogits = 2;  // every CTA's router logits are written
constexpr int kSyncAct = 3;     // (+ layer % 2) every CTA's act1 rows of a layer are written
constexpr int kSyncKinds = 5;
// the low byte of a flag value: which event, and of which layer of the launch
constexpr uint64_t kChunkFlagKind = 0x10;   // + layer: a (chunk, GEMM1 tile pair) published
constexpr uint64_t kLogitsKind = 0x30;
constexpr uint64_t kOutKind = 0x40;         // + layer
constexpr uint64_t kActKind = 0x80;         // + layer
constexpr int kMaxLaunchLayers = 16;        // layers of one chained launch (kinds stay apart)
constexpr uint64_t kChunkFlagNever = 0xFE;  // a kind no flag ever holds (forced timeout)
// bytes of scratch before the per-chunk flags: the counter (8), the abort word
// (8), the barrier flags
constexpr size_t kGridSyncBytes = 16 + (size_t)kSyncKinds * kMaxGridSync * 8;

struct GridSync {
  uint32_t* counter;      // calls completed on this scratch
  uint64_t* abort;        // tag | 0xFF once some CTA has given up
  uint64_t* flags;        // [kSyncKinds][kMaxGridSync]
  uint64_t* chunk_flags;  // [chunks][GEMM1 tile pairs][4 epilogue warps]: that quarter of h
                          // is written
  uint32_t salt;          // host call number (low 24 bits used)
};

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// this call's tag (kind bits zero); every CTA calls it once at its start
__device__ __forceinline__ uint64_t grid_sync_tag(const GridSync& g) {
  uint32_t c;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(c) : "l"(g.counter) : "memory");
  return ((uint64_t)(c + 1u) << 32) | ((uint64_t)(g.salt & 0xFFFFFFu) << 8);
}

// CTA 0, once past the launch's last barrier: the next call takes the next tag
__device__ __forceinline__ void grid_sync_retire(const GridSync& g, uint64_t tag) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(g.counter), "r"((uint32_t)(tag >> 32))
               : "memory");
}

// One thread of the CTA, after the CTA's writes are ordered before it (a
// barrier among the writing threads): make them visible, then arrive at the
// barrier in `slot` with `value` (the call's tag | the event's kind).
__device__ __forceinline__ void grid_arrive(const GridSync& g, int slot, uint64_t value) {
  __threadfence();
  st_release_u64(g.flags + (size_t)slot * kMaxGridSync + blockIdx.x, value);
}

__device__ __forceinline__ void grid_give_up(const GridSync& g, uint64_t tag) {
  st_relaxed_u64(g.abort, tag | 0xFFull);
}

__device__ __forceinline__ bool grid_aborted(const GridSync& g, uint64_t tag) {
  return ld_relaxed_u64(g.abort) == (tag | 0xFFull);
}

// Warp-collective bounded wait until every CTA of the grid has arrived at the
// barrier in `slot` with `want` (a warp-uniform result: false on timeout, on
// the CTA's own abort flag or on another CTA's give-up).  A CTA arrives at the
// barriers of a slot in one order, and no CTA can arrive at the next before
// every CTA has passed this one, so a flag never skips past the value waited
// for.
__device__ __forceinline__ bool grid_wait(const GridSync& g, int slot, uint64_t want,
                                          uint64_t tag, unsigned long long timeout_ns,
                                          const volatile int* abort_cta) {
  const int lane = threadIdx.x & 31;
  const uint64_t* f = g.flags + (size_t)slot * kMaxGridSync;
  const int G = (int)gridDim.x;
  const uint64_t deadline = ptx::globaltimer() + timeout_ns;
  uint32_t spins = 0;
  while (true) {
    // relaxed loads, all in flight at once (acquire loads would wait for one
    // another); one fence after the last round makes them an acquire
    bool mine = true;
    for (int i = lane; i < G; i += 32) mine &= ld_relaxed_u64(f + i) == want;
    if (__all_sync(0xffffffffu, mine)) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");
      return true;
    }
    bool stop = false;
    if ((++spins & 7u) == 0)
      stop = *abort_cta || grid_aborted(g, tag) || ptx::globaltimer() > deadline;
    if (__any_sync(0xffffffffu, stop)) return false;
  }
}

// One thread, after the writes of a quarter of a (chunk, tile pair) of h are
// ordered before it: publish them to the other CTAs (and their TMA reads).
__device__ __forceinline__ void publish_chunk_tile(const GridSync& g, int idx, uint64_t value) {
  __threadfence();
  st_release_u64(g.chunk_flags + idx, value);
}

// Warp-collective: are flags [first, first + n) all equal to `want`?  Relaxed
// loads; the caller issues the acquire fence once the answer is yes.
__device__ __forceinline__ bool chunk_tiles_published(const GridSync& g, int first, int n,
                                                      uint64_t want) {
  bool mine = true;
  for (int i = threadIdx.x & 31; i < n; i += 32) mine &= ld_relaxed_u64(g.chunk_flags + first + i) == want;
  return __all_sync(0xffffffffu, mine);
}

__device__ __forceinline__ void fence_acquire_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// named barrier among `threads` threads (a multiple of 32) of the CTA
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace moe
