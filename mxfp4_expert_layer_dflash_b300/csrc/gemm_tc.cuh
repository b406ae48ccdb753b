// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05), MXFP8 mode.
//
// Swap-AB: the expert's weight rows fill the 128-row MMA dimension (A) and the
// expert's tokens (a chunk of at most kChunkMax slots, padded to 16) are N, so
// the tiny decode-time token count never pads the weight side.  A is FP4
// (E2M1) straight from HBM: TMA's 16U4_ALIGN16B mode expands each 16-element
// group into the 16-byte-aligned form the MMA reads, so no thread touches the
// weights.  B is the MXFP8-E4M3 activation tile.  The E8M0 scales of both
// operands are written into TMEM by a scale warpgroup and applied by the MMA
// per 32 elements (kind::mxf8f6f4, block_scale).  Decode is bound by weight
// bandwidth (ai.appwright.xyz, "第1層"); the pipeline keeps several weight
// tiles in flight per SM while the tensor cores work on earlier ones (the
// load/compute overlap of dothoosh.com, "TileRT", done here per kernel).
//
// Both GEMMs load two 128-row weight tiles per stage that share one
// activation tile: GEMM1 pairs gate rows [r, r+128) with up rows
// [I+r, I+r+128) (so the epilogue has both operands of silu(gate)*up for the
// same row and token); GEMM2 pairs output rows [r, r+128) with [r+128, r+256).
// Two weight boxes per pipeline round keep the fixed cost of a round small
// against the bytes it moves.
//
// Warp roles (384 threads, one CTA per SM, persistent over work items):
//   warp 0      TMA producer (weight tiles + activation tile), one lane
//   warp 2      TMEM owner and MMA issuer, one lane
//   warps 4-7   scale stagers: warp w owns TMEM lanes 32*(w%4).. and writes the
//               E8M0 words of each stage there with tcgen05.st, loading them
//               from global memory four to eight stages ahead into registers
//   warps 8-11  epilogue: TMEM -> registers -> SwiGLU + MXFP8 requant (GEMM1)
//               or fp32 rows of yp (GEMM2)
// Work item = (chunk of one expert's slots, one pair of weight tiles).
//
// Scale placement in TMEM (checked on the device by a layout probe): the MMA
// reads the A scale of row m from lane m, column sfa + m/32, and the B scale
// of token n from lane 32q + n%32 of every lane quarter q, column sfb + n/32;
// the byte inside the 32-bit word is the instruction descriptor's scale id
// (one per 32-element block of the 128-element stage).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "fmt.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kTcThreads = 384;
constexpr int kBlockK = 128;   // K elements per stage: one TMA box of FP4
constexpr int kBoxRowsB = 16;  // activation rows per TMA box
constexpr int kSfGroup = 4;    // fills per scale load group (16 bytes of scales per row)

// Tuning knob (compile-time): MOE_TC_PF_W = L2 prefetch distance of weight
// tiles in pipeline fills (0 = off)
#ifndef MOE_TC_PF_W
#define MOE_TC_PF_W 0
#endif
#ifndef MOE_TC_PF_EVERY
#define MOE_TC_PF_EVERY 1  // prefetch every k-stage's boxes (or every n-th)
#endif
// MOE_TC_PF_LSU = distance in fills at which warp 1 prefetches weight rows into
// L2 with plain prefetch instructions (which bypass the TMA engine); 0 = off
#ifndef MOE_TC_PF_LSU
#define MOE_TC_PF_LSU 0
#endif

struct TcParams {
  CUtensorMap map_w;  // FP4 weights [E*R rows, K], 16U4_ALIGN16B, box {128, 128}, SW128
  CUtensorMap map_x;  // E4M3 activations [T*k rows, K], u8, box {128, 16}, SW128
  const uint8_t* w_packed;  // [E*R, K/2] the packed weights map_w describes
  const uint8_t* w_sf;  // [E*R, K/32]
  const uint8_t* x_sf;  // [T*k, K/32]
  const int4* chunks;
  const int32_t* meta;
  uint8_t* hq;  // GEMM1 out: [T*k, I] E4M3
  uint8_t* hs;  // GEMM1 out: [T*k, I/32]
  float* yp;    // GEMM2 out: [T*k, H]
  int K;         // reduction length
  int R;         // weight rows per expert (2I or H)
  int m_tiles;   // tile pairs per expert (I/128 for GEMM1, H/256 for GEMM2)
  int m_stride;  // weight rows between consecutive tile pairs (128 or 256)
  int half;      // row offset of the second tile of a pair (I or 128)
  int out_dim;   // row length of the output (I or H)
  int rows_total;  // E * R: weight rows in the tensor (guards the odd last tile pair)
  int* status;
  unsigned long long timeout_ns;
};

template <bool kGated, int kNMax>
struct TcCfg {
  static constexpr int kA = 2;                 // A tiles per stage
  static constexpr int kATile = 128 * 128;     // unpacked FP4 tile bytes
  static constexpr int kBTile = kNMax * 128;
  static constexpr int kStageBytes = kA * kATile + kBTile;  // multiple of 1024
  static constexpr int kStages = (232448 - 1024 - 256) / kStageBytes;
  static constexpr int kAccCols = kA * kNMax;  // one accumulator buffer (gate|up or lo|hi)
  static constexpr int kSfStride = 16;         // TMEM columns per stage of scales
  // accumulators are double-buffered when TMEM has room for two
  static constexpr int kAccBufs = 2 * kAccCols + kStages * kSfStride <= 512 ? 2 : 1;
  static constexpr int kSfBase = kAccBufs * kAccCols;   // TMEM column of stage 0's scales
  static constexpr int kSfbCol = 4 * kA;       // B scales after the A scale columns
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kTxA = 128 * 64;   // packed bytes of one weight box
  static constexpr int kWords = kA + kNMax / 32;  // scale words per lane per stage
  static constexpr int kBarBytes = 256;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kBarBytes;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kNMax % 32 == 0 && kNMax <= 128, "B-scale columns per stage");
  static_assert(kSfBase + kStages * kSfStride <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

// Walks the (work item, k-stage) sequence of one CTA.
struct FillCursor {
  int item, ks, n_items, ksteps, m_tiles, step;
  int4 ch;
  int mt;
  __device__ __forceinline__ void start(int first, int n, int kst, int mtl, int stp,
                                        const int4* chunks) {
    item = first;
    ks = 0;
    n_items = n;
    ksteps = kst;
    m_tiles = mtl;
    step = stp;
    ch = make_int4(0, 0, 0, 0);
    mt = 0;
    load(chunks);
  }
  __device__ __forceinline__ bool valid() const { return item < n_items; }
  __device__ __forceinline__ void load(const int4* chunks) {
    if (item < n_items) {
      ch = chunks[item / m_tiles];
      mt = item % m_tiles;
    }
  }
  __device__ __forceinline__ void next(const int4* chunks) {
    if (++ks == ksteps) {
      ks = 0;
      item += step;
      load(chunks);
    }
  }
};

template <bool kGated, int kNMax>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<kGated, kNMax>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* prod_fill = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1 + 4);  // TMA arrive.expect_tx + one arrival per scale warp
      ptx::mbar_init(&empty[s], 1);     // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&acc_full[b], 1);   // MMA commit
      ptx::mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }  // (only C::kAccBufs of the two are used)
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    *prod_fill = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 2) {
    ptx::tmem_alloc(tmem_slot, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&p.map_w);
    ptx::prefetch_tmap(&p.map_x);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  const int n_items = p.meta[0] * p.m_tiles;
  const int ksteps = p.K / kBlockK;
  const int sf_row = p.K / 32;  // scale bytes per row
  auto fail = [&](int code) {
    set_status(p.status, code);
    *abort_flag = 1;
  };
  auto deadline = [&]() { return ptx::globaltimer() + p.timeout_ns; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = ptx::policy_evict_first(), pol_x = ptx::policy_evict_last();
      FillCursor pf;  // lookahead: weight tiles prefetched into L2 MOE_TC_PF_W fills ahead
      pf.start(blockIdx.x, n_items, ksteps, p.m_tiles, gridDim.x, p.chunks);
      auto pf_step = [&]() {
        if (pf.valid() && (pf.ks % MOE_TC_PF_EVERY) == 0) {
          const int prow = pf.ch.x * p.R + pf.mt * p.m_stride;
          ptx::tma_prefetch_2d(&p.map_w, pf.ks * kBlockK, prow);
          ptx::tma_prefetch_2d(&p.map_w, pf.ks * kBlockK, prow + p.half);
        }
        pf.next(p.chunks);
      };
      for (int i = 0; i < MOE_TC_PF_W; ++i) pf_step();
      FillCursor c;
      c.start(blockIdx.x, n_items, ksteps, p.m_tiles, gridDim.x, p.chunks);
      for (uint32_t fill = 0; c.valid(); ++fill, c.next(p.chunks)) {
        const int s = (int)(fill % C::kStages);
        const uint32_t use = fill / C::kStages;
        if (!ptx::mbar_wait(&empty[s], (use & 1) ^ 1, deadline(), abort_flag)) {
          fail(kStatusTimeout);
          break;
        }
        const int nrows = (c.ch.z + 15) & ~15;
        const int row0 = c.ch.x * p.R + c.mt * p.m_stride;
        const uint32_t tx = C::kA * C::kTxA + (uint32_t)nrows * 128;
        uint8_t* st = smem + s * C::kStageBytes;
        ptx::mbar_arrive_expect_tx(&full[s], tx);
        ptx::tma_load_2d(st, &p.map_w, &full[s], c.ks * kBlockK, row0, pol_w);
        ptx::tma_load_2d(st + C::kATile, &p.map_w, &full[s], c.ks * kBlockK, row0 + p.half, pol_w);
        for (int r = 0; r < nrows; r += kBoxRowsB)
          ptx::tma_load_2d(st + C::kA * C::kATile + r * 128, &p.map_x, &full[s], c.ks * kBlockK,
                           c.ch.y + r, pol_x);
        if (MOE_TC_PF_W > 0) pf_step();
        if (MOE_TC_PF_LSU > 0) *prod_fill = fill + 1;
      }
    }
  } else if (warp == 1 && MOE_TC_PF_LSU > 0) {
    // ------------------------------------------------------------ L2 prefetcher
    // Keeps the weight rows of the fills MOE_TC_PF_LSU ahead of the TMA
    // producer in L2; one 128-byte line per row covers two k-stages.
    FillCursor pf;
    pf.start(blockIdx.x, n_items, ksteps, p.m_tiles, gridDim.x, p.chunks);
    const uint8_t* wbase = reinterpret_cast<const uint8_t*>(p.w_packed);
    const int64_t row_bytes = p.K / 2;
    uint32_t pfill = 0;
    uint64_t idle_since = ptx::globaltimer();
    while (pf.valid() && !*abort_flag) {
      if (pfill < *prod_fill + MOE_TC_PF_LSU) {
        if ((pf.ks & 1) == 0) {
          const int64_t row0 = (int64_t)pf.ch.x * p.R + pf.mt * p.m_stride;
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const int64_t row = row0 + a * p.half + qq * 32 + lane;
              if (row < p.rows_total) ptx::prefetch_l2(wbase + row * row_bytes + pf.ks * 64);
            }
        }
        ++pfill;
        pf.next(p.chunks);
        idle_since = ptx::globaltimer();
      } else if (ptx::globaltimer() - idle_since > p.timeout_ns) {
        break;  // the producer stopped advancing; nothing to report, just stop prefetching
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t fill = 0;
      bool ok = true;
      int j = 0;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++j) {
        const int4 ch = p.chunks[item / p.m_tiles];
        const uint32_t N = (uint32_t)((ch.z + 15) & ~15);
        const int b = j % C::kAccBufs;
        const uint32_t u = (uint32_t)(j / C::kAccBufs);
        if (!ptx::mbar_wait(&acc_empty[b], (u & 1) ^ 1, deadline(), abort_flag)) {
          fail(kStatusTimeout);
          break;
        }
        ptx::tc_fence_after();
        const uint32_t acc0 = tbase + b * C::kAccCols;
        const uint32_t acc1 = acc0 + kNMax;
        for (int ks = 0; ks < ksteps; ++ks, ++fill) {
          const int s = (int)(fill % C::kStages);
          const uint32_t use = fill / C::kStages;
          if (!ptx::mbar_wait(&full[s], use & 1, deadline(), abort_flag)) {
            fail(kStatusTimeout);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t st = ptx::smem_u32(smem + s * C::kStageBytes);
          const uint32_t sa0 = st, sa1 = st + C::kATile, sb = st + C::kA * C::kATile;
          const uint32_t tsf = tbase + C::kSfBase + s * C::kSfStride;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t idesc = ptx::idesc_mxf8f6f4(N, kk, kk);
            const uint32_t accum = (ks | kk) ? 1u : 0u;
            ptx::mma_mxf8f6f4(acc0, ptx::desc_kmajor_sw128(sa0 + 32 * kk),
                              ptx::desc_kmajor_sw128(sb + 32 * kk), idesc, tsf, tsf + C::kSfbCol,
                              accum);
            ptx::mma_mxf8f6f4(acc1, ptx::desc_kmajor_sw128(sa1 + 32 * kk),
                              ptx::desc_kmajor_sw128(sb + 32 * kk), idesc, tsf + 4,
                              tsf + C::kSfbCol, accum);
          }
          ptx::mma_commit(&empty[s]);  // frees the smem stage and its scale columns
        }
        if (!ok) break;
        ptx::mma_commit(&acc_full[b]);
      }
      ptx::mma_commit(drain);
      if (!ptx::mbar_wait(drain, 0, deadline(), abort_flag)) fail(kStatusTimeout);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ scale stagers
    // Scale words are loaded a group of kSfGroup fills at a time, one group
    // ahead of the group being written into TMEM.  When the scale rows allow it
    // (K a multiple of 512), one 16-byte load per row covers the whole group,
    // which keeps the scale traffic to a quarter of the L2 requests.
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const bool vec = (sf_row % 16) == 0 && (ksteps % kSfGroup) == 0;
    FillCursor ld, stc;
    ld.start(blockIdx.x, n_items, ksteps, p.m_tiles, gridDim.x, p.chunks);
    stc = ld;
    // words of one fill for this lane: A scales of rows 32q+lane (+ second
    // tile), then B scales of tokens 32j+lane; absent words are 0
    uint32_t grp[2][kSfGroup][C::kWords];
    auto load_group = [&](uint32_t (&g)[kSfGroup][C::kWords]) {
#pragma unroll
      for (int i = 0; i < kSfGroup; ++i)
#pragma unroll
        for (int w = 0; w < C::kWords; ++w) g[i][w] = 0;
      if (vec) {  // the group's fills are ks .. ks+3 of one work item
        if (ld.valid()) {
          const int64_t row = (int64_t)ld.ch.x * p.R + ld.mt * p.m_stride + q * 32 + lane;
#pragma unroll
          for (int a = 0; a < C::kA; ++a) {
            if (row + a * p.half < p.rows_total) {
              const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                  p.w_sf + (row + a * p.half) * sf_row + ld.ks * 4));
              g[0][a] = v.x;
              g[1][a] = v.y;
              g[2][a] = v.z;
              g[3][a] = v.w;
            }
          }
#pragma unroll
          for (int jb = 0; jb < kNMax / 32; ++jb) {
            const int n = jb * 32 + lane;
            if (n < ld.ch.z) {
              const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                  p.x_sf + (int64_t)(ld.ch.y + n) * sf_row + ld.ks * 4));
              g[0][C::kA + jb] = v.x;
              g[1][C::kA + jb] = v.y;
              g[2][C::kA + jb] = v.z;
              g[3][C::kA + jb] = v.w;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < kSfGroup; ++i) ld.next(p.chunks);
      } else {
#pragma unroll
        for (int i = 0; i < kSfGroup; ++i) {
          if (ld.valid()) {
            const int64_t row = (int64_t)ld.ch.x * p.R + ld.mt * p.m_stride + q * 32 + lane;
#pragma unroll
            for (int a = 0; a < C::kA; ++a)
              if (row + a * p.half < p.rows_total)
                g[i][a] = __ldg(reinterpret_cast<const uint32_t*>(
                    p.w_sf + (row + a * p.half) * sf_row + ld.ks * 4));
#pragma unroll
            for (int jb = 0; jb < kNMax / 32; ++jb) {
              const int n = jb * 32 + lane;
              if (n < ld.ch.z)
                g[i][C::kA + jb] = __ldg(reinterpret_cast<const uint32_t*>(
                    p.x_sf + (int64_t)(ld.ch.y + n) * sf_row + ld.ks * 4));
            }
          }
          ld.next(p.chunks);
        }
      }
    };
    load_group(grp[0]);
    load_group(grp[1]);
    bool ok = true;
    uint32_t fill = 0;
    while (ok && stc.valid()) {
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
#pragma unroll
        for (int i = 0; i < kSfGroup; ++i) {
          if (ok && stc.valid()) {
            const int s = (int)(fill % C::kStages);
            const uint32_t use = fill / C::kStages;
            if (!ptx::mbar_wait(&empty[s], (use & 1) ^ 1, deadline(), abort_flag)) {
              if (lane == 0) fail(kStatusTimeout);
              ok = false;
            } else {
              ptx::tc_fence_after();
              const uint32_t tsf = tbase + lane_off + C::kSfBase + s * C::kSfStride;
#pragma unroll
              for (int a = 0; a < C::kA; ++a) ptx::tmem_st_x1(tsf + 4 * a + q, grp[gi][i][a]);
#pragma unroll
              for (int jb = 0; jb < kNMax / 32; ++jb)
                ptx::tmem_st_x1(tsf + C::kSfbCol + jb, grp[gi][i][C::kA + jb]);
              ptx::tmem_st_wait();
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(&full[s]);
              ++fill;
              stc.next(p.chunks);
            }
          }
        }
        if (ok && stc.valid()) load_group(grp[gi]);  // the group two ahead
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int j = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++j) {
      const int4 ch = p.chunks[item / p.m_tiles];
      const int mt = item % p.m_tiles;
      const int b = j % C::kAccBufs;
      const uint32_t u = (uint32_t)(j / C::kAccBufs);
      if (!ptx::mbar_wait(&acc_full[b], u & 1, deadline(), abort_flag)) {
        if (lane == 0) fail(kStatusTimeout);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t acc0 = tbase + lane_off + b * C::kAccCols;
      const int row = mt * p.m_stride + q * 32 + lane;  // output row within the expert
      for (int n0 = 0; n0 < ch.z; n0 += 8) {
        uint32_t v0[8], v1[8];
        ptx::tmem_ld_x8(acc0 + n0, v0);
        ptx::tmem_ld_x8(acc0 + kNMax + n0, v1);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (n0 + t < ch.z) {  // warp-uniform
            const int64_t slot = ch.y + n0 + t;
            if (kGated) {
              const float g = __uint_as_float(v0[t]), up = __uint_as_float(v1[t]);
              const float h = g / (1.0f + expf(-g)) * up;
              const int code = block_scale_code(warp_max(fabsf(h)), 8);
              p.hq[slot * p.out_dim + row] = e4m3_encode_satfinite(h * exp2_exact(127 - code));
              if (lane == 0) p.hs[slot * (p.out_dim / 32) + row / 32] = (uint8_t)code;
            } else {
              p.yp[slot * p.out_dim + row] = __uint_as_float(v0[t]);
              if (row + 128 < p.out_dim) p.yp[slot * p.out_dim + row + 128] = __uint_as_float(v1[t]);
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&acc_empty[b]);
    }
  }

  if (*abort_flag) {  // let copies already in flight land before the CTA exits
    const uint64_t until = ptx::globaltimer() + 2000000ull;
    while (ptx::globaltimer() < until) {
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 2) ptx::tmem_dealloc(tbase, C::kTmemCols);
}

}  // namespace moe
