// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05), MXFP8 mode.
//
// Swap-AB: the expert's weight rows fill the 128-row MMA dimension (A) and the
// expert's tokens (a chunk of at most kChunkMax slots, padded to 16) are N, so
// the tiny decode-time token count never pads the weight side.  A is FP4
// (E2M1) straight from HBM: TMA's 16U4_ALIGN16B mode expands each 16-element
// group into the 16-byte-aligned form the MMA reads, so no thread touches the
// weights.  B is the MXFP8-E4M3 activation tile.  Both E8M0 scale sets go
// to TMEM through tcgen05.cp and the MMA applies them per 32 elements
// (kind::mxf8f6f4, block_scale).  Decode is bound by weight bandwidth
// (ai.appwright.xyz, "第1層"); the pipeline keeps several weight tiles in
// flight per SM while the tensor cores work on the previous ones (the
// load/compute overlap of dothoosh.com, "TileRT", done here per kernel).
//
// Warp roles (256 threads, one CTA per SM, persistent over work items):
//   warp 0     TMA producer (weights + activations), one lane
//   warp 1     scale producer: cp.async of the E8M0 words into the layout
//              tcgen05.cp expects, generic->async proxy fence, mbarrier arrive
//   warp 2     TMEM owner and MMA issuer, one lane
//   warps 4-7  epilogue: TMEM -> registers -> SwiGLU + MXFP8 requant (GEMM1)
//              or fp32 rows of yp (GEMM2); warp w reads TMEM lanes 32*(w%4)..
// Work item = (chunk of one expert's slots, 128-row tile of the output).
// GEMM1 tiles pair gate rows [r, r+128) with up rows [I+r, I+r+128), so the
// epilogue has both operands of silu(gate)*up for the same (row, token).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "fmt.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kTcThreads = 256;
constexpr int kBlockK = 128;  // K elements per stage: one TMA box of FP4
constexpr int kBoxRowsB = 16; // activation rows per TMA box
constexpr int kNMax = kChunkMax;
constexpr int kSfLag = 2;     // stages the scale producer runs ahead of its arrivals

struct TcParams {
  CUtensorMap map_w;  // FP4 weights [E*R rows, K], 16U4_ALIGN16B, box {128, 128}, SW128
  CUtensorMap map_x;  // E4M3 activations [T*k rows, K], u8, box {128, 16}, SW128
  const uint8_t* w_sf;  // [E*R, K/32]
  const uint8_t* x_sf;  // [T*k, K/32]
  const int4* chunks;
  const int32_t* meta;
  uint8_t* hq;  // GEMM1 out: [T*k, I] E4M3
  uint8_t* hs;  // GEMM1 out: [T*k, I/32]
  float* yp;    // GEMM2 out: [T*k, H]
  int K;        // reduction length
  int R;        // weight rows per expert (2I or H)
  int m_tiles;  // 128-row output tiles per expert (I/128 or H/128)
  int half;     // GEMM1: row offset of the up half (I)
  int out_dim;  // row length of the output (I or H)
  int* status;
  unsigned long long timeout_ns;
};

template <bool kGated>
struct TcCfg {
  static constexpr int kA = kGated ? 2 : 1;           // A tiles per stage
  static constexpr int kATile = 128 * 128;            // unpacked FP4 tile bytes
  static constexpr int kBTile = kNMax * 128;
  static constexpr int kSf = 512;                     // one scale set: 32 rows x 16 B
  static constexpr int kStageBytes = ((kA * kATile + kBTile + (kA + 1) * kSf) + 1023) / 1024 * 1024;
  static constexpr int kStages = kGated ? 5 : 8;
  static constexpr int kAccCols = kA * kNMax;         // one accumulator buffer
  static constexpr int kSfBase = 2 * kAccCols;        // TMEM column of stage 0's scales
  static constexpr int kSfStride = 16;                // TMEM columns per stage of scales
  static constexpr int kTmemCols = kGated ? 512 : 256;
  static constexpr uint32_t kTxA = 128 * 64;          // packed bytes of one weight box
  static constexpr int kBarBytes = 256;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kBarBytes;
  static_assert(kSfBase + kStages * kSfStride <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool kGated>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<kGated>;
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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1 + 32);  // TMA arrive.expect_tx + 32 scale-producer lanes
      ptx::mbar_init(&empty[s], 1);      // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&acc_full[b], 1);   // MMA commit
      ptx::mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
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
      uint32_t fill = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
        const int4 ch = p.chunks[item / p.m_tiles];
        const int mt = item % p.m_tiles;
        const int nrows = (ch.z + 15) & ~15;
        const int row0 = ch.x * p.R + mt * 128;
        const uint32_t tx = C::kA * C::kTxA + (uint32_t)(nrows / kBoxRowsB) * (kBoxRowsB * 128);
        for (int ks = 0; ks < ksteps; ++ks, ++fill) {
          const int s = (int)(fill % C::kStages);
          const uint32_t use = fill / C::kStages;
          if (!ptx::mbar_wait(&empty[s], (use & 1) ^ 1, deadline(), abort_flag)) {
            fail(kStatusTimeout);
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::kStageBytes;
          ptx::mbar_arrive_expect_tx(&full[s], tx);
          ptx::tma_load_2d(st, &p.map_w, &full[s], ks * kBlockK, row0, pol_w);
          if (kGated)
            ptx::tma_load_2d(st + C::kATile, &p.map_w, &full[s], ks * kBlockK, row0 + p.half,
                             pol_w);
          for (int r = 0; r < nrows; r += kBoxRowsB)
            ptx::tma_load_2d(st + C::kA * C::kATile + r * 128, &p.map_x, &full[s], ks * kBlockK,
                             ch.y + r, pol_x);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ scale producer
    // Stage layout of one scale set: 32 rows x 16 B; row L, word q holds the
    // four E8M0 bytes (one per 32-element block of this stage) of operand row
    // 32q + L.  tcgen05.cp 32x128b.warpx4 then puts operand row m at TMEM lane m
    // of column m/32, which is where the block-scaled MMA reads it.
    uint32_t fill = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const int4 ch = p.chunks[item / p.m_tiles];
      const int mt = item % p.m_tiles;
      const int row0 = ch.x * p.R + mt * 128;
      for (int ks = 0; ks < ksteps; ++ks, ++fill) {
        const int s = (int)(fill % C::kStages);
        const uint32_t use = fill / C::kStages;
        if (!ptx::mbar_wait(&empty[s], (use & 1) ^ 1, deadline(), abort_flag)) {
          if (lane == 0) fail(kStatusTimeout);
          ok = false;
          break;
        }
        uint8_t* sf = smem + s * C::kStageBytes + C::kA * C::kATile + C::kBTile;
#pragma unroll
        for (int a = 0; a < C::kA; ++a) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int64_t row = (int64_t)row0 + a * p.half + q * 32 + lane;
            ptx::cp_async_4(sf + a * C::kSf + lane * 16 + q * 4,
                            p.w_sf + row * sf_row + ks * 4, 4);
          }
        }
        uint8_t* sfb = sf + C::kA * C::kSf;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int n = q * 32 + lane;
          const bool valid = n < ch.z;
          const uint8_t* src = valid ? p.x_sf + (int64_t)(ch.y + n) * sf_row + ks * 4 : p.x_sf;
          ptx::cp_async_4(sfb + lane * 16 + q * 4, src, valid ? 4u : 0u);
        }
        cp_async_commit();
        if (fill >= (uint32_t)kSfLag) {
          cp_async_wait_group<kSfLag>();
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive(&full[(fill - kSfLag) % C::kStages]);
        }
      }
    }
    cp_async_wait_group<0>();
    ptx::fence_proxy_async_smem();
    if (ok) {
      const uint32_t first = fill > (uint32_t)kSfLag ? fill - kSfLag : 0;
      for (uint32_t f = first; f < fill; ++f) ptx::mbar_arrive(&full[f % C::kStages]);
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
        const int b = j & 1;
        const uint32_t u = (uint32_t)(j >> 1);
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
          const uint32_t ssf = sb + C::kBTile;
          const uint32_t tsf = tbase + C::kSfBase + s * C::kSfStride;
#pragma unroll
          for (int a = 0; a <= C::kA; ++a)
            ptx::tmem_cp_32x128b_warpx4(tsf + 4 * a, ptx::smem_desc(ssf + a * C::kSf, 0, 128, 0));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t idesc = ptx::idesc_mxf8f6f4(N, kk, kk);
            const uint32_t accum = (ks | kk) ? 1u : 0u;
            ptx::mma_mxf8f6f4(acc0, ptx::desc_kmajor_sw128(sa0 + 32 * kk),
                              ptx::desc_kmajor_sw128(sb + 32 * kk), idesc, tsf, tsf + 4 * C::kA,
                              accum);
            if (kGated)
              ptx::mma_mxf8f6f4(acc1, ptx::desc_kmajor_sw128(sa1 + 32 * kk),
                                ptx::desc_kmajor_sw128(sb + 32 * kk), idesc, tsf + 4,
                                tsf + 4 * C::kA, accum);
          }
          ptx::mma_commit(&empty[s]);  // frees the smem stage once these MMAs finish
        }
        if (!ok) break;
        ptx::mma_commit(&acc_full[b]);
      }
      ptx::mma_commit(drain);
      if (!ptx::mbar_wait(drain, 0, deadline(), abort_flag)) fail(kStatusTimeout);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int j = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++j) {
      const int4 ch = p.chunks[item / p.m_tiles];
      const int mt = item % p.m_tiles;
      const int b = j & 1;
      const uint32_t u = (uint32_t)(j >> 1);
      if (!ptx::mbar_wait(&acc_full[b], u & 1, deadline(), abort_flag)) {
        if (lane == 0) fail(kStatusTimeout);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t acc0 = tbase + lane_off + b * C::kAccCols;
      const int row = mt * 128 + q * 32 + lane;  // output row within the expert
      for (int n0 = 0; n0 < ch.z; n0 += 8) {
        uint32_t v0[8], v1[8];
        ptx::tmem_ld_x8(acc0 + n0, v0);
        if (kGated) ptx::tmem_ld_x8(acc0 + kNMax + n0, v1);
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
