// Dense split-K GEMM on tcgen05 for decode-sized token counts:
//   part[ks][t][m] = sum over the ks-th range of K of A[m, k] * B[t, k]
// A = weights [M, K] (one 128-row tile per work item), B = activations [T, K].
//
// It serves the steps beside the expert layer whose output dimension is too
// small to give every SM a weight tile of its own: the router (E logits per
// token; expert routing is part of the pipeline the runtime is built around:
// techllm.github.io, "Xiaomi MiMo and TileRT ...", section "3. TileRT") and a
// dense projection kept at FP8 (the same page, section "1. MXFP4 — MoE에만
// 걸린 양자화").  K is split across work items and the fp32 partials are
// summed afterwards in a fixed order, so results are deterministic.
//
// Work item = (128-row weight tile, block of up to kNMax tokens, K range).
// Instantiations:
//   kDenseBf16  kind::f16, bf16 A and B (the router, x W_r^T), kNMax = 256
//   kDenseMxf8  kind::mxf8f6f4 block_scale, E4M3 A and B with E8M0 scales per
//               32 elements (a dense MXFP8 projection), kNMax = 128; the scales
//               are staged in TMEM exactly as in the expert GEMMs
// Warp roles as in the expert GEMMs: warp 0 TMA producer and warp 2 MMA
// issuer (convergent warps, one elected lane issues), warps 4-7 scale stagers
// (MXFP8 only), warps 8-11 epilogue (TMEM -> fp32 partials).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "fmt.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kDenseBf16 = 0, kDenseMxf8 = 1;
constexpr int kDenseThreads = 384;
constexpr int kDenseBoxRowsB = 64;  // largest activation TMA box (token rows)
constexpr int kDenseMaxSplits = 64;

struct DenseParams {
  CUtensorMap map_a;    // weights [M, K]: bf16 box {64, 128} or u8 box {128, 128}, SW128
  CUtensorMap map_b;    // activations [T, K]: bf16 box {64, box_rows_b} or u8 box
                        // {128, box_rows_b}, SW128
  const uint8_t* a_sf;  // [M, K/32] E8M0 (MXFP8 kind)
  const uint8_t* b_sf;  // [T, K/32] E8M0 (MXFP8 kind)
  float* part;          // [k_splits][T][M] fp32 partial sums
  int M, T;
  int m_tiles, n_blocks, k_splits;
  int kb_per_split, kb_total;  // stages (128-byte K blocks) per item and in all of K
  int box_rows_b;              // token rows per activation TMA box (16, 32 or 64)
  int* status;
  unsigned long long timeout_ns;
};

template <int kKind, int kNMax>
struct DenseCfg {
  static constexpr int kATile = 128 * 128;  // 128 rows x 128 bytes of K
  static constexpr int kBTile = kNMax * 128;
  static constexpr int kStageBytes = kATile + kBTile;
  static constexpr int kStages = (232448 - 1024 - 256) / kStageBytes;
  static constexpr int kSfStride = kKind == kDenseMxf8 ? 16 : 0;  // TMEM scale columns / stage
  static constexpr int kAccBufs = 2 * kNMax + kStages * kSfStride <= 512 ? 2 : 1;
  static constexpr int kSfBase = kAccBufs * kNMax;  // TMEM column of stage 0's scales
  static constexpr int kSfbCol = 4;                 // B scales after the 4 A scale columns
  static constexpr int kTmemCols = 512;
  static constexpr int kElemsPerBlock = kKind == kDenseBf16 ? 64 : 128;  // K elements / stage
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + 256;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kNMax % 16 == 0 && kNMax <= 256, "token block");
  // (activation boxes of 16, 32 or 64 rows: a launch with kNMax < 64 only
  // takes token counts whose box fits, T <= kNMax)
  static_assert(kKind == kDenseBf16 || kSfbCol + kNMax / 32 <= kSfStride, "B scale columns");
  static_assert(kSfBase + kStages * kSfStride <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

// position of one work item
struct DenseItem {
  int mt, nb, ks, kb0, kb1, tok0, nvalid;
  __device__ __forceinline__ void decode(const DenseParams& p, int item, int n_max) {
    ks = item % p.k_splits;
    const int rest = item / p.k_splits;
    nb = rest % p.n_blocks;
    mt = rest / p.n_blocks;
    kb0 = ks * p.kb_per_split;
    kb1 = min(kb0 + p.kb_per_split, p.kb_total);
    tok0 = nb * n_max;
    nvalid = min(n_max, p.T - tok0);
  }
};

template <int kKind, int kNMax>
__global__ void __launch_bounds__(kDenseThreads, 1)
    dense_tc_kernel(const __grid_constant__ DenseParams p) {
  using C = DenseCfg<kKind, kNMax>;
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
      // TMA arrive.expect_tx (+ one arrival per scale warp in the MXFP8 kind)
      ptx::mbar_init(&full[s], 1 + (kKind == kDenseMxf8 ? 4 : 0));
      ptx::mbar_init(&empty[s], 1);  // MMA commit
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
    ptx::prefetch_tmap(&p.map_a);
    ptx::prefetch_tmap(&p.map_b);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // the activations (and their scales) come from the preceding kernel
  grid_dependency_wait();

  const int items = p.m_tiles * p.n_blocks * p.k_splits;
  auto fail = [&](int code) {
    set_status(p.status, code);
    *abort_flag = 1;
  };
  auto deadline = [&]() { return ptx::globaltimer() + p.timeout_ns; };
  // bounded wait whose outcome is the same in every lane of the warp
  auto wait_all = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, deadline(), abort_flag));
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_a = ptx::policy_evict_first(), pol_b = ptx::policy_evict_last();
    uint32_t fill = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < items; item += gridDim.x) {
      DenseItem it;
      it.decode(p, item, kNMax);
      const int nrows = (it.nvalid + 15) & ~15;
      const int nboxes = (nrows + p.box_rows_b - 1) / p.box_rows_b;
      const uint32_t tx = (uint32_t)C::kATile + (uint32_t)nboxes * p.box_rows_b * 128;
      for (int kb = it.kb0; kb < it.kb1; ++kb, ++fill) {
        const int s = (int)(fill % C::kStages);
        const uint32_t use = fill / C::kStages;
        if (!wait_all(&empty[s], (use & 1) ^ 1)) {
          if (lane == 0) fail(kStatusTimeout);
          ok = false;
          break;
        }
        uint8_t* st = smem + s * C::kStageBytes;
        const int x = kb * C::kElemsPerBlock;
        ptx::mbar_arrive_expect_tx_warp(&full[s], tx);
        ptx::tma_load_2d_warp(st, &p.map_a, &full[s], x, it.mt * 128, pol_a);
        for (int b = 0; b < nboxes; ++b)
          ptx::tma_load_2d_warp(st + C::kATile + b * p.box_rows_b * 128, &p.map_b, &full[s],
                                x, it.tok0 + b * p.box_rows_b, pol_b);
      }
    }
    grid_launch_dependents();
  } else if (warp == 2) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t fill = 0;
    bool ok = true;
    int j = 0;
    for (int item = blockIdx.x; ok && item < items; item += gridDim.x, ++j) {
      DenseItem it;
      it.decode(p, item, kNMax);
      const uint32_t N = (uint32_t)((it.nvalid + 15) & ~15);
      const int b = j % C::kAccBufs;
      const uint32_t u = (uint32_t)(j / C::kAccBufs);
      if (!wait_all(&acc_empty[b], (u & 1) ^ 1)) {
        if (lane == 0) fail(kStatusTimeout);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t acc = tbase + b * kNMax;
      for (int kb = it.kb0; kb < it.kb1; ++kb, ++fill) {
        const int s = (int)(fill % C::kStages);
        const uint32_t use = fill / C::kStages;
        if (!wait_all(&full[s], use & 1)) {
          if (lane == 0) fail(kStatusTimeout);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(smem + s * C::kStageBytes), sb = sa + C::kATile;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t accum = (kb > it.kb0 || kk > 0) ? 1u : 0u;
          if (kKind == kDenseBf16) {
            ptx::mma_bf16_warp(acc, ptx::desc_kmajor_sw128(sa + 32 * kk),
                               ptx::desc_kmajor_sw128(sb + 32 * kk), ptx::idesc_bf16(N), accum);
          } else {
            const uint32_t tsf = tbase + C::kSfBase + s * C::kSfStride;
            ptx::mma_mxf8f6f4_warp(acc, ptx::desc_kmajor_sw128(sa + 32 * kk),
                                   ptx::desc_kmajor_sw128(sb + 32 * kk),
                                   ptx::idesc_mxf8f6f4(N, kk, kk, ptx::kFmtE4M3), tsf,
                                   tsf + C::kSfbCol, accum);
          }
        }
        ptx::mma_commit_warp(&empty[s]);  // frees the smem stage (and its scale columns)
      }
      if (!ok) break;
      ptx::mma_commit_warp(&acc_full[b]);
    }
    ptx::mma_commit_warp(drain);
    if (!wait_all(drain, 0) && lane == 0) fail(kStatusTimeout);
  } else if (kKind == kDenseMxf8 && warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ scale stagers
    // Warp q (= warp % 4) owns TMEM lanes 32q..32q+31: the A scale word of
    // weight row mt*128 + 32q + lane goes to column q, the B scale word of token
    // tok0 + 32jb + lane to column kSfbCol + jb (every quarter holds all B
    // words).  Words are loaded kRing fills ahead of the fill being staged;
    // the weight scales come from HBM and the distance covers its latency.
    constexpr int kRing = 8;
    constexpr int kWb = kNMax / 32;
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int sf_row = p.kb_total * 4;  // bytes of scales per row (K / 32)
    struct Pos {
      int item, kb;
      DenseItem it;
    };
    auto start = [&](Pos& c) {
      c.item = blockIdx.x;
      if (c.item < items) {
        c.it.decode(p, c.item, kNMax);
        c.kb = c.it.kb0;
      }
    };
    auto advance = [&](Pos& c) {
      if (++c.kb == c.it.kb1) {
        c.item += gridDim.x;
        if (c.item < items) {
          c.it.decode(p, c.item, kNMax);
          c.kb = c.it.kb0;
        }
      }
    };
    uint32_t wa[kRing], wb[kRing][kWb];
    auto load = [&](const Pos& c, uint32_t& a, uint32_t (&bw)[kWb]) {
      const int row = c.it.mt * 128 + q * 32 + lane;
      a = row < p.M ? __ldg(reinterpret_cast<const uint32_t*>(p.a_sf + (int64_t)row * sf_row +
                                                              c.kb * 4))
                    : 0u;
#pragma unroll
      for (int jb = 0; jb < kWb; ++jb) {
        const int n = jb * 32 + lane;
        bw[jb] = n < c.it.nvalid
                     ? __ldg(reinterpret_cast<const uint32_t*>(
                           p.b_sf + (int64_t)(c.it.tok0 + n) * sf_row + c.kb * 4))
                     : 0u;
      }
    };
    Pos ld, stg;
    start(ld);
    stg = ld;
#pragma unroll
    for (int r = 0; r < kRing; ++r) {
      if (ld.item < items) {
        load(ld, wa[r], wb[r]);
        advance(ld);
      }
    }
    uint32_t fill = 0;
    bool ok = true;
    while (ok && stg.item < items) {
#pragma unroll
      for (int r = 0; r < kRing; ++r) {
        if (ok && stg.item < items) {
          const int s = (int)(fill % C::kStages);
          const uint32_t use = fill / C::kStages;
          if (!wait_all(&empty[s], (use & 1) ^ 1)) {
            if (lane == 0) fail(kStatusTimeout);
            ok = false;
          } else {
            ptx::tc_fence_after();
            const uint32_t tsf = tbase + lane_off + C::kSfBase + s * C::kSfStride;
            ptx::tmem_st_x1(tsf + q, wa[r]);
#pragma unroll
            for (int jb = 0; jb < kWb; ++jb) ptx::tmem_st_x1(tsf + C::kSfbCol + jb, wb[r][jb]);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&full[s]);
            ++fill;
            advance(stg);
            if (ld.item < items) {
              load(ld, wa[r], wb[r]);
              advance(ld);
            }
          }
        }
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int j = 0;
    for (int item = blockIdx.x; item < items; item += gridDim.x, ++j) {
      DenseItem it;
      it.decode(p, item, kNMax);
      const int b = j % C::kAccBufs;
      const uint32_t u = (uint32_t)(j / C::kAccBufs);
      if (!wait_all(&acc_full[b], u & 1)) {
        if (lane == 0) fail(kStatusTimeout);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t acc = tbase + lane_off + b * kNMax;
      const int row = it.mt * 128 + q * 32 + lane;
      float* dst = p.part + ((int64_t)it.ks * p.T + it.tok0) * p.M + row;
      // 32 tokens (accumulator columns) per wait: four loads in flight (the
      // columns past the block exist and are not stored)
      for (int n0 = 0; n0 < it.nvalid; n0 += 32) {
        uint32_t v[4][8];
#pragma unroll
        for (int g = 0; g < 4; ++g)
          if (n0 + 8 * g < kNMax) ptx::tmem_ld_x8(acc + n0 + 8 * g, v[g]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int t = 0; t < 8; ++t)
            if (n0 + 8 * g + t < it.nvalid && row < p.M)
              dst[(int64_t)(n0 + 8 * g + t) * p.M] = __uint_as_float(v[g][t]);
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

// y[t, m] = bf16_RNE( sum over ks = 0..k_splits-1 of part[ks][t][m] ), fixed
// order; four outputs per thread (M % 4 == 0)
__global__ void __launch_bounds__(256) splitk_reduce_bf16_kernel(const float* __restrict__ part,
                                                                 int k_splits, int T, int M,
                                                                 uint16_t* __restrict__ y) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int64_t total = (int64_t)T * M / 4;
  const int64_t stride = (int64_t)T * M;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 a = reinterpret_cast<const float4*>(part)[i];
    for (int ks = 1; ks < k_splits; ++ks) {
      const float4 b = reinterpret_cast<const float4*>(part + ks * stride)[i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    const uint32_t lo = (uint32_t)float_to_bf16_bits(a.x) | ((uint32_t)float_to_bf16_bits(a.y) << 16);
    const uint32_t hi = (uint32_t)float_to_bf16_bits(a.z) | ((uint32_t)float_to_bf16_bits(a.w) << 16);
    reinterpret_cast<uint2*>(y)[i] = make_uint2(lo, hi);
  }
}

}  // namespace moe
