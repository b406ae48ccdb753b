// Grouped expert GEMMs of the bf16-activation mode on tcgen05 (kind::f16):
// the MXFP4 weights are decoded to bf16 ("bf16 after dequant") straight into
// tensor memory, where the MMA reads its A operand, and multiplied with bf16
// activations from shared memory.
//
// Same work decomposition as the MXFP8 GEMMs (swap-AB, one chunk of an
// expert's slots x one pair of 128-row weight tiles per item; GEMM1 pairs gate
// and up rows for the SwiGLU epilogue, GEMM2 pairs rows r and r+128).  Per
// pipeline stage (128 elements of K):
//   producer (warp 0)   TMA of the two packed FP4 tiles (128 rows x 64 bytes,
//                       64-byte swizzle) and of the bf16 activation tile (two
//                       128-byte-swizzled halves of 64 elements)
//   MMA (warp 1)        16 x tcgen05.mma.kind::f16 (K = 16) per stage, A from
//                       TMEM, B from shared memory
//   epilogue (4-7)      silu(gate) * up -> bf16 h (GEMM1) or fp32 rows (GEMM2)
//   decoders (8-23)     one per tile, TMEM lane quarter and half of the stage's
//                       K (lane = weight row): read the row's 32 packed bytes,
//                       decode the 64 values exactly to bf16 and store them into
//                       TMEM with one tcgen05.st (A in TMEM: row m on lane m,
//                       element k at column k/2, even k in the low half —
//                       established by a device probe).  Four decoder warps per
//                       scheduler hide each other's shared-memory and TMEM
//                       latencies; three decoded buffers let decode run ahead of
//                       the MMA.
// Decode: the bits (m << 6) | (sign << 15) of an E2M1 code with magnitude m
// are, read as bf16, exactly e2m1 * 2^-126 (m = 1 lands on the subnormal
// 2^-127 = 0.5 * 2^-126); one bf16 multiply by 2^(c-1) (two, by 2^126 and
// 2^(c-127), when c > 128) applies the block's E8M0 scale exactly.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "fmt.cuh"
#include "ptx.cuh"

namespace moe {

constexpr int kChunkBf16Wide = 64;     // wide chunks of this mode (its TMEM holds 2 x 2 x 64)
constexpr int kBfThreads = 768;        // 24 warps
constexpr int kBfDecoders = 16;        // decoder warps (8..23)
// Per token-chunk width kNMax (32, or 64 for large token counts: fewer
// chunks per expert, so each expert's weights are decoded fewer times).
template <int kNMax>
struct BfCfg {
  static constexpr int kPackedTile = 128 * 64;                  // 128 rows x 128 FP4 (packed)
  static constexpr int kBHalf = kNMax * 128;                    // kNMax rows x 64 bf16
  static constexpr int kStageBytes = 2 * kPackedTile + 2 * kBHalf;
  static constexpr int kStages = (232448 - 1024 - 256) / kStageBytes;
  static constexpr int kAccCols = 2 * kNMax;                    // gate|up (or lo|hi) accumulators
  static constexpr int kDecCol0 = 2 * kAccCols;                 // first TMEM column of decoded A
  static constexpr int kDecCols = 2 * 64;                       // two tiles x 64 columns
  static constexpr int kDecBufs = (512 - kDecCol0) / kDecCols;  // decoded-A buffers: 3 or 2
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + 256;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(kDecBufs >= 2 && kDecCol0 + kDecBufs * kDecCols <= 512, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kNMax % 16 == 0 && kNMax <= 64, "token block");
  static_assert(8 * (2 * kStages + 2 * kDecBufs + 5) + 8 <= 256, "barrier area");
};

struct BfParams {
  CUtensorMap map_w;    // packed FP4 weights [E*R rows, K/2 bytes], u8 box {64, 128}, 64B swizzle
  CUtensorMap map_x;    // bf16 activations [T*k rows, K], box {64, 16}, 128B swizzle
  const uint8_t* w_sf;  // [E*R, K/32]
  const int4* chunks;
  const int32_t* meta;  // meta[0] = chunk count
  uint16_t* hq;         // GEMM1 output h [T*k, I] bf16
  float* yp;            // GEMM2 output [T*k, H] fp32
  int K, R, m_tiles, m_stride, half, out_dim, rows_total;
  int* status;
  unsigned long long timeout_ns;
  int stall_decode;  // debug: decoded buffers are never handed back (the wait runs out)
};

// D[tmem] (+)= A[tmem] x B[smem]^T, bf16, fp32 accumulation; warp-collective
// (one elected lane issues)
__device__ __forceinline__ void mma_bf16_tmem_a_warp(uint32_t d_tmem, uint32_t a_tmem,
                                                     uint64_t b_desc, uint32_t idesc,
                                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// byte permute with the PTX default mode (a selector nibble with bit 3 set
// replicates the sign bit of the chosen byte)
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 64 values of one weight row (two E8M0 blocks), decoded and stored to TMEM.
// Packed byte i holds elements 2i (low nibble) and 2i+1 (high nibble).  For a
// 32-bit word of 8 codes, e / o hold the even / odd codes one per byte; the
// permute puts code 2j in bits 0-3 and code 2j+1 in bits 16-19 with zero bytes
// between, the multiply by 0x1040 copies each code to bits 6-9 and 12-15 (no
// overlap, so no carries), and the mask keeps the magnitude at 6-8 and the
// sign at 15: the bf16 bits of e2m1 * 2^-126.
// kTwoStep: some code of the pair exceeds 128, where 2^(c-1) is not a bf16;
// those blocks multiply by 2^126 and then by 2^(c-127) (exact: the first
// product is the e2m1 value itself).
template <bool kTwoStep>
__device__ __forceinline__ void bf_decode_half(const uint4 (&packed)[2], uint32_t scale_pair,
                                               uint32_t taddr) {
  uint32_t out[32];
#pragma unroll
  for (int j = 0; j < 2; ++j) {  // 32 values per E8M0 block
    const uint32_t c = (scale_pair >> (8 * j)) & 0xFFu;
    const bool one_step = !kTwoStep || c <= 128;  // 2^(c-1) is a normal bf16
    const uint32_t e1 = one_step ? c + 126 : 253;  // 2^(c-1), or 2^126 then 2^(c-127)
    const uint32_t f1 = (e1 << 7) * 0x00010001u;
    const uint32_t f2 = one_step ? 0x3F803F80u : (c << 7) * 0x00010001u;  // 1.0 or 2^(c-127)
    const uint32_t w[4] = {packed[j].x, packed[j].y, packed[j].z, packed[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t e = w[i] & 0x0F0F0F0Fu, o = (w[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t q = prmt(e, o, 0x8080u | (uint32_t)b | ((uint32_t)(4 + b) << 8));
        uint32_t v = bf16x2_mul((q * 0x1040u) & 0x81C081C0u, f1);
        if (kTwoStep) v = bf16x2_mul(v, f2);
        out[j * 16 + i * 4 + b] = v;  // column: elements 2*word, 2*word+1 of the half
      }
    }
  }
  tmem_st_x32(taddr, out);
}

template <int kNMax, bool kGated>
__global__ void __launch_bounds__(kBfThreads, 1) gemm_bf16_kernel(const __grid_constant__ BfParams p) {
  using C = BfCfg<kNMax>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* dec_full = empty + C::kStages;
  uint64_t* dec_empty = dec_full + C::kDecBufs;
  uint64_t* acc_full = dec_empty + C::kDecBufs;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      ptx::mbar_init(&full[s], 1);       // TMA arrive.expect_tx
      ptx::mbar_init(&empty[s], 1 + kBfDecoders);  // MMA commit (B read) + decoders (A read)
    }
    for (int d = 0; d < C::kDecBufs; ++d) {
      ptx::mbar_init(&dec_full[d], kBfDecoders);
      ptx::mbar_init(&dec_empty[d], 1);  // MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&acc_full[b], 1);
      ptx::mbar_init(&acc_empty[b], 4);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 512);
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
  grid_dependency_wait();

  const int n_chunks = p.meta[0];
  const int items = n_chunks * p.m_tiles;
  const int ksteps = p.K / 128;
  auto fail = [&](int code) {
    set_status(p.status, code);
    *abort_flag = 1;
  };
  auto wait_all = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, ptx::mbar_wait_for(bar, parity, p.timeout_ns, abort_flag));
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint64_t pol_w = ptx::policy_evict_first(), pol_x = ptx::policy_evict_last();
    uint32_t fill = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < items; item += gridDim.x) {
      const int4 ch = p.chunks[item / p.m_tiles];
      const int mt = item % p.m_tiles;
      const int nrows = (ch.z + 15) & ~15;
      const int row0 = ch.x * p.R + mt * p.m_stride;
      const uint32_t tx = 2u * C::kPackedTile + 2u * (uint32_t)nrows * 128u;
      for (int ks = 0; ks < ksteps; ++ks, ++fill) {
        const int s = (int)(fill % C::kStages);
        const uint32_t use = fill / C::kStages;
        if (!wait_all(&empty[s], (use & 1) ^ 1)) {
          if (lane == 0) fail(kStatusTimeout);
          ok = false;
          break;
        }
        uint8_t* st = smem + s * C::kStageBytes;
        ptx::mbar_arrive_expect_tx_warp(&full[s], tx);
        ptx::tma_load_2d_warp(st, &p.map_w, &full[s], ks * 64, row0, pol_w);
        ptx::tma_load_2d_warp(st + C::kPackedTile, &p.map_w, &full[s], ks * 64, row0 + p.half,
                              pol_w);
        for (int h = 0; h < 2; ++h)
          for (int r = 0; r < nrows; r += 16)
            ptx::tma_load_2d_warp(st + 2 * C::kPackedTile + h * C::kBHalf + r * 128, &p.map_x,
                                  &full[s], ks * 128 + h * 64, ch.y + r, pol_x);
      }
    }
    grid_launch_dependents();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    uint32_t fill = 0;
    bool ok = true;
    int j = 0;
    for (int item = blockIdx.x; ok && item < items; item += gridDim.x, ++j) {
      const int4 ch = p.chunks[item / p.m_tiles];
      const uint32_t N = (uint32_t)((ch.z + 15) & ~15);
      const uint32_t idesc = ptx::idesc_bf16(N);
      const int b = j & 1;
      const uint32_t u = (uint32_t)(j >> 1);
      if (!wait_all(&acc_empty[b], (u & 1) ^ 1)) {
        if (lane == 0) fail(kStatusTimeout);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t acc = tbase + b * C::kAccCols;
      for (int ks = 0; ks < ksteps; ++ks, ++fill) {
        const int s = (int)(fill % C::kStages);
        const uint32_t use = fill / C::kStages;
        const int d = (int)(fill % C::kDecBufs);
        const uint32_t duse = fill / C::kDecBufs;
        if (!wait_all(&full[s], use & 1) || !wait_all(&dec_full[d], duse & 1)) {
          if (lane == 0) fail(kStatusTimeout);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sb = ptx::smem_u32(smem + s * C::kStageBytes + 2 * C::kPackedTile);
        const uint32_t a0 = tbase + C::kDecCol0 + d * C::kDecCols;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t accum = (ks | kk) ? 1u : 0u;
            mma_bf16_tmem_a_warp(acc + t * kNMax, a0 + t * 64 + kk * 8,
                                 ptx::desc_kmajor_sw128(sb + (kk >> 2) * C::kBHalf + 32 * (kk & 3)),
                                 idesc, accum);
          }
        }
        ptx::mma_commit_warp(&empty[s]);      // the activation tile is read
        if (!p.stall_decode) ptx::mma_commit_warp(&dec_empty[d]);  // the decoded weights are read
      }
      if (!ok) break;
      ptx::mma_commit_warp(&acc_full[b]);
    }
    ptx::mma_commit_warp(drain);
    if (!wait_all(drain, 0) && lane == 0) fail(kStatusTimeout);
  } else if (warp >= 8) {
    // ------------------------------------------------------------ decoders
    const int t = ((warp - 8) >> 2) & 1, q = warp & 3, kh = (warp - 8) >> 3;
    const int r = q * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int sf_row = p.K / 32;
    // this CTA's stages: ksteps per item, items blockIdx.x, + gridDim.x, ...
    const int my_items = blockIdx.x < items ? (items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const uint32_t n_fills = (uint32_t)my_items * (uint32_t)ksteps;
    // scale pairs kRing fills ahead (this row's two E8M0 codes of the stage
    // half); the row pointer is found once per item and then advances 4 bytes
    // a stage
    constexpr int kRing = 4;
    uint32_t sw[kRing];
    int ld_item = blockIdx.x - (int)gridDim.x, ld_left = 0;
    const uint16_t* ld_ptr = nullptr;
    auto load_sw = [&](uint32_t& dst) {
      if (ld_left == 0) {
        ld_item += gridDim.x;
        ld_left = ksteps;
        ld_ptr = nullptr;
        if (ld_item < items) {
          const int4 ch = p.chunks[ld_item / p.m_tiles];
          const int64_t row = (int64_t)ch.x * p.R + (ld_item % p.m_tiles) * p.m_stride +
                              t * p.half + r;
          if (row < p.rows_total)
            ld_ptr = reinterpret_cast<const uint16_t*>(p.w_sf + row * sf_row + kh * 2);
        }
      }
      dst = ld_ptr ? __ldg(ld_ptr) : 0u;
      if (ld_ptr) ld_ptr += 2;
      --ld_left;
    };
#pragma unroll
    for (int i = 0; i < kRing; ++i) load_sw(sw[i]);
    // per-lane constants: the row's two swizzled 16-byte chunks (64B swizzle:
    // chunk c of a 64-byte row sits at c ^ ((r >> 1) & 3)) and its TMEM columns
    const uint32_t off0 = t * C::kPackedTile + r * 64 + (((2 * kh) ^ ((r >> 1) & 3)) << 4);
    const uint32_t off1 = t * C::kPackedTile + r * 64 + (((2 * kh + 1) ^ ((r >> 1) & 3)) << 4);
    const uint32_t tcol0 = tbase + lane_off + C::kDecCol0 + t * 64 + kh * 32;
    int s = 0, d = 0;
    uint32_t full_par = 0, dec_par = 1;
    for (uint32_t fill = 0; fill < n_fills;) {
#pragma unroll
      for (int i = 0; i < kRing; ++i, ++fill) {
        if (fill < n_fills) {
          if (!wait_all(&full[s], full_par) || !wait_all(&dec_empty[d], dec_par)) {
            if (lane == 0) fail(kStatusTimeout);
            fill = n_fills;
            break;
          }
          ptx::tc_fence_after();
          const uint8_t* st = smem + s * C::kStageBytes;
          uint4 pk[2];
          pk[0] = *reinterpret_cast<const uint4*>(st + off0);
          pk[1] = *reinterpret_cast<const uint4*>(st + off1);
          const uint32_t taddr = tcol0 + d * C::kDecCols;
          if (__all_sync(0xffffffffu, (sw[i] & 0xFFu) <= 128u && (sw[i] >> 8) <= 128u))
            bf_decode_half<false>(pk, sw[i], taddr);
          else
            bf_decode_half<true>(pk, sw[i], taddr);
          ptx::tmem_st_wait();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            ptx::mbar_arrive(&dec_full[d]);
            ptx::mbar_arrive(&empty[s]);
          }
          load_sw(sw[i]);
          if (++s == C::kStages) {
            s = 0;
            full_par ^= 1;
          }
          if (++d == C::kDecBufs) {
            d = 0;
            dec_par ^= 1;
          }
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    int j = 0;
    for (int item = blockIdx.x; item < items; item += gridDim.x, ++j) {
      const int4 ch = p.chunks[item / p.m_tiles];
      const int mt = item % p.m_tiles;
      const int b = j & 1;
      const uint32_t u = (uint32_t)(j >> 1);
      if (!wait_all(&acc_full[b], u & 1)) {
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
        for (int tt = 0; tt < 8; ++tt) {
          if (n0 + tt < ch.z) {
            const int64_t slot = ch.y + n0 + tt;
            if (kGated) {
              const float g = __uint_as_float(v0[tt]), up = __uint_as_float(v1[tt]);
              p.hq[slot * p.out_dim + row] = float_to_bf16_bits(g / (1.0f + expf(-g)) * up);
            } else {
              p.yp[slot * p.out_dim + row] = __uint_as_float(v0[tt]);
              if (row + 128 < p.out_dim) p.yp[slot * p.out_dim + row + 128] = __uint_as_float(v1[tt]);
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
  if (warp == 1) ptx::tmem_dealloc(tbase, 512);
}

}  // namespace moe
