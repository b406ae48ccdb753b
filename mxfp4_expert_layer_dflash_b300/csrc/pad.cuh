// Zero-padded copies of row-major byte matrices, for layers whose widths the
// GEMMs cannot take directly.  The GEMM kernels load FP4 weights by TMA in
// rows of 128 elements (the 16U4_ALIGN16B operand form tcgen05's kind::mxf8f6f4
// reads, 128 expanded bytes per swizzled row), so H and I must be multiples of
// 128 there.  A layer with H or I a multiple of 32 only is run on copies whose
// widths are rounded up to 128 with zeros: zero weight codes (scale code 0)
// and zero activations add nothing to any dot product, and whole zero blocks
// of 32 quantise to zero, so the padded layer computes the same y on the
// original rows and columns (every block of 32 has its own scale, so the
// padding never changes a real block's scale).
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {

// dst [groups][dst_rows][dst_row_bytes] from src [groups][src_rows][src_row_bytes]:
// destination row r of a group takes source row s0 + (r - d0) when r is in
// [d0, d0 + n0), s1 + (r - d1) when r is in [d1, d1 + n1), and is zero
// otherwise; the bytes of a row past the source row's length are zero (a
// narrower destination keeps the first dst_row_bytes of each source row).
struct PadSpec {
  const uint8_t* src;
  uint8_t* dst;
  int64_t groups;
  int64_t src_rows, dst_rows;
  int64_t src_row_bytes, dst_row_bytes;  // dst_row_bytes a multiple of 4
  int64_t d0, n0, s0, d1, n1, s1;
};

// one 4-byte word of the destination per thread and step; rows whose length
// is a multiple of 4 are read a word at a time, others byte by byte
__global__ void __launch_bounds__(256) pad_rows_kernel(PadSpec p) {
  grid_dependency_wait();
  const int64_t wpr = p.dst_row_bytes / 4;
  const int64_t words = p.groups * p.dst_rows * wpr;
  const bool word_rows = (p.src_row_bytes & 3) == 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / wpr, c = (i - row * wpr) * 4;
    const int64_t g = row / p.dst_rows, r = row - g * p.dst_rows;
    int64_t s = -1;
    if (r >= p.d0 && r < p.d0 + p.n0) s = p.s0 + (r - p.d0);
    else if (r >= p.d1 && r < p.d1 + p.n1) s = p.s1 + (r - p.d1);
    uint32_t v = 0;
    if (s >= 0 && c < p.src_row_bytes) {
      const uint8_t* sp = p.src + (g * p.src_rows + s) * p.src_row_bytes + c;
      if (word_rows) {
        v = *reinterpret_cast<const uint32_t*>(sp);
      } else {
        for (int b = 0; b < 4 && c + b < p.src_row_bytes; ++b) v |= (uint32_t)sp[b] << (8 * b);
      }
    }
    *reinterpret_cast<uint32_t*>(p.dst + row * p.dst_row_bytes + c) = v;
  }
  grid_launch_dependents();
}

}  // namespace moe
