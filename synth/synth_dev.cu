// Device build of the counter-based synthetic input generator (definitions in
// synth_core.h).  Test and benchmark infrastructure: it fills full-size fp32
// expert weights on the GPU, chunk by chunk, so that multi-gigabyte layers need
// no host generation or upload.  Bit-identical to synth_fill_normal_f32 in
// synth.c: integer hashing, exact conversions and the same sequence of fp32
// operations, each rounded to nearest (the _rn intrinsics), then one
// multiply by sigma (__fmul_rn).
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth_core.h"

__global__ void synth_normal_f32_kernel(uint64_t key, uint64_t start, uint64_t n,
                                        float sigma, float* __restrict__ out) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    out[j] = __fmul_rn(sigma, synth_normal(key, start + j));
  }
}

extern "C" int synth_dev_fill_normal_f32(uint64_t seed, uint32_t tensor_id, uint64_t start,
                                         uint64_t n, float sigma, float* dev_out,
                                         cudaStream_t stream) {
  if (n == 0) return 0;
  if (dev_out == nullptr) return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -4;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -4;
  uint64_t blocks = (n + 255) / 256;
  uint64_t cap = (uint64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  synth_normal_f32_kernel<<<(unsigned)blocks, 256, 0, stream>>>(synth_key(seed, tensor_id), start,
                                                                 n, sigma, dev_out);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
