// Measurement helper: a register-only fp32 FMA loop used to read the
// device's FMA rate in the same run as the kernels it is compared with.
#include "common.cuh"

namespace {

__global__ void __launch_bounds__(256) fma_probe_kernel(int iters, float* sink) {
  float a[16];
  const float s = 1.0f + 1e-7f * (threadIdx.x & 7);
  const float t = 1e-7f * (blockIdx.x & 3);
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = (float)(threadIdx.x + i);
  for (int k = 0; k < iters; ++k) {
#pragma unroll
    for (int i = 0; i < 16; ++i) a[i] = fmaf(a[i], s, t);
  }
  float r = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) r += a[i];
  sink[blockIdx.x * 256 + threadIdx.x] = r;
}

}  // namespace

extern "C" dwconv_status_t dwconv_fma_probe(int blocks, int iters, float* sink, cudaStream_t stream) {
  if (blocks < 1 || iters < 1 || !sink) return DWCONV_ERR_INVALID_ARG;
  fma_probe_kernel<<<blocks, 256, 0, stream>>>(iters, sink);
  return cudaGetLastError() == cudaSuccess ? DWCONV_OK : DWCONV_ERR_CUDA;
}
