// Measurement and health-check helpers: a register-only fp32 FMA loop used to
// read the device's FMA rate in the same run as the kernels it is compared
// with, and a self-test of the bounded-wait give-up path.
#include "common.cuh"
#include "tma.cuh"

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

// One CTA waits on an mbarrier that expects one arrival which never comes:
// no copy and no tensor-core operation is ever pointed at it, so nothing is
// in flight while the wait runs out. The wait gives up after `polls` polls
// through the same bounded-wait routine the staging pipelines use (which
// counts the give-up in the library's timeout counter); then the barrier is
// completed by the thread that initialised it and invalidated, and the
// kernel returns.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint32_t polls, unsigned int* timeouts) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    dwconv::tma::mbar_init(&bar, 1);
    dwconv::tma::fence_init();
  }
  __syncthreads();
  const bool done = dwconv::tma::mbar_wait_n(&bar, 0, timeouts, polls);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!done) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(dwconv::tma::smem_u32(&bar)) : "memory");
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(dwconv::tma::smem_u32(&bar)) : "memory");
  }
}

}  // namespace

extern "C" dwconv_status_t dwconv_wait_selftest(unsigned int polls, cudaStream_t stream) {
  if (polls < 1 || polls > (1u << 16)) return DWCONV_ERR_INVALID_ARG;
  unsigned int* counter = dwconv::tma::timeout_counter();
  if (!counter) return DWCONV_ERR_CUDA;
  wait_selftest_kernel<<<1, 32, 0, stream>>>(polls, counter);
  return cudaGetLastError() == cudaSuccess ? DWCONV_OK : DWCONV_ERR_CUDA;
}

extern "C" dwconv_status_t dwconv_fma_probe(int blocks, int iters, float* sink, cudaStream_t stream) {
  if (blocks < 1 || iters < 1 || !sink) return DWCONV_ERR_INVALID_ARG;
  fma_probe_kernel<<<blocks, 256, 0, stream>>>(iters, sink);
  return cudaGetLastError() == cudaSuccess ? DWCONV_OK : DWCONV_ERR_CUDA;
}
