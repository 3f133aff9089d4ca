// dwconv2d_bwd_weight_noalloc: the weight/bias gradient for callers that
// cannot hand the library a device workspace.
//
// Some callers have no way to allocate device memory at the point where they
// need the weight gradient: code embedded in a host application that owns
// every device allocation through its own pool and forbids any other
// cudaMalloc, or latency-critical loops where a cudaMalloc -- which may
// synchronise the whole device -- is not acceptable. For them this entry
// point runs exactly the same two-pass computation as dwconv2d_bwd_weight,
// but its partial sums live in one fixed array compiled into the library
// instead of a caller-provided workspace. Nothing is allocated or freed per
// call.
//
// The array below is a file-scope __device__ variable: every GPU on which the
// library's device code is loaded holds these bytes until the process exits.
// In host code its name is only a host-side stand-in, never a device address;
// the real address is looked up once per device with cudaGetSymbolAddress.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB of fp32 partial sums
__device__ __align__(256) float g_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_found[kMaxDevices];
void* g_addr[kMaxDevices];

// Device address of g_scratch on the current device. Only a successful
// lookup is kept: a lookup that fails (for example one attempted while a
// stream is being captured, or with an earlier error still pending) is
// retried on the next call instead of poisoning the device for good.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_found[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
    g_found[dev] = true;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" dwconv_status_t dwconv2d_bwd_weight_noalloc(const dwconv2d_desc_t* desc, const void* x,
                                                       const void* gy, void* gw, void* gbias,
                                                       cudaStream_t stream) {
  // An invalid descriptor (workspace size 0) or a call that asks for nothing
  // gets the regular entry point's answer without touching the array.
  const size_t need = dwconv2d_bwd_weight_workspace_size(desc);
  if (need == 0 || (!gw && !gbias))
    return dwconv2d_bwd_weight(desc, x, gy, gw, gbias, nullptr, 0, stream);
  if (need > kScratchBytes) return DWCONV_ERR_WORKSPACE;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return DWCONV_ERR_CUDA;
  // The first pass writes every partial the second pass reads, so whatever
  // an earlier call left in the array is never used.
  return dwconv2d_bwd_weight(desc, x, gy, gw, gbias, ws, kScratchBytes, stream);
}
