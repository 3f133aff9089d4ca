// Large-kernel depthwise forward and stride-1 grad-input: shape support and
// dtype dispatch (kernels in large_impl.cuh, compiled once per storage type).
#include "plan.h"

namespace dwconv {
namespace large {

template <typename T>
cudaError_t fwd_t(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s);
template <typename T>
cudaError_t bwd_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s);
template <typename T>
cudaError_t wgrad_t(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s);

bool supported(const Conv& c) {
  if (!c.planes32()) return false;
  // square kernels of the compiled sizes, stride 1, dilation 1, one filter per channel,
  // planes up to 128 x 128
  if (c.kh != c.kw) return false;
  if (c.kh != 7 && c.kh != 9 && c.kh != 11 && c.kh != 13 && c.kh != 15 && c.kh != 21 && c.kh != 27 &&
      c.kh != 31)
    return false;
  if (c.sh != 1 || c.sw != 1 || c.dh != 1 || c.dw != 1 || c.m != 1) return false;
  if (c.ph != c.pw || c.ph > c.kh - 1) return false;
  if (c.H > 128 || c.W > 128 || c.Ho > 128 || c.Wo > 128) return false;
  return true;
}

// The weight gradient stages an x tile and a grad_out plane per stage, two
// stages, plus per-group sums (fp32, whatever the storage type); its planner
// gives up above 220 KB, which large planes with large filters exceed (k = 31
// from about 96 x 96). This is the same arithmetic, on the shape alone.
bool wgrad_supported(const Conv& c) {
  if (!supported(c)) return false;
  const int64_t K = c.kh, R = 4, V = 4, nt = 256;
  auto rup4 = [](int64_t v) { return (v + 3) / 4 * 4; };
  const int64_t gpitch = rup4(c.Wo);
  int64_t xpitch = rup4((K + V - 1) / V * V + gpitch + 4);
  if (xpitch < c.W + c.pw) xpitch = rup4(c.W + c.pw);
  const int64_t stage = rup4((c.Ho + K - 1) * xpitch + c.Ho * gpitch);
  const int64_t items = ((K + R - 1) / R) * ((K + V - 1) / V);
  if (items > nt) return false;
  const int64_t G = items >= nt ? 1 : nt / items;
  return (2 * stage + G * (K * K + 1) + nt / 32) * 4 <= 220 * 1024;
}

cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = fwd_t<T>(c, x, w, b, y, s));
  return e;
}

int wgrad_chunks(const Conv& c) {
  // several units per resident CTA (about 2 per SM), a bounded chain per thread
  int64_t chunks = (152 * 2 * 4 + c.C - 1) / c.C;
  if (chunks > c.N) chunks = c.N;
  if (chunks < 1) chunks = 1;
  const int64_t nb = (c.N + chunks - 1) / chunks;
  return (int)(c.N > 0 ? (c.N + nb - 1) / nb : 1);
}

cudaError_t wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = wgrad_t<T>(c, x, gy, ws, chunks, s));
  return e;
}

cudaError_t bwd_data(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = bwd_t<T>(c, gy, w, gx, acc, s));
  return e;
}

}  // namespace large
}  // namespace dwconv
