// Small-kernel depthwise forward and stride-1 grad-input: shape support and
// dtype dispatch. The kernels live in tile_fwd_impl.cuh and are compiled once
// per storage type in tile_fwd_{f32,f16,bf16}.cu.
#include "plan.h"
#include "tile_cases.h"
#include "tile_fit.h"

namespace dwconv {
namespace tile {

template <typename T>
cudaError_t fwd_t(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                  const Epi& ep);
template <typename T>
cudaError_t bwd1_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s);

namespace {
bool square(const Conv& c) {
  return c.kh == c.kw && c.sh == c.sw && c.dh == c.dw;
}
}  // namespace

bool fwd_supported(const Conv& c) {
  if (!c.planes32()) return false;
  if (!square(c) || c.W > 1024 || c.Wo > 1024) return false;
  // the planner's narrowest band must fit its 48 KB limit
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  if (band_min_bytes(c.kh, c.sh, c.dh, c.sh == 1 ? 4 : 2, 4, c.Wo, es, 1) > 48 * 1024) return false;
#define X(K, S, D) if (c.kh == K && c.sh == S && c.dh == D) return true;
  DW_FWD_CASES(X)
#undef X
  return false;
}

cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                const Epi& ep) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = fwd_t<T>(c, x, w, b, y, s, ep));
  return e;
}

bool bwd1_supported(const Conv& c) {
  if (!c.planes32()) return false;
  if (!square(c) || c.sh != 1 || c.m > 4 || c.W > 1024 || c.Wo > 1024) return false;
  if (c.ph > c.dh * (c.kh - 1) || c.pw > c.dw * (c.kw - 1)) return false;
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  if (band_min_bytes(c.kh, 1, c.dh, 4, 4, c.W, es, c.m) > 48 * 1024) return false;
#define X(K, D) if (c.kh == K && c.dh == D) return true;
  DW_BWD1_CASES(X)
#undef X
  return false;
}

cudaError_t bwd1(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = bwd1_t<T>(c, gy, w, gx, acc, s));
  return e;
}

}  // namespace tile
}  // namespace dwconv
