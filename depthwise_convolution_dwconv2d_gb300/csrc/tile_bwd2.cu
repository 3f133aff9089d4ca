// Strided (S >= 2) grad-input on shared-memory tiles, by phase.
//
// gx[ih, iw] = sum_j sum_{a,b} w[c*m+j, a, b] gy[(ih + ph - a*D)/S, (iw + pw - b*D)/S]
// over the taps whose numerators are divisible by S (the adjoint of the
// strided forward; the grad-input kernel of "Spatial Depthwise Convolution on
// the GPU #3057"). Splitting ih = S*u + phi, tap a contributes to phase phi
// only when (phi + ph - a*D) % S == 0, and then reads grad_out row
// u + (phi + ph - a*D)/S. With ph % S fixed at compile time every phase's tap
// set and row offset is a constant, so a thread computes the S x S phases of
// an R x V block of (u, v) positions -- an (S*R) x (S*V) block of gx --
// from a register window of grad_out with no per-tap divisibility tests.
//
// This file holds shape support and dtype dispatch; the kernels live in
// tile_bwd2_impl.cuh and are compiled once per storage type.
#include "plan.h"
#include "tile_cases.h"
#include "tile_fit.h"

namespace dwconv {
namespace tile {

template <typename T>
cudaError_t bwd2_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s);

bool bwd2_supported(const Conv& c) {
  if (!c.planes32()) return false;
  if (c.kh != c.kw || c.sh != c.sw || c.dh != c.dw || c.sh < 2 || c.m > 4) return false;
  if (c.W > 1024 || c.Wo > 1024) return false;
  if (c.ph % c.sh != c.pw % c.sh) return false;
  const int pm = c.ph % c.sh;
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  if (bwd2_min_bytes(c.kh, c.sh, c.dh, pm, c.W, es, c.m) > 48 * 1024) return false;
#define X(K, S, D, PM) if (c.kh == K && c.sh == S && c.dh == D && pm == PM) return true;
  DW_BWD2_CASES(X)
#undef X
  return false;
}

cudaError_t bwd2(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = bwd2_t<T>(c, gy, w, gx, acc, s));
  return e;
}

}  // namespace tile
}  // namespace dwconv
