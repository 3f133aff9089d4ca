// Large-kernel depthwise family: shape support and dispatch by filter size
// (kernels in large_impl.cuh, one translation unit per odd K from 7 to 31).
#include "large_entries.h"

namespace dwconv {
namespace large {

bool supported(const Conv& c) {
  if (!c.planes32()) return false;
  // square odd kernels 7..31, stride 1, dilation 1, one filter per channel,
  // planes up to 128 x 128
  if (c.kh != c.kw || c.kh < 7 || c.kh > 31 || (c.kh & 1) == 0) return false;
  if (c.sh != 1 || c.sw != 1 || c.dh != 1 || c.dw != 1 || c.m != 1) return false;
  if (c.ph != c.pw || c.ph > c.kh - 1) return false;
  if (c.H > 128 || c.W > 128 || c.Ho > 128 || c.Wo > 128) return false;
  return true;
}

// The weight gradient's planner decides on the shape alone whether its
// stages fit (the scalar kernel: a padded x plane and a grad_out plane per
// stage, two stages, at most 220 KB; the packed kernel cuts the plane into
// bands of output rows until they fit).
bool wgrad_supported(const Conv& c) {
  if (!supported(c)) return false;
#define X(K) \
  if (c.kh == K) return wgrad_fits_k##K(c);
  DW_LARGE_SIZES(X)
#undef X
  return false;
}

cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                const Epi& ep) {
#define X(K) \
  if (c.kh == K) return fwd_k##K(c, x, w, b, y, s, ep);
  DW_LARGE_SIZES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

cudaError_t bwd_data(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
#define X(K) \
  if (c.kh == K) return bwd_k##K(c, gy, w, gx, acc, s);
  DW_LARGE_SIZES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

// Partials per channel of the weight gradient (the planner's "chunks"):
// sample chunks for the scalar kernel, sample chunks x bands of output rows
// for the packed one. Depends on the descriptor alone.
int wgrad_chunks(const Conv& c) {
#define X(K) \
  if (c.kh == K) return wgrad_parts_k##K(c);
  DW_LARGE_SIZES(X)
#undef X
  return 1;
}

// Sample chunks of the scalar weight gradient (also the tensor-core weight
// gradient's chunks): about eight (channel, chunk) units per resident CTA.
int sample_chunks(const Conv& c) {
  int64_t chunks = (152 * 2 * 8 + c.C - 1) / c.C;
  if (chunks > c.N) chunks = c.N;
  if (chunks < 1) chunks = 1;
  const int64_t nb = (c.N + chunks - 1) / chunks;
  return (int)(c.N > 0 ? (c.N + nb - 1) / nb : 1);
}

bool wgrad_scalar_supported(const Conv& c) {
  if (!supported(c)) return false;
#define X(K) \
  if (c.kh == K) return wgrad_scalar_fits_k##K(c);
  DW_LARGE_SIZES(X)
#undef X
  return false;
}

cudaError_t wgrad_scalar(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
#define X(K) \
  if (c.kh == K) return wgrad_scalar_k##K(c, x, gy, ws, chunks, s);
  DW_LARGE_SIZES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

cudaError_t wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
#define X(K) \
  if (c.kh == K) return wgrad_k##K(c, x, gy, ws, chunks, s);
  DW_LARGE_SIZES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace large
}  // namespace dwconv
