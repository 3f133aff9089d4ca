// Entry points of the large-kernel family, one set per odd filter size K
// from 7 to 31 (defined in large_kNN.cu, dispatched by large.cu).
#pragma once

#include "plan.h"

namespace dwconv {
namespace large {

#define DW_LARGE_SIZES(X) X(7) X(9) X(11) X(13) X(15) X(17) X(19) X(21) X(23) X(25) X(27) X(29) X(31)

#define DW_LARGE_DECLARE(K)                                                                                  \
  cudaError_t fwd_k##K(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,   \
                       const Epi& ep);                                                                      \
  cudaError_t bwd_k##K(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s);   \
  cudaError_t wgrad_k##K(const Conv& c, const void* x, const void* gy, float* ws, int parts,               \
                         cudaStream_t s);                                                                   \
  int wgrad_parts_k##K(const Conv& c);                                                                      \
  bool wgrad_fits_k##K(const Conv& c);                                                                      \
  cudaError_t wgrad_scalar_k##K(const Conv& c, const void* x, const void* gy, float* ws, int chunks,       \
                                cudaStream_t s);                                                            \
  bool wgrad_scalar_fits_k##K(const Conv& c);
DW_LARGE_SIZES(DW_LARGE_DECLARE)
#undef DW_LARGE_DECLARE

}  // namespace large
}  // namespace dwconv
