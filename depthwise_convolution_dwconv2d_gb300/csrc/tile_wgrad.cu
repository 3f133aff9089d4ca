// Small-kernel weight and bias gradients, first pass, on shared-memory tiles.
//
// partial[chunk, oc, a*K + b] = sum over (n, oh, ow) in the chunk of
//     gy[n, off + oc, oh, ow] * x[n, oc/m, oh*S - ph + a*D, ow*S - pw + b*D]
// partial[chunk, oc, K*K]   = sum of gy over the chunk (bias gradient)
// ("Spatial Depthwise Convolution on the GPU #3057", the grad-weight kernel
// extended to padding, stride and dilation, and grad_bias.)
//
// A CTA owns one input channel c (all m of its output channels) and a fixed
// chunk of the batch. It stages x and grad_out tiles in shared memory; each
// thread keeps all K*K (+1) sums for its outputs in registers, walking an
// R x V block of output positions at a time with a register window over the
// x tile rows. At the end the CTA reduces the per-thread sums with a warp
// butterfly and an ordered sum over warps and writes one partial per chunk;
// the second pass (generic.cu) adds the chunks in index order. Every sum has
// a fixed order, so the result is bitwise reproducible.
//
// This file holds shape support and dtype dispatch; the kernels live in
// tile_wgrad_impl.cuh and are compiled once per storage type.
#include "plan.h"
#include "tile_cases.h"
#include "tile_fit.h"

namespace dwconv {
namespace tile {

template <typename T, int MSEL>
cudaError_t wgrad_sel_t(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s);

bool wgrad_supported(const Conv& c) {
  if (!c.planes32()) return false;
  if (c.kh != c.kw || c.sh != c.sw || c.dh != c.dw || c.W > 1024 || c.Wo > 1024) return false;
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  if (wgrad_min_bytes(c.kh, c.sh, c.dh, c.m, c.Wo, es) > 48 * 1024) return false;
#define X(K, S, D, M) if (c.kh == K && c.sh == S && c.dh == D && c.m == M) return true;
  DW_WGRAD_CASES(X)
#undef X
  return false;
}

int64_t wgrad_nb(const Conv& c) {
  // about sixteen units per SM over channels x chunks (so the last wave of
  // units is a small part of the launch), each thread's serial chain
  // (samples x positions / threads) far below 4096 terms
  int64_t chunks = (152 * 16 + c.C - 1) / c.C;
  if (chunks > c.N) chunks = c.N;
  if (chunks < 1) chunks = 1;
  int64_t nb = (c.N + chunks - 1) / chunks;
  // whole planes staged a few samples at a time: make a chunk a whole number
  // of stages (each stage about two items per thread; a block is R x 4
  // outputs, R = 2 at stride 1)
  const int64_t R = c.sh == 1 ? 2 : 1;
  const int64_t items = (c.Ho + R - 1) / R * ((c.Wo + 3) / 4);
  const int64_t spp = (2 * 256 + items - 1) / items;  // samples per stage
  if (spp > 1 && nb % spp != 0) nb = (nb + spp - 1) / spp * spp;
  if (nb > c.N) nb = c.N;
  const int64_t cap = ((int64_t)1 << 20) / (c.Ho * c.Wo > 0 ? c.Ho * c.Wo : 1);
  if (nb > cap) nb = cap > 0 ? cap : 1;
  if (nb < 1) nb = 1;
  if (c.N > 0 && (c.N + nb - 1) / nb > 65535) nb = (c.N + 65534) / 65535;
  return nb;
}

// Chunks of the (sample, band) slices of each channel. From the sample
// count above; when the batch is too small for about sixteen units per SM
// (e.g. 2 samples of 64 channels), whole samples are split further, up to
// one chunk per band the planner can cut a plane into (the kernel spreads
// its actual bands over the chunks; a chunk past the last slice writes a
// zero partial). Depends on the descriptor alone.
int wgrad_chunks(const Conv& c) {
  if (c.N <= 0) return 1;
  const int64_t nb = wgrad_nb(c);
  const int64_t by_samples = (c.N + nb - 1) / nb;
  const int64_t wanted = (152 * 16 + c.C - 1) / c.C;
  if (by_samples >= wanted || nb > 1) return (int)by_samples;
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  int64_t chunks = c.N * wgrad_max_bands(c.kh, c.sh, c.dh, c.m, c.Ho, c.Wo, es);
  if (chunks > wanted) chunks = wanted;
  if (chunks < by_samples) chunks = by_samples;
  if (chunks > 65535) chunks = 65535;
  return (int)chunks;
}

cudaError_t wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  if (c.m == 1) {
    DWCONV_DISPATCH_DTYPE(c.dtype, T, e = (wgrad_sel_t<T, 1>(c, x, gy, ws, chunks, s)));
  } else {
    DWCONV_DISPATCH_DTYPE(c.dtype, T, e = (wgrad_sel_t<T, 2>(c, x, gy, ws, chunks, s)));
  }
  return e;
}

}  // namespace tile
}  // namespace dwconv
