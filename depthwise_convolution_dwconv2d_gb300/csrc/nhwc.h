// Channels-last (NHWC) forward: shape support and entry point (nhwc.cu).
#pragma once

#include "plan.h"

// (K, S) combinations compiled for the tiled channels-last forward.
#define DW_NHWC_CASES(X) X(3, 1) X(3, 2) X(5, 1) X(5, 2) X(7, 1) X(7, 2)

namespace dwconv {
namespace nhwc {

// Shapes the tiled kernel takes: square 3x3 / 5x5 / 7x7, equal strides of 1
// or 2, dilation 1, one filter per channel, C times the element size a
// multiple of 16 bytes (a tensor-map stride rule).
bool tiled_supported(const Conv& c);
// Algo::Nhwc for the tiled kernel, Algo::Generic otherwise.
Algo plan(const Conv& c);
// x [N, H, W, C], y [N, Ho, Wo, ctot] (channels [off, off + C*m) written).
cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                const Epi& ep);

}  // namespace nhwc

// Depthwise-separable block, channels-last (separable.cu).
namespace sep {

// The generic kernel can stage the depthwise result of one pixel (C*m fp32
// values in at most 96 KB of shared memory).
bool supported(const Conv& c);
// Algo::SepTc for the tensor-core kernel, Algo::Generic otherwise.
Algo plan(const Conv& c, int64_t cout);
// x [N, H, W, C]; wd [C*m, kh, kw]; wp [cout, C*m]; y [N, Ho, Wo, ctot]
// (channels [off, off + cout) written).
cudaError_t run(const Conv& c, int64_t cout, int64_t ctot, int64_t off, const void* x, const void* wd,
                const void* s1, const void* h1, int a1, const void* wp, const void* s2, const void* h2, int a2,
                void* y, cudaStream_t s);

}  // namespace sep
}  // namespace dwconv
