// Kernel-family planner and dispatch (internal to libdwconv).
#pragma once

#include "common.cuh"

namespace dwconv {

constexpr int kMaxBranches = 8;

enum class Algo {
  Generic = 0,   // generic.cu: any shape
  Tile = 1,      // tile_fwd.cu / tile_bwd.cu: register-blocked smem tiles, small kernels
  Large = 2,     // large.cu: large-kernel direct convolution
  IBGemm = 3,    // ibgemm.cu: large-kernel implicit batched GEMM on tcgen05 (fp16 / bf16)
  Plane = 4,     // plane.cu: 3x3 on small planes, one warp per group of whole planes
  TcWgrad = 5,   // wgrad_tc.cu: large-kernel weight gradient on tcgen05 (fp16 / bf16)
  Nhwc = 6,      // nhwc.cu: channels-last forward, TMA-staged channel-vector tiles
  SepTc = 7,     // separable.cu: depthwise + pointwise block, pointwise on tcgen05 (fp16 / bf16)
};

struct WPlan {
  Algo algo;
  int chunks;    // batch chunks of the first bwd_weight pass
};

const char* algo_name(Algo a);
Algo plan_fwd(const Conv& c, bool epilogue = false);
Algo plan_bwd_data(const Conv& c);
WPlan plan_bwd_weight(const Conv& c);

cudaError_t run_fwd(Algo a, const Conv& c, const void* x, const void* w, const void* b, void* y,
                    cudaStream_t s, const Epi& ep = Epi{});
cudaError_t run_bwd_data(Algo a, const Conv& c, const void* gy, const void* w, void* gx,
                         bool accumulate, cudaStream_t s);
cudaError_t run_bwd_weight(const WPlan& p, const Conv& c, const void* x, const void* gy, void* gw,
                           void* gb, float* ws, cudaStream_t s);
cudaError_t run_fwd_multi(int nb, const Conv* cs, const void* x, const void* const* w,
                          const void* const* bias, void* y, cudaStream_t s);
cudaError_t run_bwd_data_multi(int nb, const Conv* cs, const void* gy, const void* const* w,
                               void* gx, cudaStream_t s);

namespace tile {
// tile_fwd.cu
bool fwd_supported(const Conv& c);
cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                const Epi& ep = Epi{});
bool bwd1_supported(const Conv& c);
cudaError_t bwd1(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s);
// tile_bwd2.cu
bool bwd2_supported(const Conv& c);
cudaError_t bwd2(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s);
// tile_wgrad.cu (first pass; the second pass is bwd_weight_pass2)
bool wgrad_supported(const Conv& c);
int wgrad_chunks(const Conv& c);
int64_t wgrad_nb(const Conv& c);  // samples per chunk (chunks = ceil(N / wgrad_nb))
cudaError_t wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s);
// tile_multi.cu
bool multi_supported(int nb, const Conv* cs);
cudaError_t fwd_multi(int nb, const Conv* cs, const void* x, const void* const* w,
                      const void* const* bias, void* y, cudaStream_t s);
cudaError_t bwd_multi(int nb, const Conv* cs, const void* gy, const void* const* w, void* gx,
                      cudaStream_t s);
}  // namespace tile

Algo plan_multi(int nb, const Conv* cs);

namespace large {
// large.cu: large-kernel direct convolution (fp32 FMA), stride 1
bool supported(const Conv& c);
bool wgrad_supported(const Conv& c);  // supported() and the weight-gradient stages fit shared memory
cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                const Epi& ep = Epi{});
cudaError_t bwd_data(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s);
int wgrad_chunks(const Conv& c);  // partials per channel of wgrad()
cudaError_t wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s);
// the scalar weight gradient over sample chunks, for any K (fallback of the
// tensor-core weight gradient, which uses the same chunks)
int sample_chunks(const Conv& c);
bool wgrad_scalar_supported(const Conv& c);
cudaError_t wgrad_scalar(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s);
}  // namespace large

namespace plane {
// plane.cu: 3x3 on small planes (fwd: rows of 9..16; grad-input: stride 1 and rows
// of 9..16; weight gradient: output rows of at most 16)
bool fwd_supported(const Conv& c);
bool bwd_data_supported(const Conv& c);
bool wgrad_supported(const Conv& c);
int wgrad_chunks(const Conv& c);
int64_t wgrad_nb(const Conv& c);  // samples per chunk (chunks = ceil(N / wgrad_nb))
cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s);
cudaError_t bwd_data(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s);
cudaError_t wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s);
}  // namespace plane

namespace ibg {
// ibgemm.cu: tensor-core implicit batched GEMM, stride 1, 16-bit data
bool fwd_supported(const Conv& c);
bool bwd_data_supported(const Conv& c);
// cudaErrorNotSupported when this call's input pointer is not 16-byte aligned
cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s);
cudaError_t bwd_data(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s);
}  // namespace ibg

namespace ibc {
// ibgemm_cache.cu: the implicit batched GEMM with its expanded filter (the
// kernel-side im2col) built once into a caller-owned cache
size_t cache_bytes(const Conv& c, bool flip);   // 0: the shape has no cached form
bool call_supported(const Conv& c, bool flip);  // this call's batch / plane sizes run on the cached kernel
cudaError_t build(const Conv& c, bool flip, const void* w, void* cache, cudaStream_t s);
cudaError_t run(const Conv& c, bool flip, const void* in, const void* cache, const void* bias, void* out, bool acc,
                cudaStream_t s);
}  // namespace ibc

namespace wtc {
// wgrad_tc.cu: large-kernel weight gradient (first pass) on the tensor cores,
// 16-bit data, stride 1; cudaErrorNotSupported when this call's x or grad_out
// pointer is not 16-byte aligned or the driver refuses its tensor maps
bool supported(const Conv& c);
cudaError_t wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s);
}  // namespace wtc

}  // namespace dwconv
