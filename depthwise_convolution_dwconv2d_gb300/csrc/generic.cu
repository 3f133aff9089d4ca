// Generic depthwise kernels: correct for every valid descriptor (any kernel
// size, stride, padding, dilation, multiplier, alignment), one output element
// per thread, operands read through the read-only cache. The tiled kernels
// cover the common shapes faster; these are the fallback and the baseline
// they are tested against.
//
// Forward and grad-input follow "Spatial Depthwise Convolution on the GPU
// #3057" (forward / grad-input kernels with padding, stride, dilation and the
// depth multiplier); grad-weight and grad-bias follow its grad-weight kernel
// and grad_bias, split here into a chunked first pass and an ordered second
// pass so the result is bitwise reproducible.
#include "common.cuh"

namespace dwconv {
namespace {

constexpr int kThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kThreads)
fwd_generic_kernel(Conv c, const T* __restrict__ x, const T* __restrict__ w,
                   const T* __restrict__ b, T* __restrict__ y, Epi ep) {
  const int64_t total = c.N * c.OC() * c.Ho * c.Wo;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    int64_t t = idx;
    const int64_t ow = t % c.Wo; t /= c.Wo;
    const int64_t oh = t % c.Ho; t /= c.Ho;
    const int64_t oc = t % c.OC();
    const int64_t n = t / c.OC();
    const T* xp = x + c.x_base(n, oc / c.m);
    const T* wp = w + oc * c.kh * c.kw;
    float acc = 0.f;
    for (int a = 0; a < c.kh; ++a) {
      const int64_t ih = oh * c.sh - c.ph + (int64_t)a * c.dh;
      if (ih < 0 || ih >= c.H) continue;
      for (int bb = 0; bb < c.kw; ++bb) {
        const int64_t iw = ow * c.sw - c.pw + (int64_t)bb * c.dw;
        if (iw < 0 || iw >= c.W) continue;
        acc = fmaf(ld(wp + a * c.kw + bb), ld(xp + ih * c.W + iw), acc);
      }
    }
    if (b) acc += ld(b + oc);
    if (ep.active()) {
      const float sc = ep.scale ? ld(reinterpret_cast<const T*>(ep.scale) + oc) : 1.f;
      const float sh = ep.shift ? ld(reinterpret_cast<const T*>(ep.shift) + oc) : 0.f;
      acc = epi_act(fmaf(acc, sc, sh), ep.act);
    }
    y[c.y_base(n, oc) + oh * c.Wo + ow] = from_f<T>(acc);
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_data_generic_kernel(Conv c, const T* __restrict__ gy, const T* __restrict__ w, T* gx,
                        bool accumulate) {
  const int64_t total = c.N * c.C * c.H * c.W;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    int64_t t = idx;
    const int64_t iw = t % c.W; t /= c.W;
    const int64_t ih = t % c.H; t /= c.H;
    const int64_t ch = t % c.C;
    const int64_t n = t / c.C;
    float acc = 0.f;
    for (int j = 0; j < c.m; ++j) {
      const int64_t oc = ch * c.m + j;
      const T* gp = gy + c.y_base(n, oc);
      const T* wp = w + oc * c.kh * c.kw;
      for (int a = 0; a < c.kh; ++a) {
        const int64_t nh = ih + c.ph - (int64_t)a * c.dh;
        if (nh < 0 || nh % c.sh != 0) continue;
        const int64_t oh = nh / c.sh;
        if (oh >= c.Ho) continue;
        for (int bb = 0; bb < c.kw; ++bb) {
          const int64_t nw = iw + c.pw - (int64_t)bb * c.dw;
          if (nw < 0 || nw % c.sw != 0) continue;
          const int64_t ow = nw / c.sw;
          if (ow >= c.Wo) continue;
          acc = fmaf(ld(wp + a * c.kw + bb), ld(gp + oh * c.Wo + ow), acc);
        }
      }
    }
    if (accumulate) acc += ld_rw(gx + idx);
    gx[idx] = from_f<T>(acc);
  }
}

// Sum of one value per thread over the block, in a fixed tree order.
__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x == 0) {
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
  }
  return s;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_weight_generic_pass1_kernel(Conv c, const T* __restrict__ x, const T* __restrict__ gy,
                                float* __restrict__ ws, int chunks, bool want_w, bool want_b) {
  __shared__ float red[kThreads / 32];
  const int64_t oc = blockIdx.x;
  const int chunk = blockIdx.y;
  const int64_t nb = (c.N + chunks - 1) / chunks;
  const int64_t n0 = chunk * nb;
  const int64_t n1 = n0 + nb < c.N ? n0 + nb : c.N;
  const int64_t hw = c.Ho * c.Wo;
  const int64_t P = n1 > n0 ? (n1 - n0) * hw : 0;
  const int taps = c.kh * c.kw;
  const int64_t ch = oc / c.m;
  float* out = ws + ((int64_t)chunk * c.OC() + oc) * (taps + 1);
  for (int tap = 0; tap <= taps; ++tap) {
    if (tap < taps && !want_w) continue;
    if (tap == taps && !want_b) continue;
    const int a = tap < taps ? tap / c.kw : 0;
    const int bb = tap < taps ? tap % c.kw : 0;
    float acc = 0.f;
    for (int64_t p = threadIdx.x; p < P; p += blockDim.x) {
      const int64_t n = n0 + p / hw;
      const int64_t r = p % hw;
      const int64_t oh = r / c.Wo, ow = r % c.Wo;
      const float g = ld(gy + c.y_base(n, oc) + r);
      if (tap == taps) { acc += g; continue; }
      const int64_t ih = oh * c.sh - c.ph + (int64_t)a * c.dh;
      const int64_t iw = ow * c.sw - c.pw + (int64_t)bb * c.dw;
      if (ih < 0 || ih >= c.H || iw < 0 || iw >= c.W) continue;
      acc = fmaf(g, ld(x + c.x_base(n, ch) + ih * c.W + iw), acc);
    }
    const float s = block_sum(acc, red);
    if (threadIdx.x == 0) out[tap] = s;
  }
}

// One warp per output: the lanes load chunks lane, lane + 32, ... at once
// (one memory round trip per 32 chunks instead of one per chunk), then every
// lane runs the same sum over the shuffled values in chunk index order, so
// the rounding is that of the plain sequential sum.
template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_weight_pass2_kernel(Conv c, const float* __restrict__ ws, int chunks, T* gw, T* gb) {
  const int taps = c.kh * c.kw;
  const int64_t total = c.OC() * (taps + 1);
  const int lane = threadIdx.x & 31;
  const int64_t wpb = blockDim.x >> 5;
  for (int64_t idx = blockIdx.x * wpb + (threadIdx.x >> 5); idx < total; idx += (int64_t)gridDim.x * wpb) {
    const int64_t oc = idx / (taps + 1);
    const int tap = (int)(idx % (taps + 1));
    if (tap < taps ? gw == nullptr : gb == nullptr) continue;  // warp-uniform
    float s = 0.f;
    for (int kb = 0; kb < chunks; kb += 32) {
      const float v = kb + lane < chunks ? ws[(int64_t)(kb + lane) * total + idx] : 0.f;
      const int nk = chunks - kb < 32 ? chunks - kb : 32;
      for (int j = 0; j < nk; ++j) s += __shfl_sync(0xffffffffu, v, j);
    }
    if (lane == 0) {
      if (tap < taps) gw[oc * taps + tap] = from_f<T>(s);
      else gb[oc] = from_f<T>(s);
    }
  }
}

// Sum over branches of each branch's grad-input, accumulated in fp32 and
// rounded once (the chain rule through a channel concatenation).
template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_data_multi_generic_kernel(MultiGeneric g, const T* __restrict__ gy, T* gx) {
  const Conv& c0 = g.c[0];
  const int64_t total = c0.N * c0.C * c0.H * c0.W;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    int64_t t = idx;
    const int64_t iw = t % c0.W; t /= c0.W;
    const int64_t ih = t % c0.H; t /= c0.H;
    const int64_t ch = t % c0.C;
    const int64_t n = t / c0.C;
    float acc = 0.f;
    for (int br = 0; br < g.nb; ++br) {
      const Conv& c = g.c[br];
      const T* w = (const T*)g.w[br];
      for (int j = 0; j < c.m; ++j) {
        const int64_t oc = ch * c.m + j;
        const T* gp = gy + c.y_base(n, oc);
        const T* wp = w + oc * c.kh * c.kw;
        for (int a = 0; a < c.kh; ++a) {
          const int64_t nh = ih + c.ph - (int64_t)a * c.dh;
          if (nh < 0 || nh % c.sh != 0) continue;
          const int64_t oh = nh / c.sh;
          if (oh >= c.Ho) continue;
          for (int bb = 0; bb < c.kw; ++bb) {
            const int64_t nw = iw + c.pw - (int64_t)bb * c.dw;
            if (nw < 0 || nw % c.sw != 0) continue;
            const int64_t ow = nw / c.sw;
            if (ow >= c.Wo) continue;
            acc = fmaf(ld(wp + a * c.kw + bb), ld(gp + oh * c.Wo + ow), acc);
          }
        }
      }
    }
    gx[idx] = from_f<T>(acc);
  }
}

int grid_for(int64_t total) {
  int64_t g = (total + kThreads - 1) / kThreads;
  const int64_t cap = 152 * 32;  // enough resident blocks to fill every SM
  if (g > cap) g = cap;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

cudaError_t fwd_generic(const Conv& c, const void* x, const void* w, const void* b, void* y,
                        cudaStream_t s, const Epi& ep) {
  const int g = grid_for(c.N * c.OC() * c.Ho * c.Wo);
  DWCONV_DISPATCH_DTYPE(c.dtype, T,
    fwd_generic_kernel<T><<<g, kThreads, 0, s>>>(c, (const T*)x, (const T*)w, (const T*)b, (T*)y, ep));
  return cudaGetLastError();
}

cudaError_t bwd_data_generic(const Conv& c, const void* gy, const void* w, void* gx,
                             bool accumulate, cudaStream_t s) {
  const int g = grid_for(c.N * c.C * c.H * c.W);
  DWCONV_DISPATCH_DTYPE(c.dtype, T,
    bwd_data_generic_kernel<T><<<g, kThreads, 0, s>>>(c, (const T*)gy, (const T*)w, (T*)gx, accumulate));
  return cudaGetLastError();
}

cudaError_t bwd_data_multi_generic(const MultiGeneric& m, const void* gy, void* gx, cudaStream_t s) {
  const Conv& c = m.c[0];
  const int g = grid_for(c.N * c.C * c.H * c.W);
  DWCONV_DISPATCH_DTYPE(c.dtype, T,
    bwd_data_multi_generic_kernel<T><<<g, kThreads, 0, s>>>(m, (const T*)gy, (T*)gx));
  return cudaGetLastError();
}

cudaError_t bwd_weight_generic_pass1(const Conv& c, const void* x, const void* gy, float* ws,
                                     int chunks, bool want_w, bool want_b, cudaStream_t s) {
  dim3 grid((unsigned)c.OC(), chunks);
  DWCONV_DISPATCH_DTYPE(c.dtype, T,
    bwd_weight_generic_pass1_kernel<T><<<grid, kThreads, 0, s>>>(c, (const T*)x, (const T*)gy, ws,
                                                                 chunks, want_w, want_b));
  return cudaGetLastError();
}

cudaError_t bwd_weight_pass2(const Conv& c, const float* ws, int chunks, void* gw, void* gb,
                             cudaStream_t s) {
  const int g = grid_for(c.OC() * (c.kh * c.kw + 1) * 32);  // a warp per output
  DWCONV_DISPATCH_DTYPE(c.dtype, T,
    bwd_weight_pass2_kernel<T><<<g, kThreads, 0, s>>>(c, ws, chunks, (T*)gw, (T*)gb));
  return cudaGetLastError();
}

}  // namespace dwconv
