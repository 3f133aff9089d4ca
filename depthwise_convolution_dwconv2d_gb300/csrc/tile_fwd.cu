// Small-kernel depthwise forward and stride-1 grad-input on shared-memory
// tiles (square filters K <= 7, equal stride and dilation on both axes).
//
// Forward: y[n, off + c*m + j] = b + sum_{a,b} w[c*m+j, a, b] x[n, c, oh*S - ph + a*D, ow*S - pw + b*D]
// ("Spatial Depthwise Convolution on the GPU #3057", forward kernel with
// padding, stride, dilation, multiplier and bias).
// Grad-input at stride 1 is the same stencil run on grad_out with the filter
// rotated by 180 degrees and padding D*(K-1) - pad, summed over the m output
// channels of each input channel (the adjoint of the forward; #3057's
// grad-input kernel).
#include "plan.h"
#include "tile.cuh"

namespace dwconv {
namespace tile {
namespace {

template <typename T, int K, int S, int D, int R, int V>
__global__ void __launch_bounds__(kNT)
fwd_kernel(Conv c, TileCfg g, const T* __restrict__ x, const T* __restrict__ w,
           const T* __restrict__ bias, T* __restrict__ y) {
  extern __shared__ __align__(16) float sm[];
  constexpr int Q = Geo<K, S, D>::Q;
  const int band = blockIdx.x % g.nbands;
  const int64_t p0 = (int64_t)(blockIdx.x / g.nbands) * g.ppc;  // first plane n*C + c
  const int64_t nplanes = c.N * c.C;
  const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
  const int oh0 = band * g.th;
  const int band_rows = (int)((c.Ho - oh0) < g.th ? (c.Ho - oh0) : g.th);
  const int64_t HW = c.H * c.W;
  load_planes<T>(sm, np, g.tile_floats, g.pitch, [&](int p) { return x + (p0 + p) * HW; },
                 (int)c.H, (int)c.W, oh0 * S - c.ph, g.tr, -c.pw, g.pitch, g.vec_in);
  __syncthreads();
  const int per_rb = g.cb * Q * Q;
  const int per_plane_j = g.rb * per_rb;
  const int total = np * c.m * per_plane_j;
  int cur_pj = -1;
  float wr[K * K];
  float bv = 0.f;
  int64_t oc = 0, n = 0;
  for (int it = threadIdx.x; it < total; it += kNT) {
    const int pj = it / per_plane_j;
    int rem = it - pj * per_plane_j;
    const int rbi = rem / per_rb;
    rem -= rbi * per_rb;
    const int qy = rem / (g.cb * Q);
    rem -= qy * g.cb * Q;
    const int cbi = rem / Q;
    const int qx = rem - cbi * Q;
    if (pj != cur_pj) {
      cur_pj = pj;
      const int pl = pj / c.m, j = pj - pl * c.m;
      const int64_t pin = p0 + pl;
      n = pin / c.C;
      oc = (pin - n * c.C) * c.m + j;
#pragma unroll
      for (int i = 0; i < K * K; ++i) wr[i] = ld(w + oc * (K * K) + i);
      bv = bias ? ld(bias + oc) : 0.f;
    }
    const int pl = pj / c.m;
    const int ohr = rbi * Q * R + qy;
    const int owb = cbi * Q * V + qx;
    float acc[R][V];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int v = 0; v < V; ++v) acc[r][v] = bv;
    conv_block<K, S, D, R, V, Q>(sm + pl * g.tile_floats, g.pitch, ohr * S, owb * S, wr, acc);
    store_block<T, R, V, Q>(y + c.y_base(n, oc), c.Wo, oh0 + ohr, owb, band_rows - ohr, (int)c.Wo,
                            acc, g.vec_out, false);
  }
}

// Stride-1 grad-input: gx[n, c] = sum_j corr(gy[n, off + c*m + j], rot180(w[c*m + j])).
template <typename T, int K, int D, int R, int V>
__global__ void __launch_bounds__(kNT)
bwd1_kernel(Conv c, TileCfg g, int qh, int qw, const T* __restrict__ gy, const T* __restrict__ w,
            T* gx, bool accumulate) {
  extern __shared__ __align__(16) float sm[];
  constexpr int Q = Geo<K, 1, D>::Q;
  const int band = blockIdx.x % g.nbands;
  const int64_t p0 = (int64_t)(blockIdx.x / g.nbands) * g.ppc;  // first gx plane n*C + c
  const int64_t nplanes = c.N * c.C;
  const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
  const int ih0 = band * g.th;
  const int band_rows = (int)((c.H - ih0) < g.th ? (c.H - ih0) : g.th);
  const int m = c.m;
  // staged plane s = pl * m + j holds gy[n, off + c*m + j]
  load_planes<T>(sm, np * m, g.tile_floats, g.pitch,
                 [&](int s) {
                   const int pl = s / m, j = s - pl * m;
                   const int64_t pin = p0 + pl, n = pin / c.C, ch = pin - n * c.C;
                   return gy + c.y_base(n, ch * m + j);
                 },
                 (int)c.Ho, (int)c.Wo, ih0 - qh, g.tr, -qw, g.pitch, g.vec_in);
  __syncthreads();
  const int per_rb = g.cb * Q * Q;
  const int per_plane = g.rb * per_rb;
  const int total = np * per_plane;
  int cur_pl = -1;
  float wr[K * K];
  for (int it = threadIdx.x; it < total; it += kNT) {
    const int pl = it / per_plane;
    int rem = it - pl * per_plane;
    const int rbi = rem / per_rb;
    rem -= rbi * per_rb;
    const int qy = rem / (g.cb * Q);
    rem -= qy * g.cb * Q;
    const int cbi = rem / Q;
    const int qx = rem - cbi * Q;
    const int64_t pin = p0 + pl;
    const int ihr = rbi * Q * R + qy;
    const int iwb = cbi * Q * V + qx;
    float acc[R][V];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int v = 0; v < V; ++v) acc[r][v] = 0.f;
    for (int j = 0; j < m; ++j) {
      if (m > 1 || pl != cur_pl) {
        const int64_t oc = (pin % c.C) * m + j;
#pragma unroll
        for (int i = 0; i < K * K; ++i) wr[i] = ld(w + oc * (K * K) + (K * K - 1 - i));
        cur_pl = pl;
      }
      conv_block<K, 1, D, R, V, Q>(sm + (pl * m + j) * g.tile_floats, g.pitch, ihr, iwb, wr, acc);
    }
    store_block<T, R, V, Q>(gx + pin * c.H * c.W, c.W, ih0 + ihr, iwb, band_rows - ihr, (int)c.W, acc,
                            g.vec_out, accumulate);
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool alignedn(const void* p, int n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }
int esz(int dtype) { return dtype == DWCONV_F32 ? 4 : 2; }

template <typename KernelT, typename... Args>
cudaError_t launch(KernelT kern, const TileCfg& g, cudaStream_t s, Args... args) {
  const size_t smem = smem_bytes(g);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t grid = g.groups * g.nbands;
  kern<<<(unsigned)grid, kNT, smem, s>>>(args...);
  return cudaGetLastError();
}

// Register-block shape per (K, S): R rows x V cols of outputs per thread.
template <int K, int S> struct Blk { static constexpr int R = S == 1 ? 2 : 1, V = 4; };

template <typename T, int K, int S, int D>
cudaError_t run_fwd_t(const Conv& c, const void* x, const void* w, const void* b, void* y,
                      cudaStream_t s) {
  constexpr int R = Blk<K, S>::R, V = Blk<K, S>::V, Q = Geo<K, S, D>::Q;
  VGeo vg{K, S, D, Q, R, V, c.H, c.W, c.Ho, c.Wo, c.ph, c.pw};
  const int es = esz(c.dtype);
  const bool vin = aligned16(x) && (c.W * es) % 16 == 0;
  const bool vout = Q == 1 && c.Wo % 4 == 0 && alignedn(y, 4 * es);
  TileCfg g;
  if (!make_cfg(vg, c.N * c.C, 1, c.m, vin, vout, &g)) return cudaErrorInvalidConfiguration;
  return launch(fwd_kernel<T, K, S, D, R, V>, g, s, c, g, (const T*)x, (const T*)w, (const T*)b, (T*)y);
}

template <typename T, int K, int D>
cudaError_t run_bwd1_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc,
                       cudaStream_t s) {
  constexpr int R = Blk<K, 1>::R, V = Blk<K, 1>::V, Q = Geo<K, 1, D>::Q;
  const int qh = D * (K - 1) - c.ph, qw = D * (K - 1) - c.pw;
  VGeo vg{K, 1, D, Q, R, V, c.Ho, c.Wo, c.H, c.W, qh, qw};
  const int es = esz(c.dtype);
  // gy planes start at multiples of Ho*Wo elements
  const bool vin = aligned16(gy) && (c.Wo * es) % 16 == 0;
  const bool vout = Q == 1 && c.W % 4 == 0 && alignedn(gx, 4 * es);
  TileCfg g;
  if (!make_cfg(vg, c.N * c.C, c.m, 1, vin, vout, &g)) return cudaErrorInvalidConfiguration;
  return launch(bwd1_kernel<T, K, D, R, V>, g, s, c, g, qh, qw, (const T*)gy, (const T*)w, (T*)gx, acc);
}

// (K, S, D) combinations compiled for the forward tile kernel.
#define DW_FWD_CASES(X) X(1, 1, 1) X(3, 1, 1) X(3, 2, 1) X(5, 1, 1) X(5, 2, 1) X(7, 1, 1) \
  X(7, 2, 1) X(3, 1, 2) X(3, 1, 3) X(3, 1, 5) X(5, 1, 2) X(3, 2, 2)
// (K, D) combinations compiled for the stride-1 grad-input tile kernel.
#define DW_BWD1_CASES(X) X(1, 1) X(3, 1) X(5, 1) X(7, 1) X(3, 2) X(3, 3) X(3, 5) X(5, 2)

bool square(const Conv& c) {
  return c.kh == c.kw && c.sh == c.sw && c.dh == c.dw;
}

}  // namespace

bool fwd_supported(const Conv& c) {
  if (!square(c) || c.W > 1024 || c.Wo > 1024) return false;
#define X(K, S, D) if (c.kh == K && c.sh == S && c.dh == D) return true;
  DW_FWD_CASES(X)
#undef X
  return false;
}

template <typename T>
cudaError_t fwd_t(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s) {
#define X(K, S, D) if (c.kh == K && c.sh == S && c.dh == D) return run_fwd_t<T, K, S, D>(c, x, w, b, y, s);
  DW_FWD_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = fwd_t<T>(c, x, w, b, y, s));
  return e;
}

bool bwd1_supported(const Conv& c) {
  if (!square(c) || c.sh != 1 || c.m > 4 || c.W > 1024 || c.Wo > 1024) return false;
  if (c.ph > c.dh * (c.kh - 1) || c.pw > c.dw * (c.kw - 1)) return false;
#define X(K, D) if (c.kh == K && c.dh == D) return true;
  DW_BWD1_CASES(X)
#undef X
  return false;
}

template <typename T>
cudaError_t bwd1_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
#define X(K, D) if (c.kh == K && c.dh == D) return run_bwd1_t<T, K, D>(c, gy, w, gx, acc, s);
  DW_BWD1_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

cudaError_t bwd1(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = bwd1_t<T>(c, gy, w, gx, acc, s));
  return e;
}

}  // namespace tile
}  // namespace dwconv
