// Fused multi-branch depthwise forward and grad-input (stride 1, m = 1).
//
// The DynamicConvolutionOperator README ("Solution") computes the dilation 1,
// 3 and 5 branches of one input in a single launch and stores each branch's
// result through strided pointers straight into its slice of the
// concatenated output, so no unfold buffer and no torch.cat copy exist.
// Here one CTA stages a band of x once (with the largest branch's halo) and
// evaluates every branch from that tile, each with the thread spacing that
// suits its dilation, writing branch b into channels [off_b, off_b + C).
// The grad-input of the concatenation is the sum of the branches' grad-inputs;
// it is computed in one launch from the branches' grad_out slices, summed in
// fp32 and rounded once.
#include "plan.h"
#include "tile.cuh"

namespace dwconv {
namespace tile {
namespace {

constexpr int kR = 2, kV = 4;

struct MultiArgs {
  int nb;
  int pad_h[3], pad_w[3];     // per-branch padding
  int oy[3], ox[3];           // per-branch offset of tap (0,0) in the tile
  int rb[3], cb[3];           // item grid per branch
  int items[3];               // items per plane per branch
  int64_t off[3];             // channel offset of each branch slice
  const void* w[3];
  const void* bias[3];
  int tr[3], tile_floats[3];  // bwd: per-branch tiles
  int iy0[3], ix0[3];         // bwd: tile origins relative to the band
};

template <int K, int D, int Q, typename T>
__device__ __forceinline__ void fwd_branch(const Conv& c, const MultiArgs& a, int b, const float* t,
                                           int pitch, int item, int64_t n, int64_t ch, int oh0,
                                           int band_rows, const T* w, const T* bias, T* y) {
  const int per_rb = a.cb[b] * Q * Q;
  const int rbi = item / per_rb;
  int rem = item - rbi * per_rb;
  const int qy = rem / (a.cb[b] * Q);
  rem -= qy * a.cb[b] * Q;
  const int cbi = rem / Q;
  const int qx = rem - cbi * Q;
  float wr[K * K];
#pragma unroll
  for (int i = 0; i < K * K; ++i) wr[i] = ld(w + ch * (K * K) + i);
  const float bv = bias ? ld(bias + ch) : 0.f;
  float acc[kR][kV];
#pragma unroll
  for (int r = 0; r < kR; ++r)
#pragma unroll
    for (int v = 0; v < kV; ++v) acc[r][v] = bv;
  const int ohr = rbi * Q * kR + qy;
  const int owb = cbi * Q * kV + qx;
  conv_block<K, 1, D, kR, kV, Q>(t, pitch, ohr + a.oy[b], owb + a.ox[b], wr, acc);
  const bool vec = Q == 1 && c.Wo % 4 == 0 &&
                   (reinterpret_cast<uintptr_t>(y) % (4 * sizeof(T))) == 0;
  store_block<T, kR, kV, Q>(y + (n * c.ctot + a.off[b] + ch) * c.Ho * c.Wo, c.Wo, oh0 + ohr, owb,
                            band_rows - ohr, (int)c.Wo, acc, vec, false);
}

template <typename T, int K, int NB, int D0, int D1, int D2>
__global__ void __launch_bounds__(kNT)
fwd_multi_kernel(Conv c, TileCfg g, MultiArgs a, const T* __restrict__ x, T* __restrict__ y) {
  extern __shared__ __align__(16) float sm[];
  const int band = blockIdx.x % g.nbands;
  const int64_t p0 = (int64_t)(blockIdx.x / g.nbands) * g.ppc;
  const int64_t nplanes = c.N * c.C;
  const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
  const int oh0 = band * g.th;
  const int band_rows = (int)((c.Ho - oh0) < g.th ? (c.Ho - oh0) : g.th);
  const int64_t HW = c.H * c.W;
  load_planes<T>(sm, np, g.tile_floats, g.pitch, [&](int p) { return x + (p0 + p) * HW; },
                 (int)c.H, (int)c.W, oh0 + a.iy0[0], g.tr, a.ix0[0], g.pitch, g.vec_in);
  __syncthreads();
  const int i0 = a.items[0], i1 = a.items[1], i2 = NB > 2 ? a.items[2] : 0;
  const int per_plane = i0 + i1 + i2;
  for (int it = threadIdx.x; it < np * per_plane; it += kNT) {
    const int pl = it / per_plane;
    const int q = it - pl * per_plane;
    const int64_t pin = p0 + pl, n = pin / c.C, ch = pin - n * c.C;
    const float* t = sm + pl * g.tile_floats;
    if (q < i0) {
      fwd_branch<K, D0, D0>(c, a, 0, t, g.pitch, q, n, ch, oh0, band_rows, (const T*)a.w[0],
                            (const T*)a.bias[0], y);
    } else if (q < i0 + i1) {
      fwd_branch<K, D1, D1>(c, a, 1, t, g.pitch, q - i0, n, ch, oh0, band_rows, (const T*)a.w[1],
                            (const T*)a.bias[1], y);
    } else if (NB > 2) {
      fwd_branch<K, D2, D2>(c, a, 2, t, g.pitch, q - i0 - i1, n, ch, oh0, band_rows,
                            (const T*)a.w[2], (const T*)a.bias[2], y);
    }
  }
}

template <typename T, int K, int NB, int D0, int D1, int D2>
__global__ void __launch_bounds__(kNT)
bwd_multi_kernel(Conv c, TileCfg g, MultiArgs a, const T* __restrict__ gy, T* gx) {
  extern __shared__ __align__(16) float sm[];
  const int band = blockIdx.x % g.nbands;
  const int64_t p0 = (int64_t)(blockIdx.x / g.nbands) * g.ppc;
  const int64_t nplanes = c.N * c.C;
  const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
  const int ih0 = band * g.th;
  const int band_rows = (int)((c.H - ih0) < g.th ? (c.H - ih0) : g.th);
  const int slice = a.tile_floats[0] + a.tile_floats[1] + (NB > 2 ? a.tile_floats[2] : 0);
  for (int b = 0; b < NB; ++b) {
    const int boff = b == 0 ? 0 : (b == 1 ? a.tile_floats[0] : a.tile_floats[0] + a.tile_floats[1]);
    load_planes<T>(sm + boff, np, slice, g.pitch,
                   [&](int p) {
                     const int64_t pin = p0 + p, n = pin / c.C, ch = pin - n * c.C;
                     return gy + (n * c.ctot + a.off[b] + ch) * c.Ho * c.Wo;
                   },
                   (int)c.Ho, (int)c.Wo, ih0 + a.iy0[b], a.tr[b], a.ix0[b], g.pitch, g.vec_in);
  }
  __syncthreads();
  const int per_rb = g.cb;
  const int per_plane = g.rb * per_rb;
  int cur = -1;
  float w0[K * K], w1[K * K], w2[K * K];
  for (int it = threadIdx.x; it < np * per_plane; it += kNT) {
    const int pl = it / per_plane;
    const int rem = it - pl * per_plane;
    const int rbi = rem / per_rb;
    const int cbi = rem - rbi * per_rb;
    const int64_t pin = p0 + pl, ch = pin % c.C;
    if (pl != cur) {
      cur = pl;
#pragma unroll
      for (int i = 0; i < K * K; ++i) {
        w0[i] = ld((const T*)a.w[0] + ch * (K * K) + (K * K - 1 - i));
        w1[i] = ld((const T*)a.w[1] + ch * (K * K) + (K * K - 1 - i));
        w2[i] = NB > 2 ? ld((const T*)a.w[2] + ch * (K * K) + (K * K - 1 - i)) : 0.f;
      }
    }
    float acc[kR][kV];
#pragma unroll
    for (int r = 0; r < kR; ++r)
#pragma unroll
      for (int v = 0; v < kV; ++v) acc[r][v] = 0.f;
    const int ihr = rbi * kR, iwb = cbi * kV;
    const float* t = sm + pl * slice;
    conv_block<K, 1, D0, kR, kV, 1>(t, g.pitch, ihr, iwb, w0, acc);
    conv_block<K, 1, D1, kR, kV, 1>(t + a.tile_floats[0], g.pitch, ihr, iwb, w1, acc);
    if (NB > 2)
      conv_block<K, 1, D2, kR, kV, 1>(t + a.tile_floats[0] + a.tile_floats[1], g.pitch, ihr, iwb, w2, acc);
    store_block<T, kR, kV, 1>(gx + pin * c.H * c.W, c.W, ih0 + ihr, iwb, band_rows - ihr, (int)c.W,
                              acc, g.vec_out, false);
  }
}

int lcm(int a, int b) {
  int x = a, y = b;
  while (y) { const int t = x % y; x = y; y = t; }
  return a / x * b;
}

int64_t read_cols(int K, int D, int Q, int cb) {
  const int WN = (kV - 1) * Q + (K - 1) * D + 1;
  if (Q == 1) return (int64_t)(cb - 1) * kV + (WN + 3) / 4 * 4;
  const int64_t owb = (int64_t)(cb - 1) * Q * kV + Q - 1;
  return owb + WN;
}

template <typename T, int K, int NB, int D0, int D1, int D2>
cudaError_t run_fwd_multi(const Conv* cs, const void* x, const void* const* w, const void* const* bias,
                          void* y, cudaStream_t s) {
  const Conv& c = cs[0];
  const int Ds[3] = {D0, D1, D2};
  MultiArgs a{};
  a.nb = NB;
  int hh = 0, hw = 0;
  for (int b = 0; b < NB; ++b) {
    a.pad_h[b] = cs[b].ph; a.pad_w[b] = cs[b].pw;
    hh = cs[b].ph > hh ? cs[b].ph : hh;
    hw = cs[b].pw > hw ? cs[b].pw : hw;
    a.off[b] = cs[b].off;
    a.w[b] = w[b];
    a.bias[b] = bias ? bias[b] : nullptr;
  }
  // column origin: every dilation-1 branch needs its tap-(0,0) column at a
  // multiple of 4 (float4 windows)
  int e = 0;
  for (; e < 4; ++e) {
    bool ok = true;
    for (int b = 0; b < NB; ++b)
      if (Ds[b] == 1 && (hw + e - cs[b].pw) % 4 != 0) ok = false;
    if (ok) break;
  }
  if (e == 4) return cudaErrorInvalidConfiguration;
  int L = 1;
  for (int b = 0; b < NB; ++b) L = lcm(L, Ds[b] * kR);
  TileCfg g{};
  int64_t need_cols = c.W + hw + e;
  for (int b = 0; b < NB; ++b) {
    a.oy[b] = hh - cs[b].ph;
    a.ox[b] = hw + e - cs[b].pw;
    a.cb[b] = (int)((c.Wo + (int64_t)Ds[b] * kV - 1) / ((int64_t)Ds[b] * kV));
    const int64_t rc = a.ox[b] + read_cols(K, Ds[b], Ds[b], a.cb[b]);
    if (rc > need_cols) need_cols = rc;
  }
  g.pitch = round4(need_cols);
  auto tr_of = [&](int64_t th) {
    int64_t t = 0;
    for (int b = 0; b < NB; ++b) {
      const int64_t r = th - 1 + a.oy[b] + (int64_t)(K - 1) * Ds[b] + 1;
      if (r > t) t = r;
    }
    return t;
  };
  const int64_t target = 48 * 1024;
  int64_t th = (c.Ho + L - 1) / L * L;
  while (th > L && tr_of(th) * g.pitch * 4 > target) th -= L;
  if (tr_of(th) * g.pitch * 4 > 200 * 1024) return cudaErrorInvalidConfiguration;
  g.th = (int)th;
  g.nbands = (int)((c.Ho + th - 1) / th);
  g.tr = (int)tr_of(th);
  g.tile_floats = g.tr * g.pitch;
  g.ntile = 1;
  int64_t items = 0;
  for (int b = 0; b < NB; ++b) {
    a.rb[b] = (int)(th / (Ds[b] * kR));
    a.items[b] = a.rb[b] * a.cb[b] * Ds[b] * Ds[b];
    items += a.items[b];
  }
  a.iy0[0] = -hh;
  a.ix0[0] = -(hw + e);
  const int64_t nplanes = c.N * c.C;
  int64_t ppc = 1;
  if (g.nbands == 1) {
    ppc = (2 * kNT + items - 1) / items;
    const int64_t cap = target / ((int64_t)g.tile_floats * 4);
    if (ppc > cap) ppc = cap;
    if ((nplanes + ppc - 1) / ppc < 152 * 4) ppc = (nplanes + 152 * 4 - 1) / (152 * 4);
    if (ppc < 1) ppc = 1;
  }
  g.ppc = (int)ppc;
  g.groups = (nplanes + ppc - 1) / ppc;
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  g.vec_in = ((reinterpret_cast<uintptr_t>(x) & 15) == 0) && (c.W * es) % 16 == 0;
  const size_t smem = (size_t)g.ppc * g.tile_floats * 4;
  auto kern = fwd_multi_kernel<T, K, NB, D0, D1, D2>;
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  kern<<<(unsigned)(g.groups * g.nbands), kNT, smem, s>>>(c, g, a, (const T*)x, (T*)y);
  return cudaGetLastError();
}

template <typename T, int K, int NB, int D0, int D1, int D2>
cudaError_t run_bwd_multi(const Conv* cs, const void* gy, const void* const* w, void* gx,
                          cudaStream_t s) {
  const Conv& c = cs[0];
  const int Ds[3] = {D0, D1, D2};
  MultiArgs a{};
  a.nb = NB;
  TileCfg g{};
  g.cb = (int)((c.W + kV - 1) / kV);
  int64_t need_cols = 0;
  for (int b = 0; b < NB; ++b) {
    const int qh = Ds[b] * (K - 1) - cs[b].ph, qw = Ds[b] * (K - 1) - cs[b].pw;
    if (qh < 0 || qw < 0) return cudaErrorInvalidConfiguration;
    a.off[b] = cs[b].off;
    a.w[b] = w[b];
    a.iy0[b] = -qh;
    a.ix0[b] = -qw;
    int64_t rc = read_cols(K, Ds[b], 1, g.cb);
    if (c.Wo + qw > rc) rc = c.Wo + qw;
    if (rc > need_cols) need_cols = rc;
  }
  g.pitch = round4(need_cols);
  auto bytes_of = [&](int64_t th) {
    int64_t t = 0;
    for (int b = 0; b < NB; ++b) t += (th - 1 + (int64_t)(K - 1) * Ds[b] + 1) * g.pitch;
    return t * 4;
  };
  const int64_t target = 48 * 1024;
  int64_t th = (c.H + kR - 1) / kR * kR;
  while (th > kR && bytes_of(th) > target) th -= kR;
  if (bytes_of(th) > 200 * 1024) return cudaErrorInvalidConfiguration;
  g.th = (int)th;
  g.rb = (int)(th / kR);
  g.nbands = (int)((c.H + th - 1) / th);
  for (int b = 0; b < NB; ++b) {
    a.tr[b] = (int)(th - 1 + (int64_t)(K - 1) * Ds[b] + 1);
    a.tile_floats[b] = a.tr[b] * g.pitch;
  }
  g.ntile = NB;
  const int64_t slice_bytes = bytes_of(th);
  const int64_t items = (int64_t)g.rb * g.cb;
  const int64_t nplanes = c.N * c.C;
  int64_t ppc = 1;
  if (g.nbands == 1) {
    ppc = (2 * kNT + items - 1) / items;
    const int64_t cap = target / slice_bytes;
    if (ppc > cap) ppc = cap;
    if ((nplanes + ppc - 1) / ppc < 152 * 4) ppc = (nplanes + 152 * 4 - 1) / (152 * 4);
    if (ppc < 1) ppc = 1;
  }
  g.ppc = (int)ppc;
  g.groups = (nplanes + ppc - 1) / ppc;
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  g.vec_in = ((reinterpret_cast<uintptr_t>(gy) & 15) == 0) && (c.Wo * es) % 16 == 0;
  g.vec_out = c.W % 4 == 0 && (reinterpret_cast<uintptr_t>(gx) % (4 * es)) == 0;
  const size_t smem = (size_t)g.ppc * slice_bytes;
  auto kern = bwd_multi_kernel<T, K, NB, D0, D1, D2>;
  if (smem > 48 * 1024) {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
  }
  kern<<<(unsigned)(g.groups * g.nbands), kNT, smem, s>>>(c, g, a, (const T*)gy, (T*)gx);
  return cudaGetLastError();
}

// Dilation sets compiled for the fused path (3x3 filters).
#define DW_MULTI_CASES(X) X(3, 3, 1, 3, 5) X(3, 2, 1, 2, 0) X(3, 2, 1, 3, 0) X(3, 3, 1, 2, 3)

bool same_geometry(int nb, const Conv* cs) {
  for (int b = 0; b < nb; ++b) {
    const Conv& c = cs[b];
    if (c.kh != c.kw || c.sh != 1 || c.sw != 1 || c.dh != c.dw || c.m != 1) return false;
    if (c.W > 512) return false;
  }
  return nb == 2 || nb == 3;
}

template <typename T>
cudaError_t fwd_multi_t(int nb, const Conv* cs, const void* x, const void* const* w,
                        const void* const* bias, void* y, cudaStream_t s) {
#define X(K, NB, D0, D1, D2)                                                                 \
  if (nb == NB && cs[0].kh == K && cs[0].dh == D0 && cs[1].dh == D1 && (NB < 3 || cs[2].dh == D2)) \
    return run_fwd_multi<T, K, NB, D0, D1, D2>(cs, x, w, bias, y, s);
  DW_MULTI_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

template <typename T>
cudaError_t bwd_multi_t(int nb, const Conv* cs, const void* gy, const void* const* w, void* gx,
                        cudaStream_t s) {
#define X(K, NB, D0, D1, D2)                                                                 \
  if (nb == NB && cs[0].kh == K && cs[0].dh == D0 && cs[1].dh == D1 && (NB < 3 || cs[2].dh == D2)) \
    return run_bwd_multi<T, K, NB, D0, D1, D2>(cs, gy, w, gx, s);
  DW_MULTI_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace

bool multi_supported(int nb, const Conv* cs) {
  if (!same_geometry(nb, cs)) return false;
  for (int b = 0; b < nb; ++b)
    if (cs[b].kh != cs[0].kh) return false;
#define X(K, NB, D0, D1, D2) \
  if (nb == NB && cs[0].kh == K && cs[0].dh == D0 && cs[1].dh == D1 && (NB < 3 || cs[2].dh == D2)) return true;
  DW_MULTI_CASES(X)
#undef X
  return false;
}

cudaError_t fwd_multi(int nb, const Conv* cs, const void* x, const void* const* w,
                      const void* const* bias, void* y, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(cs[0].dtype, T, e = fwd_multi_t<T>(nb, cs, x, w, bias, y, s));
  return e;
}

cudaError_t bwd_multi(int nb, const Conv* cs, const void* gy, const void* const* w, void* gx,
                      cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(cs[0].dtype, T, e = bwd_multi_t<T>(nb, cs, gy, w, gx, s));
  return e;
}

}  // namespace tile
}  // namespace dwconv
