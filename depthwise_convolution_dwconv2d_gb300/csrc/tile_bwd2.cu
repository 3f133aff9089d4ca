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
#include "plan.h"
#include "tile.cuh"

namespace dwconv {
namespace tile {
namespace {

template <int K, int S, int D, int PM>
struct Phase {
  static constexpr bool valid(int phi, int a) { return (phi + PM - a * D) % S == 0; }
  static constexpr int off(int phi, int a) { return (phi + PM - a * D) / S; }
  static constexpr int omin() {
    int o = 1 << 20;
    for (int p = 0; p < S; ++p)
      for (int a = 0; a < K; ++a)
        if (valid(p, a) && off(p, a) < o) o = off(p, a);
    return o;
  }
  static constexpr int omax() {
    int o = -(1 << 20);
    for (int p = 0; p < S; ++p)
      for (int a = 0; a < K; ++a)
        if (valid(p, a) && off(p, a) > o) o = off(p, a);
    return o;
  }
  static constexpr int span = omax() - omin();
};

struct Bwd2Cfg {
  int ppc, thu, nbands, tr, pitch, rb, cb, tile_floats, vec_in, vec_out;
  int64_t groups;
  int row0, col0;  // grad_out row / col of tile (0, 0) relative to u_band0 / 0
};

template <typename T, int K, int S, int D, int PM, int R, int V>
__global__ void __launch_bounds__(kNT)
bwd2_kernel(Conv c, Bwd2Cfg g, const T* __restrict__ gy, const T* __restrict__ w, T* gx,
            bool accumulate) {
  extern __shared__ __align__(16) float sm[];
  using P = Phase<K, S, D, PM>;
  constexpr int OM = P::omin(), SP = P::span;
  constexpr int WN = V + SP;
  constexpr int WN4 = (WN + 3) / 4 * 4;
  const int band = blockIdx.x % g.nbands;
  const int64_t p0 = (int64_t)(blockIdx.x / g.nbands) * g.ppc;
  const int64_t nplanes = c.N * c.C;
  const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
  const int u0 = band * g.thu;  // first u row of the band (gx row S*u0)
  const int m = c.m;
  load_planes<T>(sm, np * m, g.tile_floats, g.pitch,
                 [&](int s) {
                   const int pl = s / m, j = s - pl * m;
                   const int64_t pin = p0 + pl, n = pin / c.C, ch = pin - n * c.C;
                   return gy + c.y_base(n, ch * m + j);
                 },
                 (int)c.Ho, (int)c.Wo, u0 + g.row0, g.tr, g.col0, g.pitch, g.vec_in);
  __syncthreads();
  const int per_plane = g.rb * g.cb;
  const int total = np * per_plane;
  float wr[K * K];
  int cur_pl = -1;
  for (int it = threadIdx.x; it < total; it += kNT) {
    const int pl = it / per_plane;
    int rem = it - pl * per_plane;
    const int rbi = rem / g.cb;
    const int cbi = rem - rbi * g.cb;
    const int64_t pin = p0 + pl;
    float acc[R][S][V][S];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int ph = 0; ph < S; ++ph)
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
          for (int pw = 0; pw < S; ++pw) acc[r][ph][v][pw] = 0.f;
    for (int j = 0; j < m; ++j) {
      if (m > 1 || pl != cur_pl) {
        const int64_t oc = (pin % c.C) * m + j;
#pragma unroll
        for (int i = 0; i < K * K; ++i) wr[i] = ld(w + oc * (K * K) + i);
        cur_pl = pl;
      }
      const float* t = sm + (pl * m + j) * g.tile_floats + (rbi * R) * g.pitch + cbi * V;
#pragma unroll
      for (int ut = 0; ut < R + SP; ++ut) {
        float win[WN4];
#pragma unroll
        for (int i = 0; i < WN4 / 4; ++i) {
          const float4 f = *reinterpret_cast<const float4*>(t + ut * g.pitch + 4 * i);
          win[4 * i] = f.x; win[4 * i + 1] = f.y; win[4 * i + 2] = f.z; win[4 * i + 3] = f.w;
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int ph = 0; ph < S; ++ph)
#pragma unroll
            for (int a = 0; a < K; ++a) {
              if (!P::valid(ph, a) || r + P::off(ph, a) - OM != ut) continue;
#pragma unroll
              for (int pw = 0; pw < S; ++pw)
#pragma unroll
                for (int b = 0; b < K; ++b) {
                  if (!P::valid(pw, b)) continue;
#pragma unroll
                  for (int v = 0; v < V; ++v)
                    acc[r][ph][v][pw] = fmaf(wr[a * K + b], win[v + P::off(pw, b) - OM], acc[r][ph][v][pw]);
                }
            }
      }
    }
    // store rows S*(u0 + rbi*R + r) + ph, cols S*cbi*V .. + S*V
    T* plane = gx + pin * c.H * c.W;
    const int col0 = S * V * cbi;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int ph = 0; ph < S; ++ph) {
        const int64_t ih = (int64_t)S * (u0 + rbi * R + r) + ph;
        if (ih >= c.H) continue;
        T* rowp = plane + ih * c.W;
        float o[S * V];
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
          for (int pw = 0; pw < S; ++pw) o[v * S + pw] = acc[r][ph][v][pw];
        if (g.vec_out && (S * V) % 4 == 0 && col0 + S * V <= c.W) {
#pragma unroll
          for (int q = 0; q < S * V / 4; ++q) {
            float f[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) f[i] = accumulate ? o[4 * q + i] + ld_rw(rowp + col0 + 4 * q + i) : o[4 * q + i];
            store_vec<T, 4>(rowp + col0 + 4 * q, f);
          }
        } else {
#pragma unroll
          for (int i = 0; i < S * V; ++i) {
            const int iw = col0 + i;
            if (iw < c.W) rowp[iw] = from_f<T>(accumulate ? o[i] + ld_rw(rowp + iw) : o[i]);
          }
        }
      }
  }
}

template <typename T, int K, int S, int D, int PM>
cudaError_t run_bwd2_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc,
                       cudaStream_t s) {
  constexpr int R = 2, V = 4;
  using P = Phase<K, S, D, PM>;
  constexpr int OM = P::omin(), SP = P::span;
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  Bwd2Cfg g{};
  const int64_t U = (c.H + S - 1) / S;  // u rows of gx
  g.cb = (int)((c.W + (int64_t)S * V - 1) / ((int64_t)S * V));
  const int WN4 = (V + SP + 3) / 4 * 4;
  g.pitch = round4((int64_t)(g.cb - 1) * V + WN4);
  g.row0 = (c.ph - PM) / S + OM;
  g.col0 = (c.pw - PM) / S + OM;
  const int64_t target = 40 * 1024;
  const int64_t row_bytes = (int64_t)g.pitch * 4 * c.m;
  int64_t thu = (U + R - 1) / R * R;
  if ((thu + SP) * row_bytes > target) {
    thu = (target / row_bytes - SP) / R * R;
    if (thu < R) thu = R;
    if ((thu + SP) * row_bytes > 96 * 1024) return cudaErrorInvalidConfiguration;
  }
  g.thu = (int)thu;
  g.rb = (int)(thu / R);
  g.nbands = (int)((U + thu - 1) / thu);
  g.tr = (int)(thu + SP);
  g.tile_floats = g.tr * g.pitch;
  const int64_t items = (int64_t)g.rb * g.cb;
  const int64_t nplanes = c.N * c.C;
  int64_t ppc = 1;
  if (g.nbands == 1) {
    ppc = (2 * kNT + items - 1) / items;
    const int64_t cap = target / ((int64_t)g.tile_floats * 4 * c.m);
    if (ppc > cap) ppc = cap;
    if ((nplanes + ppc - 1) / ppc < 152 * 4) ppc = (nplanes + 152 * 4 - 1) / (152 * 4);
    if (ppc < 1) ppc = 1;
  }
  g.ppc = (int)ppc;
  g.groups = (nplanes + ppc - 1) / ppc;
  g.vec_in = ((reinterpret_cast<uintptr_t>(gy) & 15) == 0) && (c.Wo * es) % 16 == 0;
  g.vec_out = (reinterpret_cast<uintptr_t>(gx) % (4 * es) == 0) && c.W % 4 == 0;
  const size_t smem = (size_t)g.ppc * c.m * g.tile_floats * sizeof(float);
  auto kern = bwd2_kernel<T, K, S, D, PM, R, V>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)(g.groups * g.nbands), kNT, smem, s>>>(c, g, (const T*)gy, (const T*)w, (T*)gx, acc);
  return cudaGetLastError();
}

#define DW_BWD2_CASES(X) X(3, 2, 1, 0) X(3, 2, 1, 1) X(5, 2, 1, 0) X(5, 2, 1, 1) X(7, 2, 1, 1) X(7, 2, 1, 0)

template <typename T>
cudaError_t bwd2_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
  const int pm = c.ph % c.sh;
#define X(K, S, D, PM) \
  if (c.kh == K && c.sh == S && c.dh == D && pm == PM) return run_bwd2_t<T, K, S, D, PM>(c, gy, w, gx, acc, s);
  DW_BWD2_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace

bool bwd2_supported(const Conv& c) {
  if (c.kh != c.kw || c.sh != c.sw || c.dh != c.dw || c.sh < 2 || c.m > 4) return false;
  if (c.W > 1024 || c.Wo > 1024) return false;
  if (c.ph % c.sh != c.pw % c.sh) return false;
  const int pm = c.ph % c.sh;
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
