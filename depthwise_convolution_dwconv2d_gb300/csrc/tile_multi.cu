// Fused multi-branch depthwise forward and grad-input (stride 1, m = 1).
//
// The DynamicConvolutionOperator README ("Solution") computes the dilation 1,
// 3 and 5 branches of one input in a single launch and stores each branch's
// result through strided pointers straight into its slice of the
// concatenated output, so no unfold buffer and no torch.cat copy exist.
// Here one CTA stages a band of x once (with the largest branch's halo) and
// evaluates every branch from that tile, each with the thread spacing that
// suits its dilation, writing branch b into channels [off_b, off_b + C).
// The grad-input of the concatenation is the sum of the branches'
// grad-inputs; it is computed in one launch from the branches' grad_out
// slices, summed in fp32 and rounded once. Both kernels are persistent and
// stage their next tile with cp.async while computing the current one.
#include "plan.h"
#include "tile.cuh"

namespace dwconv {
namespace tile {
namespace {

constexpr int kR = 2, kV = 4;

struct MultiArgs {
  int nb;
  int oy[3], ox[3];           // per-branch offset of tap (0,0) in the tile
  int dl[3];                  // window offset inside the 4-aligned read (dilation-1 windows)
  int rb[3], cb[3];           // fwd: item grid per branch
  int items[3];               // fwd: items per plane per branch
  int64_t off[3];             // channel offset of each branch slice
  const void* w[3];
  const void* bias[3];
  int tr[3], tile_elems[3];   // bwd: per-branch tiles
  int iy0[3], ix0[3], mode[3];  // tile origins relative to the band, copy modes
  FastDiv trdiv[3];
  FastDiv d_prb[3], d_cbq[3];   // fwd: division by items per row block, by cb * Q
};

struct MCfg {
  int ppc, th, nbands, tr, pitch, rb, cb, tile_elems, stage_elems, vec_out, mode, ix0;
  int64_t groups;
  FastDiv trdiv, d_bands, d_item, d_cb;
};

// Window-offset dispatch: conv_block needs its offset at compile time.
template <int K, int D, int Q, typename TS>
__device__ __forceinline__ void conv_dl(int dl, const TS* t, int pitch, int tr0, int tc0,
                                        const float (&wr)[K * K], float (&acc)[kR][kV]) {
  if (Q > 1) {
    conv_block<K, 1, D, kR, kV, Q, 0>(t, pitch, tr0, tc0 + dl, wr, acc);
    return;
  }
  switch (dl) {
    case 0: conv_block<K, 1, D, kR, kV, 1, 0>(t, pitch, tr0, tc0, wr, acc); break;
    case 1: conv_block<K, 1, D, kR, kV, 1, 1>(t, pitch, tr0, tc0, wr, acc); break;
    case 2: conv_block<K, 1, D, kR, kV, 1, 2>(t, pitch, tr0, tc0, wr, acc); break;
    default: conv_block<K, 1, D, kR, kV, 1, 3>(t, pitch, tr0, tc0, wr, acc); break;
  }
}

// One R x V output block of branch b (filter wr, bias bv already in
// registers): item -> (row block, row phase, column block, column phase).
template <int K, int D, typename T>
__device__ __forceinline__ void fwd_branch(const Conv& c, const MultiArgs& a, int b, const T* t, int pitch,
                                           int item, int64_t n, int64_t ch, int oh0, int band_rows,
                                           const float (&wr)[K * K], float bv, T* y) {
  constexpr int Q = D;
  uint32_t rbi_, qy_;
  uint32_t rem = a.d_prb[b].divmod((uint32_t)item, rbi_);
  rem = a.d_cbq[b].divmod(rem, qy_);
  const int cbi = (int)rem / Q;
  const int qx = (int)rem - cbi * Q;
  float acc[kR][kV];
#pragma unroll
  for (int r = 0; r < kR; ++r)
#pragma unroll
    for (int v = 0; v < kV; ++v) acc[r][v] = bv;
  const int ohr = (int)rbi_ * Q * kR + (int)qy_;
  const int owb = cbi * Q * kV + qx;
  conv_dl<K, D, Q>(a.dl[b], t, pitch, ohr + a.oy[b], owb + a.ox[b], wr, acc);
  const bool vec = Q == 1 && c.Wo % 4 == 0 &&
                   (reinterpret_cast<uintptr_t>(y) % (4 * sizeof(T))) == 0;
  store_block<T, kR, kV, Q>(y + (n * c.ctot + a.off[b] + ch) * c.Ho * c.Wo, c.Wo, oh0 + ohr, owb,
                            band_rows - ohr, (int)c.Wo, acc, vec, false);
}

template <int K, typename T>
__device__ __forceinline__ void load_filter(const T* w, const T* bias, int64_t ch, float (&wr)[K * K], float& bv) {
#pragma unroll
  for (int i = 0; i < K * K; ++i) wr[i] = ld(w + ch * (K * K) + i);
  bv = bias ? ld(bias + ch) : 0.f;
}

template <typename T, int K, int NB, int D0, int D1, int D2>
__global__ void __launch_bounds__(kNT)
fwd_multi_kernel(Conv c, MCfg g, MultiArgs a, const T* __restrict__ x, T* __restrict__ y) {
  extern __shared__ __align__(16) unsigned char smraw[];
  T* buf[2] = {reinterpret_cast<T*>(smraw), reinterpret_cast<T*>(smraw) + g.stage_elems};
  const int64_t nplanes = c.N * c.C;
  const int64_t units = g.groups * g.nbands;
  const int64_t HW = c.H * c.W;
  auto issue = [&](int64_t u, T* dst) {
    uint32_t grp;
    const int band = (int)g.d_bands.divmod((uint32_t)u, grp);
    const int64_t p0 = (int64_t)grp * g.ppc;
    const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
    issue_tile<T>(dst, np, g.tile_elems, g.pitch, [&](int p) { return x + (p0 + p) * HW; }, (int)c.H,
                  (int)c.W, band * g.th + a.iy0[0], g.tr, g.trdiv, g.ix0, g.mode);
  };
  int64_t u = blockIdx.x;
  if (u < units) issue(u, buf[0]);
  cp_async_commit();
  const int i0 = a.items[0], i1 = a.items[1], i2 = NB > 2 ? a.items[2] : 0;
  const int per_plane = i0 + i1 + i2;
  for (int k = 0; u < units; ++k, u += gridDim.x) {
    const T* cur = buf[k & 1];
    if (u + gridDim.x < units) issue(u + gridDim.x, buf[(k + 1) & 1]);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    uint32_t grp;
    const int band = (int)g.d_bands.divmod((uint32_t)u, grp);
    const int64_t p0 = (int64_t)grp * g.ppc;
    const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
    const int oh0 = band * g.th;
    const int band_rows = (int)((c.Ho - oh0) < g.th ? (c.Ho - oh0) : g.th);
    // A thread's items run through the planes and, within a plane, through
    // the branches in order: each branch's filter is loaded once per plane.
    int curp = -1, have = 0;
    int64_t n = 0, ch = 0;
    float w0[K * K], w1[K * K], w2[K * K], b0 = 0.f, b1 = 0.f, b2 = 0.f;
    for (int it = threadIdx.x; it < np * per_plane; it += kNT) {
      const int pl = it / per_plane;
      const int q = it - pl * per_plane;
      if (pl != curp) {
        curp = pl;
        have = 0;
        c.split(p0 + pl, n, ch);
      }
      const T* t = cur + pl * g.tile_elems;
      if (q < i0) {
        if (!(have & 1)) load_filter<K>((const T*)a.w[0], (const T*)a.bias[0], ch, w0, b0), have |= 1;
        fwd_branch<K, D0>(c, a, 0, t, g.pitch, q, n, ch, oh0, band_rows, w0, b0, y);
      } else if (q < i0 + i1) {
        if (!(have & 2)) load_filter<K>((const T*)a.w[1], (const T*)a.bias[1], ch, w1, b1), have |= 2;
        fwd_branch<K, D1>(c, a, 1, t, g.pitch, q - i0, n, ch, oh0, band_rows, w1, b1, y);
      } else if (NB > 2) {
        if (!(have & 4)) load_filter<K>((const T*)a.w[2], (const T*)a.bias[2], ch, w2, b2), have |= 4;
        fwd_branch<K, (NB > 2 ? D2 : 1)>(c, a, 2, t, g.pitch, q - i0 - i1, n, ch, oh0, band_rows, w2, b2, y);
      }
    }
    __syncthreads();
  }
}

template <typename T, int K, int NB, int D0, int D1, int D2>
__global__ void __launch_bounds__(kNT)
bwd_multi_kernel(Conv c, MCfg g, MultiArgs a, const T* __restrict__ gy, T* gx) {
  extern __shared__ __align__(16) unsigned char smraw[];
  T* buf[2] = {reinterpret_cast<T*>(smraw), reinterpret_cast<T*>(smraw) + g.stage_elems};
  const int64_t nplanes = c.N * c.C;
  const int64_t units = g.groups * g.nbands;
  const int slice = a.tile_elems[0] + a.tile_elems[1] + (NB > 2 ? a.tile_elems[2] : 0);
  auto issue = [&](int64_t u, T* dst) {
    uint32_t grp;
    const int band = (int)g.d_bands.divmod((uint32_t)u, grp);
    const int64_t p0 = (int64_t)grp * g.ppc;
    const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const int boff = b == 0 ? 0 : (b == 1 ? a.tile_elems[0] : a.tile_elems[0] + a.tile_elems[1]);
      issue_tile<T>(dst + boff, np, slice, g.pitch,
                    [&](int p) {
                      int64_t n, ch;
                      c.split(p0 + p, n, ch);
                      return gy + (n * c.ctot + a.off[b] + ch) * c.Ho * c.Wo;
                    },
                    (int)c.Ho, (int)c.Wo, band * g.th + a.iy0[b], a.tr[b], a.trdiv[b], a.ix0[b],
                    a.mode[b]);
    }
  };
  int64_t u = blockIdx.x;
  if (u < units) issue(u, buf[0]);
  cp_async_commit();
  for (int k = 0; u < units; ++k, u += gridDim.x) {
    const T* cur = buf[k & 1];
    if (u + gridDim.x < units) issue(u + gridDim.x, buf[(k + 1) & 1]);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    uint32_t grp;
    const int band = (int)g.d_bands.divmod((uint32_t)u, grp);
    const int64_t p0 = (int64_t)grp * g.ppc;
    const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
    const int ih0 = band * g.th;
    const int band_rows = (int)((c.H - ih0) < g.th ? (c.H - ih0) : g.th);
    int curp = -1;
    float w0[K * K], w1[K * K], w2[K * K];
    for (int it = threadIdx.x; it < np * (int)g.d_item.d; it += kNT) {
      uint32_t pl_, rbi_;
      const uint32_t rem = g.d_item.divmod((uint32_t)it, pl_);
      const int cbi = (int)g.d_cb.divmod(rem, rbi_);
      const int pl = (int)pl_, rbi = (int)rbi_;
      const int64_t pin = p0 + pl;
      int64_t n_, ch;
      c.split(pin, n_, ch);
      if (pl != curp) {
        curp = pl;
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
      const T* t = cur + pl * slice;
      conv_dl<K, D0, 1>(a.dl[0], t, g.pitch, ihr, iwb + a.ox[0], w0, acc);
      conv_dl<K, D1, 1>(a.dl[1], t + a.tile_elems[0], g.pitch, ihr, iwb + a.ox[1], w1, acc);
      if (NB > 2)
        conv_dl<K, (NB > 2 ? D2 : 1), 1>(a.dl[2], t + a.tile_elems[0] + a.tile_elems[1], g.pitch, ihr,
                                         iwb + a.ox[2], w2, acc);
      store_block<T, kR, kV, 1>(gx + pin * c.H * c.W, c.W, ih0 + ihr, iwb, band_rows - ihr, (int)c.W,
                                acc, g.vec_out, false);
    }
    __syncthreads();
  }
}

int lcm(int a, int b) {
  int x = a, y = b;
  while (y) { const int t = x % y; x = y; y = t; }
  return a / x * b;
}

template <typename T, int K, int NB, int D0, int D1, int D2>
cudaError_t run_fwd_multi(const Conv* cs, const void* x, const void* const* w, const void* const* bias,
                          void* y, cudaStream_t s) {
  constexpr int ES = sizeof(T);
  constexpr int PA = 16 / ES > 4 ? 16 / ES : 4;
  const Conv& c = cs[0];
  const int Ds[3] = {D0, D1, D2};
  MultiArgs a{};
  a.nb = NB;
  int hh = 0, hw = 0;
  for (int b = 0; b < NB; ++b) {
    hh = cs[b].ph > hh ? cs[b].ph : hh;
    hw = cs[b].pw > hw ? cs[b].pw : hw;
    a.off[b] = cs[b].off;
    a.w[b] = w[b];
    a.bias[b] = bias ? bias[b] : nullptr;
  }
  MCfg g{};
  int shift = 0;
  g.mode = pick_mode<T>(x, c.W, -hw, &g.ix0, &shift);
  int L = 1;
  int64_t need = 0;
  for (int b = 0; b < NB; ++b) {
    L = lcm(L, Ds[b] * kR);
    a.oy[b] = hh - cs[b].ph;
    const int off = hw - cs[b].pw + shift;  // tile column of branch b's tap-(0,0) for output col 0
    const int Q = Ds[b];
    a.cb[b] = (int)((c.Wo + (int64_t)Q * kV - 1) / ((int64_t)Q * kV));
    const int WN = (kV - 1) * Q + (K - 1) * Ds[b] + 1;
    int64_t rc;
    if (Q == 1) {
      a.dl[b] = off % 4;
      a.ox[b] = off - a.dl[b];
      rc = (int64_t)(a.cb[b] - 1) * kV + a.ox[b] + (a.dl[b] + WN + 3) / 4 * 4;
    } else {
      a.dl[b] = off;  // scalar windows: the whole offset is added to the start column
      a.ox[b] = 0;
      rc = (int64_t)(a.cb[b] - 1) * Q * kV + Q - 1 + off + WN;
    }
    if (rc > need) need = rc;
  }
  g.pitch = round_up(need, PA);
  auto tr_of = [&](int64_t th) {
    int64_t t = 0;
    for (int b = 0; b < NB; ++b) {
      const int64_t r = th - 1 + a.oy[b] + (int64_t)(K - 1) * Ds[b] + 1;
      if (r > t) t = r;
    }
    return t;
  };
  const int64_t target = 32 * 1024;
  int64_t th = (c.Ho + L - 1) / L * L;
  while (th > L && tr_of(th) * g.pitch * ES > target) th -= L;
  if (tr_of(th) * g.pitch * ES > 96 * 1024) return cudaErrorInvalidConfiguration;
  g.th = (int)th;
  g.nbands = (int)((c.Ho + th - 1) / th);
  g.tr = (int)tr_of(th);
  g.tile_elems = g.tr * g.pitch;
  int64_t items = 0;
  for (int b = 0; b < NB; ++b) {
    a.rb[b] = (int)(th / (Ds[b] * kR));
    a.items[b] = a.rb[b] * a.cb[b] * Ds[b] * Ds[b];
    a.d_prb[b] = FastDiv((uint32_t)(a.cb[b] * Ds[b] * Ds[b]));
    a.d_cbq[b] = FastDiv((uint32_t)(a.cb[b] * Ds[b]));
    items += a.items[b];
  }
  a.iy0[0] = -hh;
  const int64_t nplanes = c.N * c.C;
  int64_t ppc = 1;
  if (g.nbands == 1) {
    ppc = (2 * kNT + items - 1) / items;
    const int64_t cap = target / ((int64_t)g.tile_elems * ES);
    if (ppc > cap) ppc = cap;
    if (ppc < 1) ppc = 1;
  }
  g.ppc = (int)ppc;
  g.groups = (nplanes + ppc - 1) / ppc;
  g.stage_elems = g.ppc * g.tile_elems;
  g.trdiv = FastDiv((uint32_t)g.tr);
  g.d_bands = FastDiv((uint32_t)g.nbands);
  const size_t smem = 2 * (size_t)g.stage_elems * ES;
  auto kern = fwd_multi_kernel<T, K, NB, D0, D1, D2>;
  cudaError_t err = set_smem(kern, smem);
  if (err != cudaSuccess) return err;
  const int grid = persistent_grid(kern, smem, g.groups * g.nbands);
  kern<<<grid, kNT, smem, s>>>(c, g, a, (const T*)x, (T*)y);
  return cudaGetLastError();
}

template <typename T, int K, int NB, int D0, int D1, int D2>
cudaError_t run_bwd_multi(const Conv* cs, const void* gy, const void* const* w, void* gx,
                          cudaStream_t s) {
  constexpr int ES = sizeof(T);
  constexpr int PA = 16 / ES > 4 ? 16 / ES : 4;
  const Conv& c = cs[0];
  const int Ds[3] = {D0, D1, D2};
  MultiArgs a{};
  a.nb = NB;
  MCfg g{};
  g.cb = (int)((c.W + kV - 1) / kV);
  int64_t need = 0;
  for (int b = 0; b < NB; ++b) {
    const int qh = Ds[b] * (K - 1) - cs[b].ph, qw = Ds[b] * (K - 1) - cs[b].pw;
    if (qh < 0 || qw < 0) return cudaErrorInvalidConfiguration;
    a.off[b] = cs[b].off;
    a.w[b] = w[b];
    a.iy0[b] = -qh;
    int shift = 0;
    a.mode[b] = pick_mode<T>(gy, c.Wo, -qw, &a.ix0[b], &shift);
    a.dl[b] = shift % 4;
    a.ox[b] = shift - a.dl[b];
    const int WN = (kV - 1) + (K - 1) * Ds[b] + 1;
    const int64_t rc = (int64_t)(g.cb - 1) * kV + a.ox[b] + (a.dl[b] + WN + 3) / 4 * 4;
    if (rc > need) need = rc;
  }
  g.pitch = round_up(need, PA);
  auto bytes_of = [&](int64_t th) {
    int64_t t = 0;
    for (int b = 0; b < NB; ++b) t += (th - 1 + (int64_t)(K - 1) * Ds[b] + 1) * g.pitch;
    return t * ES;
  };
  const int64_t target = 32 * 1024;
  int64_t th = (c.H + kR - 1) / kR * kR;
  while (th > kR && bytes_of(th) > target) th -= kR;
  if (bytes_of(th) > 96 * 1024) return cudaErrorInvalidConfiguration;
  g.th = (int)th;
  g.rb = (int)(th / kR);
  g.nbands = (int)((c.H + th - 1) / th);
  for (int b = 0; b < NB; ++b) {
    a.tr[b] = (int)(th - 1 + (int64_t)(K - 1) * Ds[b] + 1);
    a.tile_elems[b] = a.tr[b] * g.pitch;
    a.trdiv[b] = FastDiv((uint32_t)a.tr[b]);
  }
  const int64_t slice_bytes = bytes_of(th);
  const int64_t items = (int64_t)g.rb * g.cb;
  const int64_t nplanes = c.N * c.C;
  int64_t ppc = 1;
  if (g.nbands == 1) {
    ppc = (2 * kNT + items - 1) / items;
    const int64_t cap = target / slice_bytes;
    if (ppc > cap) ppc = cap;
    if (ppc < 1) ppc = 1;
  }
  g.ppc = (int)ppc;
  g.groups = (nplanes + ppc - 1) / ppc;
  g.stage_elems = (int)(g.ppc * slice_bytes / ES);
  g.vec_out = c.W % 4 == 0 && (reinterpret_cast<uintptr_t>(gx) % (4 * ES)) == 0;
  g.d_bands = FastDiv((uint32_t)g.nbands);
  g.d_item = FastDiv((uint32_t)(g.rb * g.cb));
  g.d_cb = FastDiv((uint32_t)g.cb);
  const size_t smem = 2 * (size_t)g.stage_elems * ES;
  auto kern = bwd_multi_kernel<T, K, NB, D0, D1, D2>;
  cudaError_t err = set_smem(kern, smem);
  if (err != cudaSuccess) return err;
  const int grid = persistent_grid(kern, smem, g.groups * g.nbands);
  kern<<<grid, kNT, smem, s>>>(c, g, a, (const T*)gy, (T*)gx);
  return cudaGetLastError();
}

// Dilation sets compiled for the fused path (3x3 filters; the first branch
// has dilation 1).
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

// The fused planners' narrowest bands must fit their 96 KB limit: the
// forward's has L rows (L the lcm of the branches' d*kR), the grad-input's
// kR rows per branch. Both follow the planners' arithmetic with the widest
// row pitch any pointer alignment gives (a shift of at most one 16-byte
// chunk), so a shape that passes always plans.
bool multi_fits(int nb, const Conv* cs) {
  const int64_t K = cs[0].kh, es = cs[0].dtype == DWCONV_F32 ? 4 : 2;
  const int64_t smax = 16 / es - 1, PA = 16 / es > 4 ? 16 / es : 4;
  auto rup = [](int64_t v, int64_t a) { return (v + a - 1) / a * a; };
  int64_t hh = 0, hw = 0;
  int L = 1;
  for (int b = 0; b < nb; ++b) {
    hh = cs[b].ph > hh ? cs[b].ph : hh;
    hw = cs[b].pw > hw ? cs[b].pw : hw;
    L = lcm(L, cs[b].dh * kR);
  }
  int64_t need = 0, tr = 0;
  for (int b = 0; b < nb; ++b) {
    const int64_t Q = cs[b].dh, D = cs[b].dh;
    const int64_t cb = (cs[0].Wo + Q * kV - 1) / (Q * kV);
    const int64_t WN = (kV - 1) * Q + (K - 1) * D + 1;
    const int64_t off = hw - cs[b].pw + smax;
    const int64_t rc = Q == 1 ? (cb - 1) * kV + off + WN + 3 : (cb - 1) * Q * kV + Q - 1 + off + WN;
    if (rc > need) need = rc;
    const int64_t r = L - 1 + (hh - cs[b].ph) + (K - 1) * D + 1;
    if (r > tr) tr = r;
  }
  if (tr * rup(need, PA) * es > 96 * 1024) return false;
  const int64_t cb = (cs[0].W + kV - 1) / kV;
  int64_t rows = 0;
  need = 0;
  for (int b = 0; b < nb; ++b) {
    const int64_t D = cs[b].dh;
    const int64_t rc = (cb - 1) * kV + smax + (kV - 1) + (K - 1) * D + 1 + 3;
    if (rc > need) need = rc;
    rows += kR - 1 + (K - 1) * D + 1;
  }
  return rows * rup(need, PA) * es <= 96 * 1024;
}

bool multi_supported(int nb, const Conv* cs) {
  if (!same_geometry(nb, cs) || !cs[0].planes32()) return false;
  for (int b = 0; b < nb; ++b) {
    if (cs[b].kh != cs[0].kh) return false;
    // the fused grad-input needs non-negative transposed padding
    if (cs[b].ph > cs[b].dh * (cs[b].kh - 1) || cs[b].pw > cs[b].dw * (cs[b].kw - 1)) return false;
  }
  if (!multi_fits(nb, cs)) return false;
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
