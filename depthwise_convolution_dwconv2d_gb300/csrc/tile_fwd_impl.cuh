// Implementation of the small-kernel depthwise forward and stride-1 grad-input on shared-memory
// tiles (square filters K <= 7, equal stride and dilation on both axes).
//
// Forward: y[n, off + c*m + j] = b + sum_{a,b} w[c*m+j, a, b] x[n, c, oh*S - ph + a*D, ow*S - pw + b*D]
// ("Spatial Depthwise Convolution on the GPU #3057", forward kernel with
// padding, stride, dilation, multiplier and bias).
// Grad-input at stride 1 is the same stencil run on grad_out with the filter
// rotated by 180 degrees and padding D*(K-1) - pad, summed over the m output
// channels of each input channel (the adjoint of the forward; #3057's
// grad-input kernel).
//
// Both kernels are persistent: a CTA walks work units (a group of channel
// planes x a band of output rows) with a stride of gridDim.x, staging unit
// k+1 with cp.async while it computes unit k.
#pragma once
#include "plan.h"
#include "tile_cases.h"
#include "tile_plan.cuh"
#include "tma.cuh"
#include "tile.cuh"
#include "tile_plan.cuh"

namespace dwconv {
namespace tile {
namespace {

template <typename T, int K, int S, int D, int R, int V, int DL>
__global__ void __launch_bounds__(kNT)
fwd_kernel(Conv c, Cfg g, const __grid_constant__ CUtensorMap tmap, unsigned int* timeouts,
           const T* __restrict__ x, const T* __restrict__ w, const T* __restrict__ bias,
           T* __restrict__ y, Epi ep) {
  extern __shared__ __align__(16) unsigned char smdyn[];
  __shared__ __align__(8) uint64_t bars[2];
  constexpr int Q = Geo<K, S, D>::Q;
  unsigned char* smraw = smdyn + ((128 - (tma::smem_u32(smdyn) & 127)) & 127);
  const bool use_tma = g.mode == kCopyTMA;
  if (use_tma && threadIdx.x == 0) {
    tma::mbar_init(&bars[0], 1);
    tma::mbar_init(&bars[1], 1);
    tma::fence_init();
  }
  __syncthreads();
  T* const buf0 = reinterpret_cast<T*>(smraw);
  T* const buf1 = buf0 + g.stage_elems;
  T* const stg0 = buf1 + g.stage_elems;  // dense staging (empty unless kCopyDense)
  T* const stg1 = stg0 + g.stg_elems;
  // per stage: filter taps, bias and output-plane offset of each output plane
  float* const tab0 = reinterpret_cast<float*>(stg1 + g.stg_elems);
  float* const tab1 = tab0 + g.tab_floats;
  const int64_t nplanes = c.N * c.C;
  const int64_t units = g.groups * g.nbands;
  const int64_t HW = c.H * c.W;
  const int nout = g.ppc * c.m;  // output planes per full unit
  auto issue = [&](int64_t p0, int np, int band, T* dst, T* stg, float* tab, uint64_t* bar) {
    if (use_tma) {
      if (threadIdx.x == 0) {
        tma::fence_async_smem();
        tma::mbar_expect_tx(bar, g.tma_bytes);
        tma::load_3d(dst, &tmap, g.ix0, band * g.th * S - c.ph, (int)p0, bar);
      }
    } else if (g.mode == kCopyDense) {
      if (g.contig)
        issue_contig<T>(stg, x + p0 * HW, np * HW);
      else
        issue_flat<T>(stg, np, g.seg, [&](int p) { return x + (p0 + p) * HW; }, (int)HW);
    } else {
      issue_tile<T>(dst, np, g.tile_elems, g.pitch, [&](int p) { return x + (p0 + p) * HW; },
                    (int)c.H, (int)c.W, band * g.th * S - c.ph, g.tr, g.trdiv, g.ix0, g.mode);
    }
    float* wt = tab;
    float* bt = tab + nout * (K * K);
    float* st = bt + nout;  // epilogue scale and shift (when one is fused)
    float* ht = st + nout;
    int64_t* ot = reinterpret_cast<int64_t*>(tab + g.tab_off64);
    // one output plane per thread: its taps, bias, epilogue and output offset
    for (int pj = threadIdx.x; pj < np * c.m; pj += kNT) {
      const int pl = c.m == 1 ? pj : pj / c.m;
      int64_t n, ch;
      c.split(p0 + pl, n, ch);
      const int64_t oc = ch * c.m + (pj - pl * c.m);
      const T* wp = w + oc * (K * K);
#pragma unroll
      for (int tap = 0; tap < K * K; ++tap) tab_put(wt + pj * (K * K) + tap, wp + tap);
      if (bias) tab_put(bt + pj, bias + oc);
      else bt[pj] = 0.f;
      if (ep.active()) {
        if (ep.scale) tab_put(st + pj, reinterpret_cast<const T*>(ep.scale) + oc);
        else st[pj] = 1.f;
        if (ep.shift) tab_put(ht + pj, reinterpret_cast<const T*>(ep.shift) + oc);
        else ht[pj] = 0.f;
      }
      ot[pj] = c.y_base(n, oc);
    }
  };
  const Sched sch(nplanes, units, g.ppc, g.balanced, g.d_bands);
  int64_t p0n;
  int npn, bandn;
  bool have = sch.stage(0, p0n, npn, bandn);
  if (have) issue(p0n, npn, bandn, buf0, stg0, tab0, &bars[0]);
  cp_async_commit();
  for (int k = 0; have; ++k) {
    const int64_t p0 = p0n;
    const int np = npn, band = bandn;
    T* cur = (k & 1) ? buf1 : buf0;
    const float* tab = (k & 1) ? tab1 : tab0;
    const bool more = sch.stage(k + 1, p0n, npn, bandn);
    if (more) issue(p0n, npn, bandn, (k & 1) ? buf0 : buf1, (k & 1) ? stg0 : stg1, (k & 1) ? tab0 : tab1,
                    &bars[(k + 1) & 1]);
    cp_async_commit();
    cp_async_wait<1>();
    if (use_tma && !tma::mbar_wait(&bars[k & 1], (uint32_t)(k >> 1) & 1, timeouts)) {
      // the copy never landed: let the one in flight finish (bounded), then stop
      if (more) tma::mbar_wait(&bars[(k + 1) & 1], (uint32_t)((k + 1) >> 1) & 1, nullptr);
      return;
    }
    __syncthreads();
    const T* stg = (k & 1) ? stg1 : stg0;
    const int oh0 = band * g.th;
    const int band_rows = (int)((c.Ho - oh0) < g.th ? (c.Ho - oh0) : g.th);
    const float* wt = tab;
    const float* bt = tab + nout * (K * K);
    const int64_t* ot = reinterpret_cast<const int64_t*>(tab + g.tab_off64);
    const int total = np * c.m * (int)g.d_item.d;
    for (int it = threadIdx.x; it < total; it += kNT) {
      uint32_t pj_, rbi_, qy_;
      uint32_t rem = g.d_item.divmod((uint32_t)it, pj_);
      rem = g.d_rb.divmod(rem, rbi_);
      rem = g.d_cbq.divmod(rem, qy_);
      const int pj = (int)pj_, rbi = (int)rbi_, qy = (int)qy_;
      const int cbi = (int)rem / Q;
      const int qx = (int)rem - cbi * Q;
      const int ohr = rbi * Q * R + qy;
      const int owb = cbi * Q * V + qx;
      float wr[K * K];
#pragma unroll
      for (int i = 0; i < K * K; ++i) wr[i] = wt[pj * (K * K) + i];
      const float bv = bt[pj];
      float acc[R][V];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < V; ++v) acc[r][v] = bv;
      if (g.mode == kCopyDense) {
        const int pl = pj / c.m;
        const T* dp = g.contig ? dense_at(stg, x + p0 * HW, pl * (int)HW)
                               : dense_plane(stg, g.seg, pl, x + (p0 + pl) * HW);
        conv_block_dense<K, S, D, R, V, Q>(dp, (int)c.H, (int)c.W,
                                           ohr * S - c.ph, owb * S - c.pw, wr, acc);
      } else {
        conv_block<K, S, D, R, V, Q, DL>(cur + (pj / c.m) * g.tile_elems, g.pitch, ohr * S, owb * S + g.cshift, wr, acc);
      }
      if (ep.active()) {
        const float sc = bt[nout + pj], sh = bt[2 * nout + pj];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int v = 0; v < V; ++v) acc[r][v] = epi_act(fmaf(acc[r][v], sc, sh), ep.act);
      }
      store_block<T, R, V, Q>(y + ot[pj], c.Wo, oh0 + ohr, owb, band_rows - ohr, (int)c.Wo, acc,
                              g.vec_out, false);
    }
    __syncthreads();
    have = more;
  }
}

// Stride-1 grad-input: gx[n, c] = sum_j corr(gy[n, off + c*m + j], rot180(w[c*m + j])).
template <typename T, int K, int D, int R, int V, int DL>
__global__ void __launch_bounds__(kNT)
bwd1_kernel(Conv c, Cfg g, const __grid_constant__ CUtensorMap tmap, unsigned int* timeouts, int qh,
            const T* __restrict__ gy, const T* __restrict__ w, T* gx, bool accumulate) {
  extern __shared__ __align__(16) unsigned char smdyn[];
  __shared__ __align__(8) uint64_t bars[2];
  constexpr int Q = Geo<K, 1, D>::Q;
  unsigned char* smraw = smdyn + ((128 - (tma::smem_u32(smdyn) & 127)) & 127);
  const bool use_tma = g.mode == kCopyTMA;
  if (use_tma && threadIdx.x == 0) {
    tma::mbar_init(&bars[0], 1);
    tma::mbar_init(&bars[1], 1);
    tma::fence_init();
  }
  __syncthreads();
  T* const buf0 = reinterpret_cast<T*>(smraw);
  T* const buf1 = buf0 + g.stage_elems;
  T* const stg0 = buf1 + g.stage_elems;  // dense staging (empty unless kCopyDense)
  T* const stg1 = stg0 + g.stg_elems;
  // per stage: rotated filters of each (gx plane, j) and each gx plane's offset
  float* const tab0 = reinterpret_cast<float*>(stg1 + g.stg_elems);
  float* const tab1 = tab0 + g.tab_floats;
  const int64_t nplanes = c.N * c.C;
  const int64_t units = g.groups * g.nbands;
  const int m = c.m;
  auto gy_plane = [&](int64_t p0, int s) {
    const int pl = m == 1 ? s : s / m, j = s - pl * m;
    int64_t n, ch;
    c.split(p0 + pl, n, ch);
    return gy + c.y_base(n, ch * m + j);
  };
  auto issue = [&](int64_t p0, int np, int band, T* dst, T* stg, float* tab, uint64_t* bar) {
    // staged plane s = pl * m + j holds gy[n, off + c*m + j]
    if (g.mode == kCopyDense) {
      if (g.contig)
        issue_contig<T>(stg, gy_plane(p0, 0), (int64_t)np * m * c.Ho * c.Wo);
      else
        issue_flat<T>(stg, np * m, g.seg, [&](int s) { return gy_plane(p0, s); }, (int)(c.Ho * c.Wo));
    } else if (use_tma) {
      if (threadIdx.x == 0) {
        int64_t n, ch;
        c.split(p0, n, ch);  // units never straddle samples
        tma::fence_async_smem();
        tma::mbar_expect_tx(bar, g.tma_bytes);
        tma::load_3d(dst, &tmap, g.ix0, band * g.th - qh, (int)(n * c.ctot + c.off + ch * m), bar);
      }
    } else {
      issue_tile<T>(dst, np * m, g.tile_elems, g.pitch,
                    [&](int s) { return gy_plane(p0, s); },
                    (int)c.Ho, (int)c.Wo, band * g.th - qh, g.tr, g.trdiv, g.ix0, g.mode);
    }
    int64_t* ot = reinterpret_cast<int64_t*>(tab + g.tab_off64);
    // one staged plane per thread: its rotated filter
    for (int s = threadIdx.x; s < np * m; s += kNT) {
      const int pl = m == 1 ? s : s / m;
      int64_t n, ch;
      c.split(p0 + pl, n, ch);
      const T* wp = w + (ch * m + (s - pl * m)) * (K * K);
#pragma unroll
      for (int tap = 0; tap < K * K; ++tap) tab_put(tab + s * (K * K) + tap, wp + (K * K - 1 - tap));
    }
    for (int pl = threadIdx.x; pl < np; pl += kNT) ot[pl] = (p0 + pl) * c.H * c.W;
  };
  const Sched sch(nplanes, units, g.ppc, g.balanced, g.d_bands);
  int64_t p0n;
  int npn, bandn;
  bool have = sch.stage(0, p0n, npn, bandn);
  if (have) issue(p0n, npn, bandn, buf0, stg0, tab0, &bars[0]);
  cp_async_commit();
  for (int k = 0; have; ++k) {
    const int64_t p0 = p0n;
    const int np = npn, band = bandn;
    T* cur = (k & 1) ? buf1 : buf0;
    const float* tab = (k & 1) ? tab1 : tab0;
    const bool more = sch.stage(k + 1, p0n, npn, bandn);
    if (more) issue(p0n, npn, bandn, (k & 1) ? buf0 : buf1, (k & 1) ? stg0 : stg1, (k & 1) ? tab0 : tab1,
                    &bars[(k + 1) & 1]);
    cp_async_commit();
    cp_async_wait<1>();
    if (use_tma && !tma::mbar_wait(&bars[k & 1], (uint32_t)(k >> 1) & 1, timeouts)) {
      if (more) tma::mbar_wait(&bars[(k + 1) & 1], (uint32_t)((k + 1) >> 1) & 1, nullptr);
      return;
    }
    __syncthreads();
    const T* stg = (k & 1) ? stg1 : stg0;
    const int ih0 = band * g.th;
    const int band_rows = (int)((c.H - ih0) < g.th ? (c.H - ih0) : g.th);
    const int64_t* ot = reinterpret_cast<const int64_t*>(tab + g.tab_off64);
    const int total = np * (int)g.d_item.d;
    for (int it = threadIdx.x; it < total; it += kNT) {
      uint32_t pl_, rbi_, qy_;
      uint32_t rem = g.d_item.divmod((uint32_t)it, pl_);
      rem = g.d_rb.divmod(rem, rbi_);
      rem = g.d_cbq.divmod(rem, qy_);
      const int pl = (int)pl_, rbi = (int)rbi_, qy = (int)qy_;
      const int cbi = (int)rem / Q;
      const int qx = (int)rem - cbi * Q;
      const int ihr = rbi * Q * R + qy;
      const int iwb = cbi * Q * V + qx;
      float acc[R][V];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < V; ++v) acc[r][v] = 0.f;
      for (int j = 0; j < m; ++j) {
        float wr[K * K];
#pragma unroll
        for (int i = 0; i < K * K; ++i) wr[i] = tab[(pl * m + j) * (K * K) + i];
        if (g.mode == kCopyDense) {
          const int sp = pl * m + j;
          const T* dp = g.contig ? dense_at(stg, gy_plane(p0, 0), sp * (int)(c.Ho * c.Wo))
                                 : dense_plane(stg, g.seg, sp, gy_plane(p0, sp));
          conv_block_dense<K, 1, D, R, V, Q>(dp, (int)c.Ho,
                                             (int)c.Wo, ihr - qh, iwb - (D * (K - 1) - c.pw), wr, acc);
        } else {
          conv_block<K, 1, D, R, V, Q, DL>(cur + (pl * m + j) * g.tile_elems, g.pitch, ihr, iwb + g.cshift, wr, acc);
        }
      }
      store_block<T, R, V, Q>(gx + ot[pl], c.W, ih0 + ihr, iwb, band_rows - ihr, (int)c.W, acc,
                              g.vec_out, accumulate);
    }
    __syncthreads();
    have = more;
  }
}

// Register-block shape per (K, S): R rows x V cols of outputs per thread.
template <int K, int S> struct Blk { static constexpr int R = S == 1 ? 4 : 2, V = 4; };

template <typename T, int K, int S, int D, int DL>
cudaError_t launch_fwd(const Conv& c, const Cfg& g, const CUtensorMap& map, const void* x, const void* w,
                       const void* b, void* y, cudaStream_t s, const Epi& ep) {
  constexpr int R = Blk<K, S>::R, V = Blk<K, S>::V;
  auto kern = fwd_kernel<T, K, S, D, R, V, DL>;
  const size_t smem = 128 + 2 * ((size_t)g.stage_elems + g.stg_elems) * sizeof(T) + 2 * (size_t)g.tab_floats * 4;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = persistent_grid(kern, smem, g.groups * g.nbands);
  kern<<<grid, kNT, smem, s>>>(c, g, map, tma::timeout_counter(), (const T*)x, (const T*)w, (const T*)b, (T*)y,
                               ep);
  return cudaGetLastError();
}

template <typename T, int K, int S, int D>
cudaError_t run_fwd_t(const Conv& c, const void* x, const void* w, const void* b, void* y,
                      cudaStream_t s, const Epi& ep) {
  constexpr int R = Blk<K, S>::R, V = Blk<K, S>::V, Q = Geo<K, S, D>::Q;
  const bool vout = Q == 1 && c.Wo % 4 == 0 && alignedn(y, 4 * sizeof(T));
  Cfg g;
  int dl = 0;
  alignas(64) CUtensorMap map{};
  if (!plan_tile<T, K, S, D, R, V>(c.N * c.C, 1, c.m, c.H, c.W, c.Ho, c.Wo, c.pw, x, vout, &g, &dl, 0,
                                   c.N * c.C, &map))
    return cudaErrorInvalidConfiguration;
  g.contig = g.mode == kCopyDense;  // x planes n*C + c are contiguous

  switch (dl) {
    case 0: return launch_fwd<T, K, S, D, 0>(c, g, map, x, w, b, y, s, ep);
    case 1: return launch_fwd<T, K, S, D, Q == 1 ? 1 : 0>(c, g, map, x, w, b, y, s, ep);
    case 2: return launch_fwd<T, K, S, D, Q == 1 ? 2 : 0>(c, g, map, x, w, b, y, s, ep);
    default: return launch_fwd<T, K, S, D, Q == 1 ? 3 : 0>(c, g, map, x, w, b, y, s, ep);
  }
}

template <typename T, int K, int D, int DL>
cudaError_t launch_bwd1(const Conv& c, const Cfg& g, const CUtensorMap& map, int qh, const void* gy,
                        const void* w, void* gx, bool acc, cudaStream_t s) {
  constexpr int R = Blk<K, 1>::R, V = Blk<K, 1>::V;
  auto kern = bwd1_kernel<T, K, D, R, V, DL>;
  const size_t smem = 128 + 2 * ((size_t)g.stage_elems + g.stg_elems) * sizeof(T) + 2 * (size_t)g.tab_floats * 4;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = persistent_grid(kern, smem, g.groups * g.nbands);
  kern<<<grid, kNT, smem, s>>>(c, g, map, tma::timeout_counter(), qh, (const T*)gy, (const T*)w, (T*)gx, acc);
  return cudaGetLastError();
}

template <typename T, int K, int D>
cudaError_t run_bwd1_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc,
                       cudaStream_t s) {
  constexpr int R = Blk<K, 1>::R, V = Blk<K, 1>::V, Q = Geo<K, 1, D>::Q;
  const int qh = D * (K - 1) - c.ph, qw = D * (K - 1) - c.pw;
  const bool vout = Q == 1 && c.W % 4 == 0 && alignedn(gx, 4 * sizeof(T));
  // grad_out plane bases are multiples of Ho*Wo elements from gy, so a
  // 16-byte aligned gy with 16-byte rows keeps every plane base aligned
  Cfg g;
  int dl = 0;
  alignas(64) CUtensorMap map{};
  if (!plan_tile<T, K, 1, D, R, V>(c.N * c.C, c.m, 1, c.Ho, c.Wo, c.H, c.W, qw, gy, vout, &g, &dl, c.C,
                                   c.N * c.ctot, &map))
    return cudaErrorInvalidConfiguration;
  // grad_out planes of consecutive (n, c) are contiguous without a channel slice
  g.contig = g.mode == kCopyDense && c.off == 0 && c.ctot == c.C * c.m;

  switch (dl) {
    case 0: return launch_bwd1<T, K, D, 0>(c, g, map, qh, gy, w, gx, acc, s);
    case 1: return launch_bwd1<T, K, D, Q == 1 ? 1 : 0>(c, g, map, qh, gy, w, gx, acc, s);
    case 2: return launch_bwd1<T, K, D, Q == 1 ? 2 : 0>(c, g, map, qh, gy, w, gx, acc, s);
    default: return launch_bwd1<T, K, D, Q == 1 ? 3 : 0>(c, g, map, qh, gy, w, gx, acc, s);
  }
}

}  // namespace

template <typename T>
cudaError_t fwd_t(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                  const Epi& ep) {
#define X(K, S, D) if (c.kh == K && c.sh == S && c.dh == D) return run_fwd_t<T, K, S, D>(c, x, w, b, y, s, ep);
  DW_FWD_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

template <typename T>
cudaError_t bwd1_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
#define X(K, D) if (c.kh == K && c.dh == D) return run_bwd1_t<T, K, D>(c, gy, w, gx, acc, s);
  DW_BWD1_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace tile
}  // namespace dwconv
