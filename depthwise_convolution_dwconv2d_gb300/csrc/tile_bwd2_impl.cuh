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
#pragma once
#include "plan.h"
#include "tile_cases.h"
#include "tma.cuh"
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
  int ppc, thu, nbands, tr, pitch, rb, cb, tile_elems, stage_elems, vec_out;
  int64_t groups;
  int row0;         // grad_out row of tile row 0, relative to the band's first u row
  int mode, ix0;    // copy mode, grad_out column of tile column 0
  int cshift;       // added to each thread's window start column
  FastDiv trdiv, d_plane, d_cb, d_bands;
  uint32_t tma_bytes;
  int seg, stg_elems;  // dense staging of whole grad_out planes
  int balanced;        // equal contiguous plane shares per CTA (see Sched)
  int contig;          // dense staging: a stage's planes are one contiguous run
  int tab_floats;      // per-stage filter table: ppc*m*K*K floats (rounded)
  int ostage;          // results of whole gx planes go through shared memory
  int ostg_elems;      // size of that output staging buffer (elements)
};

template <typename T, int K, int S, int D, int PM, int R, int V, int DL>
__global__ void __launch_bounds__(kNT)
bwd2_kernel(Conv c, Bwd2Cfg g, const __grid_constant__ CUtensorMap tmap, unsigned int* timeouts,
            const T* __restrict__ gy, const T* __restrict__ w, T* gx, bool accumulate) {
  extern __shared__ __align__(16) unsigned char smdyn[];
  __shared__ __align__(8) uint64_t bars[2];
  unsigned char* smraw = smdyn + ((128 - (tma::smem_u32(smdyn) & 127)) & 127);
  const bool use_tma = g.mode == kCopyTMA;
  if (use_tma && threadIdx.x == 0) {
    tma::mbar_init(&bars[0], 1);
    tma::mbar_init(&bars[1], 1);
    tma::fence_init();
  }
  __syncthreads();
  using P = Phase<K, S, D, PM>;
  constexpr int OM = P::omin(), SP = P::span;
  constexpr int W4 = (DL + V + SP + 3) / 4 * 4;
  T* const buf0 = reinterpret_cast<T*>(smraw);
  T* const buf1 = buf0 + g.stage_elems;
  T* const stg0 = buf1 + g.stage_elems;
  T* const stg1 = stg0 + g.stg_elems;
  // per stage: the filters of the stage's (plane, j) pairs; then the output
  // staging buffer (whole gx planes of one unit, written out coalesced)
  float* const tab0 = reinterpret_cast<float*>(stg1 + g.stg_elems);
  float* const tab1 = tab0 + g.tab_floats;
  T* const ostg = reinterpret_cast<T*>(tab1 + g.tab_floats);
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
    // one (plane, j) filter per thread
    for (int sj = threadIdx.x; sj < np * m; sj += kNT) {
      const int pl = m == 1 ? sj : sj / m;
      int64_t n, ch;
      c.split(p0 + pl, n, ch);
      const T* wp = w + (ch * m + (sj - pl * m)) * (K * K);
#pragma unroll
      for (int i = 0; i < K * K; ++i) tab_put(tab + sj * (K * K) + i, wp + i);
    }
    if (g.mode == kCopyDense) {
      if (g.contig)
        issue_contig<T>(stg, gy_plane(p0, 0), (int64_t)np * m * c.Ho * c.Wo);
      else
        issue_flat<T>(stg, np * m, g.seg, [&](int s) { return gy_plane(p0, s); }, (int)(c.Ho * c.Wo));
      return;
    }
    if (use_tma) {
      if (threadIdx.x == 0) {
        int64_t n, ch;
        c.split(p0, n, ch);  // units never straddle samples
        tma::fence_async_smem();
        tma::mbar_expect_tx(bar, g.tma_bytes);
        tma::load_3d(dst, &tmap, g.ix0, band * g.thu + g.row0, (int)(n * c.ctot + c.off + ch * m), bar);
      }
      return;
    }
    issue_tile<T>(dst, np * m, g.tile_elems, g.pitch,
                  [&](int s) { return gy_plane(p0, s); },
                  (int)c.Ho, (int)c.Wo, band * g.thu + g.row0, g.tr, g.trdiv, g.ix0, g.mode);
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
    if (more)
      issue(p0n, npn, bandn, (k & 1) ? buf0 : buf1, (k & 1) ? stg0 : stg1, (k & 1) ? tab0 : tab1,
            &bars[(k + 1) & 1]);
    cp_async_commit();
    cp_async_wait<1>();
    if (use_tma && !tma::mbar_wait(&bars[k & 1], (uint32_t)(k >> 1) & 1, timeouts)) {
      if (more) tma::mbar_wait(&bars[(k + 1) & 1], (uint32_t)((k + 1) >> 1) & 1, nullptr);
      return;
    }
    __syncthreads();
    const int u0 = band * g.thu;  // first u row of the band (gx row S*u0)
    const T* stg = (k & 1) ? stg1 : stg0;
    const bool dense = g.mode == kCopyDense;
    const int total = np * (int)g.d_plane.d;
    float wr[K * K];
    for (int it = threadIdx.x; it < total; it += kNT) {
      uint32_t pl_, rbi_;
      const uint32_t rem = g.d_plane.divmod((uint32_t)it, pl_);
      const int cbi = (int)g.d_cb.divmod(rem, rbi_);
      const int pl = (int)pl_, rbi = (int)rbi_;
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
#pragma unroll
        for (int i = 0; i < K * K; ++i) wr[i] = tab[(pl * m + j) * (K * K) + i];
        const T* t = cur + (pl * m + j) * g.tile_elems + (rbi * R) * g.pitch + cbi * V + g.cshift;
        // dense: grad_out plane coordinates of window (0, 0)
        const T* dp = !dense ? nullptr
                      : g.contig ? dense_at(stg, gy_plane(p0, 0), (pl * m + j) * (int)(c.Ho * c.Wo))
                                 : dense_plane(stg, g.seg, pl * m + j, gy_plane(p0, pl * m + j));
        const int gyr = u0 + g.row0 + rbi * R, gyc = g.ix0 + g.cshift + DL + cbi * V;
#pragma unroll
        for (int ut = 0; ut < R + SP; ++ut) {
          float win[W4];
          if (dense) {
            const int iy = gyr + ut;
            if ((unsigned)iy >= (unsigned)c.Ho) continue;
#pragma unroll
            for (int i = 0; i < V + SP; ++i) {
              const int ix = gyc + i;
              win[DL + i] = (unsigned)ix < (unsigned)c.Wo ? ld1<T>(dp + iy * c.Wo + ix) : 0.f;
            }
          } else {
#pragma unroll
            for (int i = 0; i < W4 / 4; ++i) ld4<T>(t + ut * g.pitch + 4 * i, win + 4 * i);
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
                      acc[r][ph][v][pw] = fmaf(wr[a * K + b], win[DL + v + P::off(pw, b) - OM], acc[r][ph][v][pw]);
                  }
              }
        }
      }
      // store rows S*(u0 + rbi*R + r) + ph, cols S*cbi*V .. + S*V
      const int col0 = S * V * cbi;
      if (g.ostage) {
        T* plane = ostg + pl * (int)(c.H * c.W);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int ph = 0; ph < S; ++ph) {
            const int ih = S * (u0 + rbi * R + r) + ph;
            if (ih >= c.H) continue;
#pragma unroll
            for (int v = 0; v < V; ++v)
#pragma unroll
              for (int pw = 0; pw < S; ++pw) {
                const int iw = col0 + v * S + pw;
                if (iw < c.W) plane[ih * c.W + iw] = from_f<T>(acc[r][ph][v][pw]);
              }
          }
        continue;
      }
      T* plane = gx + pin * c.H * c.W;
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
          if (g.vec_out && (S * V) % 4 == 0) {
            // W % 4 == 0 and col0 % 4 == 0: every group of four columns is
            // wholly inside the row or wholly past its end
#pragma unroll
            for (int q = 0; q < S * V / 4; ++q) {
              if (col0 + 4 * q >= c.W) break;
              float f[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                f[i] = accumulate ? o[4 * q + i] + ld_rw(rowp + col0 + 4 * q + i) : o[4 * q + i];
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
    if (g.ostage) {
      // the unit's gx planes are contiguous in memory
      __syncthreads();
      flush_staged<T>(gx + p0 * c.H * c.W, ostg, np * (int)(c.H * c.W), accumulate);
    }
    __syncthreads();
    have = more;
  }
}

template <typename T, int K, int S, int D, int PM, int DL>
cudaError_t launch_bwd2(const Conv& c, const Bwd2Cfg& g, const CUtensorMap& map, const void* gy,
                        const void* w, void* gx, bool acc, cudaStream_t s) {
  auto kern = bwd2_kernel<T, K, S, D, PM, 2, 4, DL>;
  const size_t smem = 128 + 2 * ((size_t)g.stage_elems + g.stg_elems) * sizeof(T) + 2 * (size_t)g.tab_floats * 4 +
                      (size_t)g.ostg_elems * sizeof(T);
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = persistent_grid(kern, smem, g.groups * g.nbands);
  kern<<<grid, kNT, smem, s>>>(c, g, map, tma::timeout_counter(), (const T*)gy, (const T*)w, (T*)gx, acc);
  return cudaGetLastError();
}

template <typename T, int K, int S, int D, int PM>
cudaError_t run_bwd2_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc,
                       cudaStream_t s) {
  constexpr int R = 2, V = 4;
  using P = Phase<K, S, D, PM>;
  constexpr int OM = P::omin(), SP = P::span;
  constexpr int ES = sizeof(T);
  Bwd2Cfg g{};
  const int64_t U = (c.H + S - 1) / S;  // u rows of gx
  g.cb = (int)((c.W + (int64_t)S * V - 1) / ((int64_t)S * V));
  int shift = 0;
  g.mode = pick_mode<T>(gy, c.Wo, (c.pw - PM) / S + OM, &g.ix0, &shift);
  const int dl = shift % 4;
  g.cshift = shift - dl;
  const int W4 = (dl + V + SP + 3) / 4 * 4;
  g.pitch = round_up((int64_t)(g.cb - 1) * V + g.cshift + W4, 16 / ES > 4 ? 16 / ES : 4);
  g.row0 = (c.ph - PM) / S + OM;
  const int64_t target = 32 * 1024;
  const int64_t row_bytes = (int64_t)g.pitch * ES * c.m;
  int64_t thu = (U + R - 1) / R * R;
  if ((thu + SP) * row_bytes > target) {
    thu = (target / row_bytes - SP) / R * R;
    if (thu < R) thu = R;
    if ((thu + SP) * row_bytes > 48 * 1024) return cudaErrorInvalidConfiguration;
  }
  g.thu = (int)thu;
  g.rb = (int)(thu / R);
  g.nbands = (int)((U + thu - 1) / thu);
  g.tr = (int)(thu + SP);
  g.tile_elems = g.tr * g.pitch;
  g.trdiv = FastDiv((uint32_t)g.tr);
  g.d_plane = FastDiv((uint32_t)(g.rb * g.cb));
  g.d_cb = FastDiv((uint32_t)g.cb);
  g.d_bands = FastDiv((uint32_t)g.nbands);
  const int64_t items = (int64_t)g.rb * g.cb;
  const int64_t nplanes = c.N * c.C;
  int64_t ppc = 1;
  if (g.nbands == 1) {
    ppc = (2 * kNT + items - 1) / items;
    const int64_t cap = target / ((int64_t)g.tile_elems * ES * c.m);
    if (ppc > cap) ppc = cap;
    if (ppc < 1) ppc = 1;
  }
  // dense staging of whole planes when grad_out rows are not 16-byte multiples
  if ((g.mode == kCopy4 || g.mode == kCopySync) && g.nbands == 1 &&
      (reinterpret_cast<uintptr_t>(gy) % 16) == 0) {
    const int seg = dense_seg<T>(c.Ho * c.Wo);
    const int64_t per = (int64_t)seg * ES * c.m;  // dense planes are read in place
    int64_t dppc = (2 * kNT + items - 1) / items;
    if (dppc > target / per) dppc = target / per;
    if (dppc >= 1) {
      g.mode = kCopyDense;
      g.seg = seg;
      ppc = dppc;
    }
  }
  alignas(64) CUtensorMap map{};
  bool tma = g.mode == kCopy16 && g.pitch <= 256 && g.tr <= 256 && ppc * c.m <= 256;
  if (tma) {
    while (ppc > 1 && c.C % ppc != 0) --ppc;  // units never straddle samples
    tma = tma::encode_3d(&map, gy, c.dtype, c.Wo, c.Ho, c.N * c.ctot, g.pitch, g.tr, (uint32_t)(ppc * c.m));
  }
  if (tma) g.mode = kCopyTMA;
  g.ppc = (int)ppc;
  g.groups = (nplanes + ppc - 1) / ppc;
  g.balanced = g.nbands == 1 && g.mode != kCopyTMA;
  g.contig = g.mode == kCopyDense && c.off == 0 && c.ctot == c.C * c.m;
  g.stage_elems = g.mode == kCopyDense ? 0 : stage_round((int64_t)g.ppc * c.m * g.tile_elems, ES);
  g.tma_bytes = (uint32_t)((int64_t)g.ppc * c.m * g.tile_elems * ES);
  g.stg_elems = g.mode == kCopyDense ? stage_round((int64_t)g.ppc * c.m * g.seg, ES) : 0;
  g.vec_out = (reinterpret_cast<uintptr_t>(gx) % (4 * ES) == 0) && c.W % 4 == 0;
  g.tab_floats = round_up((int64_t)g.ppc * c.m * K * K, 4);
  // small gx planes whose rows take no vector stores: whole planes through
  // shared memory (units are whole planes when there is one band)
  g.ostage = !g.vec_out && g.nbands == 1 && (int64_t)g.ppc * c.H * c.W * ES <= 64 * 1024;
  g.ostg_elems = g.ostage ? stage_round((int64_t)g.ppc * c.H * c.W, ES) : 0;
  switch (dl) {
    case 0: return launch_bwd2<T, K, S, D, PM, 0>(c, g, map, gy, w, gx, acc, s);
    case 1: return launch_bwd2<T, K, S, D, PM, 1>(c, g, map, gy, w, gx, acc, s);
    case 2: return launch_bwd2<T, K, S, D, PM, 2>(c, g, map, gy, w, gx, acc, s);
    default: return launch_bwd2<T, K, S, D, PM, 3>(c, g, map, gy, w, gx, acc, s);
  }
}

}  // namespace

template <typename T>
cudaError_t bwd2_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
  const int pm = c.ph % c.sh;
#define X(K, S, D, PM) \
  if (c.kh == K && c.sh == S && c.dh == D && pm == PM) return run_bwd2_t<T, K, S, D, PM>(c, gy, w, gx, acc, s);
  DW_BWD2_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace tile
}  // namespace dwconv
