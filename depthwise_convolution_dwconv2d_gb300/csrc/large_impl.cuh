// Large-kernel depthwise forward and stride-1 grad-input (square K up to 31,
// stride 1, dilation 1, multiplier 1), bound by fp32 FMA throughput.
//
// The MegEngine large-kernel depthwise article ("DirectConv") blocks the
// output at several levels -- CTA tile, warp rows, a few outputs per thread --
// and keeps the kernel and input windows on chip; its first simple version
// reaches 70-80 % of peak. The same idea on sm_103a: a CTA stages whole input
// planes (with their zero halo, in fp32) in shared memory together with each
// plane's filter; every thread owns an R x V block of outputs and walks the
// kernel rows, holding one filter row (K values) in registers and reading each
// input-row window with 16-byte vector loads, so every value it loads from
// shared memory feeds V*K or K fused multiply-adds. Input rows that fall in the
// zero padding are skipped, so padded kernel rows cost no FMAs.
//
// Grad-input at stride 1 is the same computation on grad_out with the filter
// rotated by 180 degrees and padding K-1-pad (the adjoint of the forward).
// The kernel is persistent and stages its next planes with cp.async while it
// computes the current ones.
#pragma once

#include "plan.h"
#include "tile.cuh"

namespace dwconv {
namespace large {
namespace {

using tile::kNT;

struct LCfg {
  int ppc;             // planes per unit
  int pitch, tr;       // tile row pitch / rows (fp32 elements): tr = Hin + 2*pad rows
  int tile_elems;      // floats per staged plane (tile + its filter)
  int wofs;            // offset of the filter inside a staged plane
  int rb, cb;          // item grid per plane: row blocks, column blocks
  int pad;             // padding of the stencil as evaluated (pad, or K-1-pad)
  int mode;            // tile::kCopy4 (fp32 cp.async) or tile::kCopySync (convert)
  int64_t groups;
  FastDiv trdiv, d_item, d_cb;
};

// Stage np planes (Hin x Win, from src_of) as fp32 rows [-pad, Hin + pad) x
// cols [-pad, -pad + pitch) plus the filter (flipped when FLIP) after each.
template <typename T, int K, bool FLIP, typename SrcOf>
__device__ __forceinline__ void stage(float* dst, const LCfg& g, int np, SrcOf src_of, const T* w,
                                      int64_t p0, int64_t C, int Hin, int Win) {
  if (g.mode == tile::kCopy4) {
    tile::issue_tile<float>(dst, np, g.tile_elems, g.pitch,
                            [&](int p) { return reinterpret_cast<const float*>(src_of(p)); }, Hin, Win,
                            -g.pad, g.tr, g.trdiv, -g.pad, tile::kCopy4);
  } else {
    // plain loads with conversion to fp32
    const int per = g.tr * g.pitch;
    for (int e = threadIdx.x; e < np * per; e += kNT) {
      const int p = e / per, q = e - p * per;
      const int r = q / g.pitch, col = q - r * g.pitch;
      const int iy = r - g.pad, ix = col - g.pad;
      dst[p * g.tile_elems + q] = (iy >= 0 && iy < Hin && ix >= 0 && ix < Win) ? ld(src_of(p) + (int64_t)iy * Win + ix) : 0.f;
    }
  }
  constexpr int KP = (K + 3) / 4 * 4;  // filter rows padded for 16-byte loads
  for (int e = threadIdx.x; e < np * K * KP; e += kNT) {
    const int p = e / (K * KP), t = e - p * (K * KP);
    const int a = t / KP, b = t - a * KP;
    const int64_t ch = (p0 + p) % C;  // the unit's planes may span two samples
    dst[p * g.tile_elems + g.wofs + t] =
        b < K ? ld(w + ch * (K * K) + (FLIP ? K * K - 1 - (a * K + b) : a * K + b)) : 0.f;
  }
}

template <typename T, int K, int R, int V, bool FLIP>
__global__ void __launch_bounds__(kNT)
large_kernel(Conv c, LCfg g, const T* __restrict__ in, const T* __restrict__ w, const T* __restrict__ bias,
             T* out, bool accumulate) {
  extern __shared__ __align__(16) unsigned char smraw[];
  constexpr int WN = V + K - 1;
  constexpr int W4 = (WN + 3) / 4 * 4;
  float* const buf0 = reinterpret_cast<float*>(smraw);
  // stencil geometry: the forward reads x (H x W) and writes y (Ho x Wo);
  // the grad-input reads grad_out (Ho x Wo) and writes gx (H x W)
  const int Hin = FLIP ? (int)c.Ho : (int)c.H, Win = FLIP ? (int)c.Wo : (int)c.W;
  const int Hout = FLIP ? (int)c.H : (int)c.Ho, Wout = FLIP ? (int)c.W : (int)c.Wo;
  const int64_t nplanes = c.N * c.C;
  const int64_t units = g.groups;
  auto src_of = [&](int64_t pin) {
    int64_t n, ch;
    c.split(pin, n, ch);
    return FLIP ? in + c.y_base(n, ch) : in + c.x_base(n, ch);
  };
  auto dst_of = [&](int64_t pin) {
    int64_t n, ch;
    c.split(pin, n, ch);
    return FLIP ? out + c.x_base(n, ch) : out + c.y_base(n, ch);
  };
  auto issue = [&](int64_t u, float* dst) {
    const int64_t p0 = u * g.ppc;
    const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
    stage<T, K, FLIP>(dst, g, np, [&](int p) { return src_of(p0 + p); }, w, p0, c.C, Hin, Win);
  };
  // one stage: the compute of a unit is long next to its load, and the
  // other CTAs resident on the SM keep it busy while this one loads
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    issue(u, buf0);
    tile::cp_async_commit();
    tile::cp_async_wait<0>();
    __syncthreads();
    const float* cur = buf0;
    const int64_t p0 = u * g.ppc;
    const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
    const int ipp = (int)g.d_item.d;
    // items ordered (row block, plane, column block): a warp's lanes share
    // output rows, so they walk the same kernel rows
    const int per_rb = np * g.cb;
    for (int it = threadIdx.x; it < np * ipp; it += kNT) {
      const int rbi = it / per_rb;
      const int rem = it - rbi * per_rb;
      uint32_t pl_;
      const int cbi = (int)g.d_cb.divmod((uint32_t)rem, pl_);
      const int pl = (int)pl_;
      const float* t = cur + pl * g.tile_elems;
      const float* wt = t + g.wofs;
      const int oh0 = rbi * R, ow0 = cbi * V;
      int64_t n_, ch_;
      c.split(p0 + pl, n_, ch_);
      const float bv = bias ? ld(bias + ch_) : 0.f;
      float acc[R][V];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < V; ++v) acc[r][v] = bv;
      // kernel rows that reach an input row inside the plane for some r
      int a_lo = g.pad - oh0 - (R - 1);
      if (a_lo < 0) a_lo = 0;
      int a_hi = Hin + g.pad - oh0;
      if (a_hi > K) a_hi = K;
      constexpr int KP = (K + 3) / 4 * 4;
      for (int a = a_lo; a < a_hi; ++a) {
        float wrow[KP];
#pragma unroll
        for (int b = 0; b < KP / 4; ++b) {
          const float4 f = *reinterpret_cast<const float4*>(wt + a * KP + 4 * b);
          wrow[4 * b] = f.x; wrow[4 * b + 1] = f.y; wrow[4 * b + 2] = f.z; wrow[4 * b + 3] = f.w;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int iy = oh0 + r + a - g.pad;  // input row
          if (iy < 0 || iy >= Hin) continue;
          const float* rowp = t + (iy + g.pad) * g.pitch + ow0;
          float win[W4];
#pragma unroll
          for (int i = 0; i < W4 / 4; ++i) {
            const float4 f = *reinterpret_cast<const float4*>(rowp + 4 * i);
            win[4 * i] = f.x; win[4 * i + 1] = f.y; win[4 * i + 2] = f.z; win[4 * i + 3] = f.w;
          }
#pragma unroll
          for (int b = 0; b < K; ++b)
#pragma unroll
            for (int v = 0; v < V; ++v) acc[r][v] = fmaf(wrow[b], win[v + b], acc[r][v]);
        }
      }
      T* dp = dst_of(p0 + pl);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int oh = oh0 + r;
        if (oh >= Hout) break;
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const int ow = ow0 + v;
          if (ow < Wout) {
            T* o = dp + (int64_t)oh * Wout + ow;
            *o = from_f<T>(accumulate ? acc[r][v] + ld_rw(o) : acc[r][v]);
          }
        }
      }
    }
    __syncthreads();
  }
}

template <typename T, int K, bool FLIP, int R>
cudaError_t run_r(const Conv& c, const void* in, const void* w, const void* bias, void* out, bool acc,
                  cudaStream_t s) {
  constexpr int V = 4;
  constexpr int W4 = (V + K - 1 + 3) / 4 * 4;
  const int Win = FLIP ? (int)c.Wo : (int)c.W;
  const int Hout = FLIP ? (int)c.H : (int)c.Ho, Wout = FLIP ? (int)c.W : (int)c.Wo;
  LCfg g{};
  g.pad = FLIP ? K - 1 - c.ph : c.ph;
  g.cb = (Wout + V - 1) / V;
  g.rb = (Hout + R - 1) / R;
  g.pitch = tile::round_up((int64_t)(g.cb - 1) * V + W4, 4);
  if (g.pitch < Win + g.pad) g.pitch = tile::round_up(Win + g.pad, 4);
  g.tr = g.rb * R + K - 1;  // rows read by every block, padded ones included
  g.wofs = tile::round_up((int64_t)g.tr * g.pitch, 4);
  g.tile_elems = tile::round_up(g.wofs + K * ((K + 3) / 4 * 4), 4);
  const int64_t plane_bytes = (int64_t)g.tile_elems * 4;
  const int64_t ipp = (int64_t)g.rb * g.cb;
  int64_t ppc = (kNT + ipp - 1) / ipp;
  const int64_t cap = (72 * 1024) / plane_bytes;
  if (ppc > cap) ppc = cap;
  if (ppc < 1) ppc = 1;
  if (ppc * plane_bytes > 200 * 1024) return cudaErrorInvalidConfiguration;
  g.ppc = (int)ppc;
  const int64_t nplanes = c.N * c.C;
  g.groups = (nplanes + ppc - 1) / ppc;
  g.mode = (sizeof(T) == 4 && (reinterpret_cast<uintptr_t>(in) % 4) == 0) ? tile::kCopy4 : tile::kCopySync;
  g.trdiv = FastDiv((uint32_t)g.tr);
  g.d_item = FastDiv((uint32_t)ipp);
  g.d_cb = FastDiv((uint32_t)g.cb);
  auto kern = large_kernel<T, K, R, V, FLIP>;
  const size_t smem = (size_t)g.ppc * g.tile_elems * 4;
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = tile::persistent_grid(kern, smem, g.groups);
  kern<<<grid, kNT, smem, s>>>(c, g, (const T*)in, (const T*)w, (const T*)bias, (T*)out, acc);
  return cudaGetLastError();
}

// ---- weight gradient --------------------------------------------------------
// gw[oc, a, b] = sum_{n, oh, ow} gy[n, oc, oh, ow] * x[n, oc, oh + a - p, ow + b - p]
// for one chunk of samples: a correlation of the padded x plane with the
// grad_out plane that produces a K x K result. A CTA owns one channel and a
// chunk of samples; a thread owns an R x V block of taps (a, b) for a subset
// of the output rows (thread group g takes rows oh = g, g + G, ...). For each
// of its rows it walks grad_out four columns at a time (one 16-byte load,
// the same address across the warp) against a sliding register window of x.
// At the end of the chunk the groups' sums are added in a fixed order and
// written as one partial per (chunk, channel); the second pass adds chunks.
struct WLCfg {
  int nb, chunks;
  int xpitch, xrows, x_elems;   // padded x tile
  int gpitch, g_elems;          // grad_out tile (Ho x gpitch)
  int stage_elems;
  int rbA, cbB, items, G;       // tap blocks and output-row groups
  int pad, mode;
  FastDiv xrdiv, grdiv;
};

template <typename T, int K, int R, int V>
__global__ void __launch_bounds__(kNT)
large_wgrad_kernel(Conv c, WLCfg g, const T* __restrict__ x, const T* __restrict__ gy, float* __restrict__ ws) {
  extern __shared__ __align__(16) unsigned char smraw[];
  float* const buf0 = reinterpret_cast<float*>(smraw);
  float* const buf1 = buf0 + g.stage_elems;
  float* const red = buf1 + g.stage_elems;  // [G][K*K + 1]
  const int64_t units = c.C * g.chunks;
  const int H = (int)c.H, W = (int)c.W, Ho = (int)c.Ho, Wo = (int)c.Wo;
  auto issue = [&](int64_t n, int64_t ch, float* dst) {
    const T* xp = x + c.x_base(n, ch);
    const T* gp = gy + c.y_base(n, ch);
    if (g.mode == tile::kCopy4) {
      tile::issue_tile<float>(dst, 1, g.x_elems, g.xpitch, [&](int) { return reinterpret_cast<const float*>(xp); },
                              H, W, -g.pad, g.xrows, g.xrdiv, -g.pad, tile::kCopy4);
      tile::issue_tile<float>(dst + g.x_elems, 1, g.g_elems, g.gpitch,
                              [&](int) { return reinterpret_cast<const float*>(gp); }, Ho, Wo, 0, Ho, g.grdiv, 0,
                              tile::kCopy4);
    } else {
      for (int e = threadIdx.x; e < g.x_elems; e += kNT) {
        const int r = e / g.xpitch, col = e - r * g.xpitch;
        const int iy = r - g.pad, ix = col - g.pad;
        dst[e] = (iy >= 0 && iy < H && ix >= 0 && ix < W) ? ld(xp + (int64_t)iy * W + ix) : 0.f;
      }
      for (int e = threadIdx.x; e < g.g_elems; e += kNT) {
        const int r = e / g.gpitch, col = e - r * g.gpitch;
        dst[g.x_elems + e] = (col < Wo) ? ld(gp + (int64_t)r * Wo + col) : 0.f;
      }
    }
  };
  // the CTA's steps: (unit u, sample s in its chunk)
  int64_t u = blockIdx.x;
  int sidx = 0;
  // unit uu = chunk * C + channel
  auto unit_n0 = [&](int64_t uu) {
    uint32_t q;
    c.dC.divmod((uint32_t)uu, q);
    return (int64_t)q * g.nb;
  };
  auto unit_ch = [&](int64_t uu) {
    uint32_t q;
    return (int64_t)c.dC.divmod((uint32_t)uu, q);
  };
  auto unit_ns = [&](int64_t uu) {
    const int64_t n0 = unit_n0(uu);
    const int64_t ns = (c.N - n0) < g.nb ? (c.N - n0) : g.nb;
    return (int)(ns > 0 ? ns : 0);
  };
  if (u < units && unit_ns(u) > 0) issue(unit_n0(u) + sidx, unit_ch(u), buf0);
  tile::cp_async_commit();
  const int tid = threadIdx.x;
  const int item = tid % g.items, grp = tid / g.items;
  const bool active = grp < g.G;
  const int a0 = (item / g.cbB) * R, b0 = (item % g.cbB) * V;
  float acc[R][V];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int v = 0; v < V; ++v) acc[r][v] = 0.f;
  float bsum = 0.f;
  for (int k = 0; u < units; ++k) {
    // next step
    int64_t un = u;
    int sn = sidx + 1;
    if (sn >= unit_ns(u)) {
      sn = 0;
      un = u + gridDim.x;
    }
    if (un < units && unit_ns(un) > 0) issue(unit_n0(un) + sn, unit_ch(un), (k & 1) ? buf0 : buf1);
    tile::cp_async_commit();
    tile::cp_async_wait<1>();
    __syncthreads();
    const float* xs = (k & 1) ? buf1 : buf0;
    const float* gs = xs + g.x_elems;
    if (unit_ns(u) > 0) {
      for (int e = tid; e < Ho * g.gpitch; e += kNT) bsum += gs[e];  // padded columns are zero
      if (active) {
        for (int oh = grp; oh < Ho; oh += g.G) {
          const float* grow = gs + oh * g.gpitch;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int a = a0 + r;
            // x tile row of input row oh + a - pad is oh + a (origin -pad)
            if (a >= K) break;
            if ((unsigned)(oh + a - g.pad) >= (unsigned)H) continue;  // a padding row: zero
            const float* xrow = xs + (oh + a) * g.xpitch + b0;
            float xw[V + 3 + 4];
            {
              const float4 f = *reinterpret_cast<const float4*>(xrow);
              xw[0] = f.x; xw[1] = f.y; xw[2] = f.z; xw[3] = f.w;
            }
            for (int ow = 0; ow < g.gpitch; ow += 4) {
              const float4 gv = *reinterpret_cast<const float4*>(grow + ow);
              const float4 f = *reinterpret_cast<const float4*>(xrow + ow + 4);
              xw[4] = f.x; xw[5] = f.y; xw[6] = f.z; xw[7] = f.w;
              const float gg[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
              for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int v = 0; v < V; ++v) acc[r][v] = fmaf(gg[j], xw[j + v], acc[r][v]);
#pragma unroll
              for (int i = 0; i < 4; ++i) xw[i] = xw[i + 4];
            }
          }
        }
      }
    }
    const bool last = (un != u) || (k >= 0 && unit_ns(u) == 0);
    if (last) {
      // fixed-order reduction of the groups' sums, then one partial per chunk
      __syncthreads();
      if (active) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int v = 0; v < V; ++v) {
            const int a = a0 + r, b = b0 + v;
            if (a < K && b < K) red[grp * (K * K + 1) + a * K + b] = acc[r][v];
            acc[r][v] = 0.f;
          }
      }
      // bias: warp butterfly, then warps in order
      float bv = bsum;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bv += __shfl_xor_sync(0xffffffffu, bv, o);
      bsum = 0.f;
      float* wred = red + g.G * (K * K + 1);
      if ((tid & 31) == 0) wred[tid >> 5] = bv;
      __syncthreads();
      uint32_t cq;
      const int64_t ch = c.dC.divmod((uint32_t)u, cq);
      const int chunk = (int)cq;
      float* dstp = ws + ((int64_t)chunk * c.OC() + ch) * (K * K + 1);
      for (int t = tid; t < K * K; t += kNT) {
        float sum = 0.f;
        for (int gi = 0; gi < g.G; ++gi) sum += red[gi * (K * K + 1) + t];
        dstp[t] = sum;
      }
      if (tid == 0) {
        float sum = 0.f;
        for (int wi = 0; wi < kNT / 32; ++wi) sum += wred[wi];
        dstp[K * K] = sum;
      }
    }
    __syncthreads();
    u = un;
    sidx = sn;
  }
}

// Two output rows per thread on planes of up to 32 rows (more blocks, so one
// or two planes fill a CTA), four on larger planes.
template <typename T, int K, bool FLIP>
cudaError_t run(const Conv& c, const void* in, const void* w, const void* bias, void* out, bool acc,
                cudaStream_t s) {
  const int64_t Hout = FLIP ? c.H : c.Ho;
  if (Hout <= 32) return run_r<T, K, FLIP, 2>(c, in, w, bias, out, acc, s);
  return run_r<T, K, FLIP, 4>(c, in, w, bias, out, acc, s);
}

template <typename T, int K>
cudaError_t run_wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
  constexpr int R = 4, V = 4;
  WLCfg g{};
  g.chunks = chunks;
  g.nb = (int)((c.N + chunks - 1) / chunks);
  g.pad = c.ph;
  g.gpitch = tile::round_up(c.Wo, 4);
  g.g_elems = (int)c.Ho * g.gpitch;
  // x columns read: b0 + ow + 7 for ow < gpitch, b0 < K
  g.xpitch = tile::round_up((int64_t)((K + V - 1) / V) * V + g.gpitch + 4, 4);
  if (g.xpitch < c.W + c.pw) g.xpitch = tile::round_up(c.W + c.pw, 4);
  g.xrows = (int)c.Ho + K - 1;
  g.x_elems = g.xrows * g.xpitch;
  g.stage_elems = tile::round_up((int64_t)g.x_elems + g.g_elems, 4);
  g.rbA = (K + R - 1) / R;
  g.cbB = (K + V - 1) / V;
  g.items = g.rbA * g.cbB;
  g.G = g.items >= kNT ? 1 : kNT / g.items;
  if (g.items > kNT) return cudaErrorInvalidConfiguration;
  g.mode = (sizeof(T) == 4 && (reinterpret_cast<uintptr_t>(x) % 4) == 0 &&
            (reinterpret_cast<uintptr_t>(gy) % 4) == 0) ? tile::kCopy4 : tile::kCopySync;
  g.xrdiv = FastDiv((uint32_t)g.xrows);
  g.grdiv = FastDiv((uint32_t)c.Ho);
  const size_t smem = (2 * (size_t)g.stage_elems + (size_t)g.G * (K * K + 1) + kNT / 32) * 4;
  if (smem > 220 * 1024) return cudaErrorInvalidConfiguration;
  auto kern = large_wgrad_kernel<T, K, R, V>;
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = tile::persistent_grid(kern, smem, c.C * chunks);
  kern<<<grid, kNT, smem, s>>>(c, g, (const T*)x, (const T*)gy, ws);
  return cudaGetLastError();
}

}  // namespace

#define DW_LARGE_CASES(X) X(7) X(9) X(11) X(13) X(15) X(21) X(27) X(31)

template <typename T>
cudaError_t fwd_t(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s) {
#define X(K) if (c.kh == K) return run<T, K, false>(c, x, w, b, y, false, s);
  DW_LARGE_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

template <typename T>
cudaError_t wgrad_t(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
#define X(K) if (c.kh == K) return run_wgrad<T, K>(c, x, gy, ws, chunks, s);
  DW_LARGE_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

template <typename T>
cudaError_t bwd_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
#define X(K) if (c.kh == K) return run<T, K, true>(c, gy, w, nullptr, gx, acc, s);
  DW_LARGE_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace large
}  // namespace dwconv
