// Large-kernel depthwise weight gradient on the fp32 FMA pipes (square odd K
// from 7 to 31, stride 1, dilation 1, one filter per channel); the forward
// and the stride-1 grad-input are in large_pair.cuh.
//
// The storage type (fp32 / fp16 / bf16) only changes how planes are staged,
// so it is a run-time argument: one kernel per K.
#pragma once

#include "large_common.cuh"
#include "large_pair.cuh"
#include "large_pwgrad.cuh"

namespace dwconv {
namespace large {

// ---- weight gradient --------------------------------------------------------
// gw[oc, a, b] = sum_{n, oh, ow} gy[n, oc, oh, ow] * x[n, oc, oh + a - p, ow + b - p]
// for one chunk of samples: a correlation of the padded x plane with the
// grad_out plane that produces a K x K result. A CTA owns one channel and a
// chunk of samples and stages one sample's padded x plane and grad_out plane
// per step (two stages). A thread owns a block of 4 filter rows x 8 filter
// columns; the threads holding all blocks of the filter form a group, and
// group g takes the output rows oh = g, g + G, ... For each of its rows a
// thread walks grad_out four columns at a time (one 16-byte load, the same
// address for the whole group) against a sliding register window of three
// 16-byte chunks of each of its four x rows, so every chunk it loads feeds 32
// fused multiply-adds. The x rows are stored with their chunks
// de-interleaved (even chunks first), with an odd number of chunks per row:
// the lanes of a quarter-warp then read eight different bank groups. At the
// end of the chunk the groups' sums are added in a fixed order and written as
// one partial per (chunk, channel); the second pass adds the chunks.
struct WLCfg {
  int nb, chunks;
  int nq, half_e, xpitch, xrows, x_elems;  // padded x tile (de-interleaved rows)
  int gpitch, g_elems;                     // grad_out tile (Ho x gpitch, plain rows)
  int buf_elems;                           // floats per stage (>= reduction buffer)
  int G;                                   // groups of output rows
  int pad, dtype, raw16;
  int rawx_elems;                          // 16-bit raw area of the x plane (elements)
  FastDiv d_xrows;
};

template <int K>
struct WGeo {
  static constexpr int RA = 4, VB = 8;
  static constexpr int NA = (K + RA - 1) / RA, NB = (K + VB - 1) / VB;
  static constexpr int items = NA * NB;
};

template <int K>
__global__ void __launch_bounds__(kNT, 2)
wgrad_kernel(Conv c, WLCfg g, const void* __restrict__ x, const void* __restrict__ gy, float* __restrict__ ws) {
  using Gm = WGeo<K>;
  constexpr int RA = Gm::RA, VB = Gm::VB, NB = Gm::NB, ITEMS = Gm::items;
  extern __shared__ __align__(16) float sm[];
  const int tid = threadIdx.x;
  const int64_t units = c.C * g.chunks;
  const int H = (int)c.H, W = (int)c.W, Ho = (int)c.Ho, Wo = (int)c.Wo;
  const int es = g.dtype == DWCONV_F32 ? 4 : 2;
  auto xsrc = [&](int64_t n, int64_t ch) { return reinterpret_cast<const char*>(x) + c.x_base(n, ch) * es; };
  auto gsrc = [&](int64_t n, int64_t ch) { return reinterpret_cast<const char*>(gy) + c.y_base(n, ch) * es; };
  const int lane = tid & 31, nw = kNT / 32;
  // fp32 data: cp.async of every element straight into the fp32 tiles
  auto issue_f32 = [&](int64_t n, int64_t ch, float* dst) {
    const void* xp = xsrc(n, ch);
    const float* gp = reinterpret_cast<const float*>(gsrc(n, ch));
    stage_planes(dst, 1, g.x_elems, g.xrows, g.nq, g.half_e, g.d_xrows, [&](int) { return xp; }, H, W, g.pad,
                 g.dtype, true);
    for (int r = tid >> 5; r < Ho; r += nw) {
      float* gd = dst + g.x_elems + r * g.gpitch;
      for (int col = lane; col < g.gpitch; col += 32) {
        const bool in = col < Wo;
        tile::cp_async4(gd + col, gp + (in ? (int64_t)r * Wo + col : 0), in ? 4 : 0);
      }
    }
  };
  // 16-bit data: 16-byte cp.async of the two dense planes into a raw area,
  // widened into the fp32 tiles by convert() once they have landed
  unsigned short* rawx = reinterpret_cast<unsigned short*>(sm + g.buf_elems);
  unsigned short* rawg = rawx + g.rawx_elems;
  auto issue_raw = [&](int64_t n, int64_t ch) {
    tile::issue_contig(rawx, reinterpret_cast<const unsigned short*>(xsrc(n, ch)), (int64_t)H * W);
    tile::issue_contig(rawg, reinterpret_cast<const unsigned short*>(gsrc(n, ch)), (int64_t)Ho * Wo);
  };
  auto convert = [&](int64_t n, int64_t ch, float* dst) {
    const unsigned short* xr = tile::dense_at(rawx, reinterpret_cast<const unsigned short*>(xsrc(n, ch)), 0);
    const unsigned short* gr = tile::dense_at(rawg, reinterpret_cast<const unsigned short*>(gsrc(n, ch)), 0);
    auto wide = [&](unsigned short b) {
      return g.dtype == DWCONV_F16 ? __half2float(__ushort_as_half(b)) : __bfloat162float(__ushort_as_bfloat16(b));
    };
    // x tile rows in the de-interleaved layout (lane offsets as in stage_planes)
    const int q0 = lane >> 2;
    const int lane_off = 4 * phys_chunk(q0, g.half_e) + (lane & 3);
    for (int r = tid >> 5; r < g.xrows; r += nw) {
      const int iy = r - g.pad;
      const bool rin = iy >= 0 && iy < H;
      float* d = dst + r * g.xpitch + lane_off;
      for (int col = lane; col < g.xpitch; col += 32, d += 16) {
        const int ix = col - g.pad;
        *d = (rin && ix >= 0 && ix < W) ? wide(xr[iy * W + ix]) : 0.f;
      }
    }
    for (int r = tid >> 5; r < Ho; r += nw) {
      float* gd = dst + g.x_elems + r * g.gpitch;
      for (int col = lane; col < g.gpitch; col += 32) gd[col] = col < Wo ? wide(gr[r * Wo + col]) : 0.f;
    }
  };
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
  // step after (uu, ss): the next sample of the unit, else the CTA's next unit
  auto next_step = [&](int64_t& uu, int& ss) {
    if (++ss >= unit_ns(uu)) {
      ss = 0;
      uu += gridDim.x;
    }
  };

  const int item = tid % ITEMS, grp = tid / ITEMS;
  const bool active = grp < g.G;
  const int ia = item / NB, ib = item - ia * NB;
  const int a0 = ia * RA, b0 = ib * VB;
  const int n4 = g.gpitch / 4;
  float acc[RA][VB];
#pragma unroll
  for (int r = 0; r < RA; ++r)
#pragma unroll
    for (int v = 0; v < VB; ++v) acc[r][v] = 0.f;
  float bsum = 0.f;

  // one step: this sample's contribution to the thread's taps
  auto compute = [&](const float* xs, const float* gs) {
    for (int e = tid; e < g.g_elems; e += kNT) bsum += gs[e];  // padded columns are zero
    if (!active) return;
    for (int oh = grp; oh < Ho; oh += g.G) {
      const float* grow = gs + oh * g.gpitch;
      // this thread's x rows oh + a0 + ra (tile row = input row + pad);
      // logical chunk 2 ib + m of a row is at pe + 4 (m / 2) for even m,
      // po + 4 (m / 2) for odd m
      const float* pe[RA];
      const float* po[RA];
#pragma unroll
      for (int ra = 0; ra < RA; ++ra) {
        pe[ra] = xs + (oh + a0 + ra) * g.xpitch + 4 * ib;
        po[ra] = pe[ra] + 4 * g.half_e;
      }
      // sliding window: three chunks per row in a ring of slots
      float xw[RA][3][4];
      auto load_chunk = [&](int ra, int slot, int m) {
        const float4 f = *reinterpret_cast<const float4*>(((m & 1) ? po[ra] : pe[ra]) + 4 * (m >> 1));
        xw[ra][slot][0] = f.x; xw[ra][slot][1] = f.y; xw[ra][slot][2] = f.z; xw[ra][slot][3] = f.w;
      };
#pragma unroll
      for (int ra = 0; ra < RA; ++ra) {
        load_chunk(ra, 0, 0);
        load_chunk(ra, 1, 1);
        load_chunk(ra, 2, 2);
      }
      // step s (ow = 4 s) uses chunks s, s+1, s+2 of the window, then loads
      // chunk s+3 into the slot of chunk s. Six steps per iteration make the
      // slot ring (3) and the chunk parity (2) static.
      for (int s0 = 0; s0 < n4; s0 += 6) {
#pragma unroll
        for (int ss = 0; ss < 6; ++ss) {
          const int s = s0 + ss;
          if (s >= n4) break;
          // grad_out values by scalar (broadcast) loads
          const float gg[4] = {grow[4 * s], grow[4 * s + 1], grow[4 * s + 2], grow[4 * s + 3]};
          const int sl0 = ss % 3, sl1 = (ss + 1) % 3, sl2 = (ss + 2) % 3;
#pragma unroll
          for (int ra = 0; ra < RA; ++ra) {
            float wv[12];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              wv[i] = xw[ra][sl0][i];
              wv[4 + i] = xw[ra][sl1][i];
              wv[8 + i] = xw[ra][sl2][i];
            }
            // input-stationary order (each x value shared by consecutive
            // FMAs); every accumulator still adds j = 0..3 in order
#pragma unroll
            for (int m = 0; m < VB + 3; ++m) {
              const float xv = wv[m];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int v = m - j;
                if (v >= 0 && v < VB) acc[ra][v] = fmaf(gg[j], xv, acc[ra][v]);
              }
            }
            // chunk s + 3 of the window (parity of ss + 3 is static)
            const int m = s + 3;
            const float4 f = *reinterpret_cast<const float4*>((((ss + 3) & 1) ? po[ra] : pe[ra]) + 4 * (m >> 1));
            xw[ra][sl0][0] = f.x; xw[ra][sl0][1] = f.y; xw[ra][sl0][2] = f.z; xw[ra][sl0][3] = f.w;
          }
        }
      }
    }
  };
  // end of a unit: fixed-order reduction of the groups' sums (in the
  // consumed fp32 buffer), one partial per (chunk, channel)
  auto finish_unit = [&](int64_t uu, float* red) {
    if (active) {
#pragma unroll
      for (int r = 0; r < RA; ++r)
#pragma unroll
        for (int v = 0; v < VB; ++v) {
          const int a = a0 + r, b = b0 + v;
          if (a < K && b < K) red[grp * (K * K) + a * K + b] = acc[r][v];
        }
    }
#pragma unroll
    for (int r = 0; r < RA; ++r)
#pragma unroll
      for (int v = 0; v < VB; ++v) acc[r][v] = 0.f;
    float bv = bsum;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bv += __shfl_xor_sync(0xffffffffu, bv, o);
    bsum = 0.f;
    float* wred = red + g.G * (K * K);
    if ((tid & 31) == 0) wred[tid >> 5] = bv;
    __syncthreads();
    uint32_t cq;
    const int64_t ch = c.dC.divmod((uint32_t)uu, cq);
    float* dstp = ws + ((int64_t)cq * c.OC() + ch) * (K * K + 1);
    for (int t = tid; t < K * K; t += kNT) {
      float sum = 0.f;
      for (int gi = 0; gi < g.G; ++gi) sum += red[gi * (K * K) + t];
      dstp[t] = sum;
    }
    if (tid == 0) {
      float sum = 0.f;
      for (int wi = 0; wi < kNT / 32; ++wi) sum += wred[wi];
      dstp[K * K] = sum;
    }
    __syncthreads();
  };

  int64_t u = blockIdx.x;
  int sidx = 0;
  if (g.raw16) {
    // one fp32 buffer; the raw area holds the next step's 16-bit planes
    int64_t u1 = u;
    int s1 = sidx;
    if (u < units && unit_ns(u) > 0) issue_raw(unit_n0(u) + sidx, unit_ch(u));
    tile::cp_async_commit();
    tile::cp_async_wait<0>();
    __syncthreads();
    if (u < units && unit_ns(u) > 0) convert(unit_n0(u) + sidx, unit_ch(u), sm);
    __syncthreads();
    next_step(u1, s1);
    if (u1 < units && unit_ns(u1) > 0) issue_raw(unit_n0(u1) + s1, unit_ch(u1));
    tile::cp_async_commit();
    while (u < units) {
      if (unit_ns(u) > 0) compute(sm, sm + g.x_elems);
      int64_t un = u;
      int sn = sidx;
      next_step(un, sn);
      __syncthreads();
      if (un != u) finish_unit(u, sm);
      tile::cp_async_wait<0>();
      __syncthreads();
      if (un < units && unit_ns(un) > 0) {
        convert(unit_n0(un) + sn, unit_ch(un), sm);
        __syncthreads();
        int64_t u2 = un;
        int s2 = sn;
        next_step(u2, s2);
        if (u2 < units && unit_ns(u2) > 0) issue_raw(unit_n0(u2) + s2, unit_ch(u2));
      }
      tile::cp_async_commit();
      u = un;
      sidx = sn;
    }
  } else {
    // two fp32 stages: the next step's copies fly while this one computes
    if (u < units && unit_ns(u) > 0) issue_f32(unit_n0(u), unit_ch(u), sm);
    tile::cp_async_commit();
    for (int k = 0; u < units; ++k) {
      int64_t un = u;
      int sn = sidx;
      next_step(un, sn);
      float* cur = sm + (k & 1) * g.buf_elems;
      if (un < units && unit_ns(un) > 0) issue_f32(unit_n0(un) + sn, unit_ch(un), sm + ((k + 1) & 1) * g.buf_elems);
      tile::cp_async_commit();
      tile::cp_async_wait<1>();
      __syncthreads();
      if (unit_ns(u) > 0) compute(cur, cur + g.x_elems);
      __syncthreads();
      if (un != u) finish_unit(u, cur);
      u = un;
      sidx = sn;
    }
  }
  tile::cp_async_wait<0>();
}

// ---- host planners ----------------------------------------------------------
// Shared-memory plan of the weight gradient (host; also used by the
// support predicate so that a supported shape always launches).
template <int K>
bool plan_wgrad(const Conv& c, int chunks, WLCfg* out_cfg, size_t* smem_out) {
  using Gm = WGeo<K>;
  WLCfg g{};
  g.chunks = chunks;
  g.nb = (int)((c.N + chunks - 1) / chunks);
  g.pad = c.ph;
  g.dtype = c.dtype;
  g.gpitch = (int)((c.Wo + 3) / 4 * 4);
  g.g_elems = (int)c.Ho * g.gpitch;
  const int n4 = g.gpitch / 4;
  // chunks read: up to n4 - 1 + 2 (NB - 1) + 3; and the real input columns
  int nq = n4 + 2 * (Gm::NB - 1) + 3;
  const int need = (int)((c.W + c.pw + 3) / 4);
  if (nq < need) nq = need;
  if ((nq & 1) == 0) ++nq;  // odd: rows four apart start four banks apart
  g.nq = nq;
  g.half_e = (nq + 1) / 2;
  g.xpitch = 4 * nq;
  g.xrows = (int)c.Ho + Gm::NA * Gm::RA - 1;  // rows oh + a for a < NA * RA
  g.x_elems = g.xrows * g.xpitch;
  g.G = kNT / Gm::items;
  const int64_t stage = (int64_t)g.x_elems + g.g_elems;
  const int64_t red = (int64_t)g.G * K * K + kNT / 32;
  int64_t be = stage > red ? stage : red;
  be = (be + 3) / 4 * 4;
  g.buf_elems = (int)be;
  // fp32: two fp32 buffers; 16-bit: one fp32 buffer and a raw area for the
  // next step's two dense 16-bit planes
  g.raw16 = c.dtype != DWCONV_F32;
  g.rawx_elems = tile::dense_seg<unsigned short>(c.H * c.W);
  const int64_t rawg_elems = tile::dense_seg<unsigned short>(c.Ho * c.Wo);
  const size_t smem = g.raw16 ? (size_t)be * 4 + (size_t)(g.rawx_elems + rawg_elems) * 2 : (size_t)2 * be * 4;
  if (smem > 220 * 1024) return false;
  g.d_xrows = FastDiv((uint32_t)g.xrows);
  if (out_cfg) *out_cfg = g;
  if (smem_out) *smem_out = smem;
  return true;
}

template <int K>
cudaError_t run_wgrad_k(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
  WLCfg g;
  size_t smem = 0;
  if (!plan_wgrad<K>(c, chunks, &g, &smem)) return cudaErrorInvalidConfiguration;
  auto kern = wgrad_kernel<K>;
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = tile::persistent_grid(kern, smem, c.C * chunks);
  kern<<<grid, kNT, smem, s>>>(c, g, x, gy, ws);
  return cudaGetLastError();
}

// Weight-gradient kernel per filter size: the packed sample-pair kernel
// (large_pwgrad.cuh) from 13 taps, where it is faster (6-13 % at 13 and 31,
// 10-15 % at 21, 4-7 % at 27 on 32..64-row planes); the scalar kernel above
// below 13 taps.
template <int K>
constexpr bool kPackedWgrad = K >= 13;

// Batch chunks of the scalar weight gradient: about eight (channel, chunk)
// units per resident CTA (two per SM), so the persistent CTAs end close
// together.
inline int scalar_wgrad_chunks(const Conv& c) {
  int64_t chunks = (152 * 2 * 8 + c.C - 1) / c.C;
  if (chunks > c.N) chunks = c.N;
  if (chunks < 1) chunks = 1;
  const int64_t nb = (c.N + chunks - 1) / chunks;
  return (int)(c.N > 0 ? (c.N + nb - 1) / nb : 1);
}

// Per-K entry points: one translation unit per K (large_kNN.cu) defines them
// with this macro; large_entries.h declares them. wgrad_parts_kK is the
// number of partials per channel the weight gradient writes (the second
// pass sums them); the wgrad_scalar_* entries run the scalar kernel over
// sample chunks whatever K is (the fallback of the tensor-core weight
// gradient, which chunks the batch the same way).
#define DW_LARGE_DEFINE(K)                                                                                   \
  cudaError_t fwd_k##K(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,   \
                       const Epi& ep) {                                                                     \
    return run_fwd_k<K>(c, x, w, b, y, false, false, s, ep);                                                \
  }                                                                                                         \
  cudaError_t bwd_k##K(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {  \
    return run_fwd_k<K>(c, gy, w, nullptr, gx, true, acc, s, Epi{});                                        \
  }                                                                                                         \
  cudaError_t wgrad_k##K(const Conv& c, const void* x, const void* gy, float* ws, int parts,               \
                         cudaStream_t s) {                                                                  \
    if constexpr (kPackedWgrad<K>) return run_pwgrad_k<K>(c, x, gy, ws, parts, s);                         \
    else return run_wgrad_k<K>(c, x, gy, ws, parts, s);                                                     \
  }                                                                                                         \
  int wgrad_parts_k##K(const Conv& c) {                                                                     \
    if constexpr (kPackedWgrad<K>) return pwgrad_parts<K>(c);                                               \
    else return scalar_wgrad_chunks(c);                                                                     \
  }                                                                                                         \
  bool wgrad_fits_k##K(const Conv& c) {                                                                     \
    if constexpr (kPackedWgrad<K>) return plan_pwgrad<K>(c, nullptr, nullptr);                              \
    else return plan_wgrad<K>(c, 1, nullptr, nullptr);                                                      \
  }                                                                                                         \
  cudaError_t wgrad_scalar_k##K(const Conv& c, const void* x, const void* gy, float* ws, int chunks,       \
                                cudaStream_t s) {                                                           \
    return run_wgrad_k<K>(c, x, gy, ws, chunks, s);                                                         \
  }                                                                                                         \
  bool wgrad_scalar_fits_k##K(const Conv& c) { return plan_wgrad<K>(c, 1, nullptr, nullptr); }

}  // namespace large
}  // namespace dwconv
