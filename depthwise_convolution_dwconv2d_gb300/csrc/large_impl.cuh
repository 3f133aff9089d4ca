// Large-kernel depthwise convolution on the fp32 FMA pipes (square odd K from
// 7 to 31, stride 1, dilation 1, one filter per channel): the forward and the
// stride-1 grad-input share one correlation kernel; the weight gradient has
// its own.
//
// The MegEngine large-kernel depthwise article ("DirectConv") blocks the
// output at several levels -- CTA tile, warp rows, a few outputs per thread --
// and keeps the kernel and input windows on chip. The same idea on sm_103a:
//  * A CTA stages whole input planes (with their zero halo, widened to fp32)
//    and each plane's filter in shared memory, two stages deep when they fit,
//    so the next planes arrive while the current ones are computed.
//  * Every thread owns two pairs of output rows x 8 columns: rows 2j, 2j+1
//    and the mirror pair counted from the bottom of the plane. Kernel rows
//    that only meet zero padding are skipped, so rows near the top and the
//    bottom cost less; pairing each with its mirror gives every thread the
//    same work, and no warp waits long at the stage barriers.
//  * For each pair the thread walks the kernel rows holding one filter row
//    (K values) in registers and reads each input-row window (8 + K - 1
//    values) with 16-byte loads, so every value read from shared memory
//    feeds 8 * K / (8 + K - 1) fused multiply-adds.
//  * Rows are stored with their 16-byte chunks de-interleaved (even chunks,
//    then odd chunks): windows of neighbouring threads start 32 bytes apart,
//    and in this layout they read consecutive chunks, free of bank conflicts.
//  * Kernel rows whose input rows are zero padding for every thread of a
//    warp are skipped.
// Grad-input at stride 1 is the same computation on grad_out with the filter
// rotated by 180 degrees and padding K-1-pad (the adjoint of the forward).
//
// The storage type (fp32 / fp16 / bf16) only changes how planes are staged
// and outputs stored, so it is a run-time argument: one kernel per K.
#pragma once

#include "plan.h"
#include "tile.cuh"

namespace dwconv {
namespace large {

constexpr int kNT = 256;
constexpr int kV = 8;  // output columns per thread (forward / grad-input)

// Physical chunk of logical 16-byte chunk q in a row whose even chunks come
// first (half_e = number of even chunks).
__host__ __device__ __forceinline__ int phys_chunk(int q, int half_e) {
  return (q & 1) ? half_e + (q >> 1) : (q >> 1);
}

__device__ __forceinline__ float ld_any(const void* p, int64_t i, int dtype) {
  if (dtype == DWCONV_F32) return __ldg(reinterpret_cast<const float*>(p) + i);
  if (dtype == DWCONV_F16) return __half2float(__ldg(reinterpret_cast<const __half*>(p) + i));
  return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(p) + i));
}

__device__ __forceinline__ float ld_rw_any(const void* p, int64_t i, int dtype) {
  if (dtype == DWCONV_F32) return reinterpret_cast<const float*>(p)[i];
  if (dtype == DWCONV_F16) return __half2float(reinterpret_cast<const __half*>(p)[i]);
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
}

__device__ __forceinline__ void st_any(void* p, int64_t i, float v, int dtype) {
  if (dtype == DWCONV_F32) reinterpret_cast<float*>(p)[i] = v;
  else if (dtype == DWCONV_F16) reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
  else reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

// Stage rows [0, tr) x logical columns [0, 4 nq) of np planes: tile row r,
// column t hold input element (r - pad, t - pad) of plane p (zero outside);
// rows in the de-interleaved chunk layout, planes plane_elems floats apart.
// A warp stages whole rows, its lanes sweeping the columns (coalesced reads).
// Lane l covers columns l + 32 k, which lie in chunks (l >> 2) + 8 k: all of
// one parity, so a lane's destinations are a per-lane base plus 16 k floats.
// fp32 data is copied asynchronously (cp.async with zero fill); 16-bit data
// is widened through registers.
template <typename SrcOf>
__device__ __forceinline__ void stage_planes(float* dst, int np, int plane_elems, int tr, int nq, int half_e,
                                             const FastDiv& d_tr, SrcOf src_of, int Hin, int Win, int pad,
                                             int dtype, bool async4) {
  const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int pitch = 4 * nq;
  const int q0 = lane >> 2;
  const int lane_off = 4 * phys_chunk(q0, half_e) + (lane & 3);
  for (int row = threadIdx.x >> 5; row < np * tr; row += nw) {
    uint32_t p;
    const int r = (int)d_tr.divmod((uint32_t)row, p);
    const int iy = r - pad;
    const bool rin = iy >= 0 && iy < Hin;
    float* d = dst + (int)p * plane_elems + r * pitch + lane_off;
    const char* srow = reinterpret_cast<const char*>(src_of((int)p));
    const int64_t ro = (int64_t)(rin ? iy : 0) * Win;
    for (int col = lane; col < pitch; col += 32, d += 16) {
      const int ix = col - pad;
      const bool in = rin && ix >= 0 && ix < Win;
      if (async4) {
        const float* sp = reinterpret_cast<const float*>(srow) + (in ? ro + ix : 0);
        tile::cp_async4(d, sp, in ? 4 : 0);
      } else {
        *d = in ? ld_any(srow, ro + ix, dtype) : 0.f;
      }
    }
  }
}

// ---- forward / stride-1 grad-input ----------------------------------------
struct LCfg {
  int ppc;               // planes per unit
  int nq, half_e, pitch; // chunks per staged row, even chunks, floats per row
  int tr;                // staged rows per plane (rb * R + K - 1)
  int tile_elems;        // floats per staged plane (tile + filter)
  int wofs;              // filter offset inside a staged plane
  int rb, cb;            // row blocks / column blocks per plane
  int pad;               // padding of the correlation as evaluated
  int Hin, Win, Hout, Wout;
  int flip;              // grad-input: read grad_out, rotate the filter, write gx
  int dtype, async4, acc, stages;
  int stage_elems;       // floats per stage
  int64_t units;
  FastDiv d_tr;
};

template <int K, int R>
__global__ void __launch_bounds__(kNT, 2)
dconv_kernel(Conv c, LCfg g, const void* __restrict__ in, const void* __restrict__ w,
             const void* __restrict__ bias, void* out, Epi ep) {
  extern __shared__ __align__(16) float sm[];
  constexpr int KP = (K + 3) / 4 * 4;          // filter row stride (16-byte rows)
  constexpr int NCH = (kV + K - 1 + 3) / 4;    // window chunks per input row
  const int tid = threadIdx.x, nt = blockDim.x;
  const int64_t nplanes = c.N * c.C;
  const int es = g.dtype == DWCONV_F32 ? 4 : 2;
  auto issue = [&](int64_t u, float* dst) {
    const int64_t p0 = u * g.ppc;
    const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
    stage_planes(dst, np, g.tile_elems, g.tr, g.nq, g.half_e, g.d_tr,
                 [&](int p) -> const void* {
                   int64_t n, ch;
                   c.split(p0 + p, n, ch);
                   const int64_t base = g.flip ? c.y_base(n, ch) : c.x_base(n, ch);
                   return reinterpret_cast<const char*>(in) + base * es;
                 },
                 g.Hin, g.Win, g.pad, g.dtype, g.async4 != 0);
    // each plane's filter (rotated for the grad-input), rows padded to KP
    for (int p = 0; p < np; ++p) {
      int64_t n_, ch;
      c.split(p0 + p, n_, ch);
      float* fd = dst + p * g.tile_elems + g.wofs;
      for (int t = tid; t < K * KP; t += nt) {
        const int a = t / KP, b = t - a * KP;
        const int src_t = g.flip ? (K * K - 1 - (a * K + b)) : (a * K + b);
        fd[t] = b < K ? ld_any(w, ch * (K * K) + src_t, g.dtype) : 0.f;
      }
    }
  };

  int stage = 0;
  int64_t u = blockIdx.x;
  if (u < g.units) issue(u, sm);
  tile::cp_async_commit();
  for (; u < g.units; u += gridDim.x) {
    const int64_t un = u + gridDim.x;
    float* cur = sm + stage * g.stage_elems;
    if (g.stages == 2) {
      if (un < g.units) issue(un, sm + (stage ^ 1) * g.stage_elems);
      tile::cp_async_commit();
      tile::cp_async_wait<1>();
    } else {
      tile::cp_async_wait<0>();
    }
    __syncthreads();

    const int64_t p0 = u * g.ppc;
    const int np = (int)((nplanes - p0) < g.ppc ? (nplanes - p0) : g.ppc);
    const int per_rb = np * g.cb;
    const int nitems = per_rb * g.rb;
    // items ordered (row block, plane, column block): the lanes of a warp
    // share output rows, so they walk the same kernel rows
    for (int it = tid; it < nitems; it += nt) {
      const int rbi = it / per_rb;
      const int rem = it - rbi * per_rb;
      const int pl = rem / g.cb;
      const int cbi = rem - pl * g.cb;
      const float* t = cur + pl * g.tile_elems;
      const float* wt = t + g.wofs;
      const int oh0 = rbi * R, ow0 = cbi * kV;
      int64_t n_, ch_;
      c.split(p0 + pl, n_, ch_);
      const float bv = bias ? ld_any(bias, ch_, g.dtype) : 0.f;
      float acc[R][kV];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int v = 0; v < kV; ++v) acc[r][v] = bv;
      // kernel rows that reach a real input row for some output row of the
      // warp (the others read zero padding rows of the tile); the warp's
      // items are it - lane .. it - lane + 31, so the bounds are uniform
      const int it0 = it - (tid & 31);
      const int it1 = (it0 + 31) < (nitems - 1) ? (it0 + 31) : (nitems - 1);
      const int oh_first = (it0 / per_rb) * R, oh_last = (it1 / per_rb) * R;
      int a_lo = g.pad - oh_last - (R - 1);
      a_lo = a_lo < 0 ? 0 : a_lo;
      int a_hi = g.Hin + g.pad - oh_first;
      a_hi = a_hi > K ? K : a_hi;
      const float* colbase = t + 4 * cbi;  // even chunks of this thread's window
      for (int a = a_lo; a < a_hi; ++a) {
        // filter taps by scalar (broadcast) loads
        float wr[K];
#pragma unroll
        for (int b = 0; b < K; ++b) wr[b] = wt[a * KP + b];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float* pe = colbase + (oh0 + r + a) * g.pitch;
          const float* po = pe + 4 * g.half_e;
          float win[4 * NCH];
#pragma unroll
          for (int q = 0; q < NCH; ++q) {
            const float4 f = *reinterpret_cast<const float4*>(((q & 1) ? po : pe) + 4 * (q >> 1));
            win[4 * q] = f.x; win[4 * q + 1] = f.y; win[4 * q + 2] = f.z; win[4 * q + 3] = f.w;
          }
          // input-stationary order: each window value is the operand shared
          // by the (up to 8) consecutive FMAs that use it; every accumulator
          // still sums its taps in increasing filter column order
#pragma unroll
          for (int j = 0; j < kV + K - 1; ++j) {
            const float xv = win[j];
#pragma unroll
            for (int v = 0; v < kV; ++v) {
              const int b = j - v;
              if (b >= 0 && b < K) acc[r][v] = fmaf(wr[b], xv, acc[r][v]);
            }
          }
        }
      }
      if (ep.active()) {
        const float sc = ep.scale ? ld_any(ep.scale, ch_, g.dtype) : 1.f;
        const float sh = ep.shift ? ld_any(ep.shift, ch_, g.dtype) : 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int v = 0; v < kV; ++v) acc[r][v] = epi_act(fmaf(acc[r][v], sc, sh), ep.act);
      }
      const int64_t ob = g.flip ? c.x_base(n_, ch_) : c.y_base(n_, ch_);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int oh = oh0 + r;
        if (oh >= g.Hout) break;
        const int64_t o = ob + (int64_t)oh * g.Wout + ow0;
        if (g.dtype == DWCONV_F32 && !g.acc && ow0 + kV <= g.Wout &&
            (reinterpret_cast<uintptr_t>(reinterpret_cast<float*>(out) + o) & 15) == 0) {
          float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + o);
          d[0] = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
          d[1] = make_float4(acc[r][4], acc[r][5], acc[r][6], acc[r][7]);
        } else {
#pragma unroll
          for (int v = 0; v < kV; ++v)
            if (ow0 + v < g.Wout) {
              const float val = g.acc ? acc[r][v] + ld_rw_any(out, o + v, g.dtype) : acc[r][v];
              st_any(out, o + v, val, g.dtype);
            }
        }
      }
    }
    __syncthreads();
    if (g.stages == 1) {
      if (un < g.units) issue(un, sm);
      tile::cp_async_commit();
    } else {
      stage ^= 1;
    }
  }
  tile::cp_async_wait<0>();
}

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
// Forward plan for R output rows per thread: the staged plane (rows
// rb * R + K - 1 of 4 * nq floats plus the filter), planes per unit, stages
// and threads per CTA (the items of a unit, rounded up to whole warps, at
// most 256).
template <int K, int R>
bool plan_dconv(const Conv& c, bool flip, LCfg* out_cfg, int* threads) {
  constexpr int KP = (K + 3) / 4 * 4;
  constexpr int NCH = (kV + K - 1 + 3) / 4;
  LCfg g{};
  g.flip = flip;
  g.dtype = c.dtype;
  g.Hin = (int)(flip ? c.Ho : c.H);
  g.Win = (int)(flip ? c.Wo : c.W);
  g.Hout = (int)(flip ? c.H : c.Ho);
  g.Wout = (int)(flip ? c.W : c.Wo);
  g.pad = flip ? K - 1 - c.ph : c.ph;
  g.cb = (g.Wout + kV - 1) / kV;
  g.rb = (g.Hout + R - 1) / R;
  // chunks per row: every window of every column block, and the real
  // columns of the input (the rest of a row is zero)
  int nq = 2 * (g.cb - 1) + NCH;
  const int need = (g.Win + g.pad + 3) / 4;
  if (nq < need) nq = need;
  g.tr = g.rb * R + K - 1;
  const int64_t ipp = (int64_t)g.rb * g.cb;
  int64_t ppc = (kNT + ipp - 1) / ipp;
  if (ppc < 1) ppc = 1;
  int te = 0;
  auto layout = [&]() {
    g.nq = nq;
    g.half_e = (nq + 1) / 2;
    g.pitch = 4 * nq;
    g.wofs = g.tr * g.pitch;
    te = (g.wofs + K * KP + 3) / 4 * 4;
  };
  layout();
  if (g.cb < 8 && ppc == 1) {
    // A quarter-warp (8 lanes) spans several row blocks of cb column blocks:
    // starting each row block cb chunks further in the bank space keeps its
    // 16-byte loads on distinct banks (R * nq reaches only some residues:
    // try at most eight widths)
    for (int extra = 0; extra < 8; ++extra)
      if (((R * (nq + extra)) & 7) == (g.cb & 7)) {
        nq += extra;
        layout();
        break;
      }
  }
  const int64_t two_cta = 110 * 1024;  // per CTA, for two CTAs on an SM
  auto plane_bytes = [&]() { return (int64_t)te * 4; };
  int64_t cap1 = two_cta / plane_bytes();
  if (cap1 < 1) cap1 = (210 * 1024) / plane_bytes();
  if (cap1 < 1) return false;
  if (ppc > cap1) ppc = cap1;
  if (g.cb < 8 && ppc > 1) {
    // planes cb chunks apart in the bank space, as above
    while (((te / 4) & 7) != (g.cb & 7)) te += 4;
  }
  g.tile_elems = te;
  g.stages = (2 * ppc * plane_bytes() <= two_cta) ? 2 : 1;
  g.ppc = (int)ppc;
  g.stage_elems = (int)(ppc * te);
  g.units = (c.N * c.C + ppc - 1) / ppc;
  g.d_tr = FastDiv((uint32_t)g.tr);
  int64_t items = ppc * ipp;
  if (items > kNT) items = kNT;
  if (out_cfg) *out_cfg = g;
  if (threads) *threads = (int)((items + 31) / 32 * 32);
  return true;
}

template <int K, int R>
cudaError_t launch_dconv(const Conv& c, const LCfg& g0, int threads, const void* in, const void* w,
                         const void* bias, void* out, bool acc, cudaStream_t s, const Epi& ep) {
  LCfg g = g0;
  g.acc = acc;
  g.async4 = (c.dtype == DWCONV_F32) ? 1 : 0;  // fp32 pointers are 4-byte aligned
  auto kern = dconv_kernel<K, R>;
  const size_t smem = (size_t)g.stages * g.stage_elems * 4;
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 152, per_sm = 1;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t cap = (int64_t)sms * per_sm;
  const int grid = (int)(g.units < cap ? g.units : cap);
  kern<<<grid, threads, smem, s>>>(c, g, in, w, bias, out, ep);
  return cudaGetLastError();
}

// Rows per thread: the plan whose unit keeps the most thread slots busy, then
// the one with two stages, then four rows (fewer filter-row loads).
template <int K>
cudaError_t run_fwd_k(const Conv& c, const void* in, const void* w, const void* bias, void* out, bool flip,
                      bool acc, cudaStream_t s, const Epi& ep) {
  LCfg g2, g4;
  int t2 = 0, t4 = 0;
  const bool ok2 = plan_dconv<K, 2>(c, flip, &g2, &t2);
  const bool ok4 = plan_dconv<K, 4>(c, flip, &g4, &t4);
  if (!ok2 && !ok4) return cudaErrorInvalidConfiguration;
  // busy fraction of a full CTA's thread slots (a smaller CTA leaves the SM
  // fewer warps)
  auto fill = [&](const LCfg& g, int t) {
    const int64_t items = (int64_t)g.ppc * g.rb * g.cb;
    const int64_t rounds = (items + t - 1) / t;
    return (double)items / (double)(rounds * kNT);
  };
  bool use4 = ok4;
  if (ok2 && ok4) {
    const double f2 = fill(g2, t2), f4 = fill(g4, t4);
    if (f2 > f4 + 0.05) use4 = false;
    else if (f4 > f2 + 0.05) use4 = true;
    else use4 = !(g2.stages == 2 && g4.stages == 1);
  } else {
    use4 = !ok2;
  }
  if (use4) return launch_dconv<K, 4>(c, g4, t4, in, w, bias, out, acc, s, ep);
  return launch_dconv<K, 2>(c, g2, t2, in, w, bias, out, acc, s, ep);
}

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

// Per-K entry points: one translation unit per K (large_kNN.cu) defines them
// with this macro; large_entries.h declares them.
#define DW_LARGE_DEFINE(K)                                                                                   \
  cudaError_t fwd_k##K(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,   \
                       const Epi& ep) {                                                                     \
    return run_fwd_k<K>(c, x, w, b, y, false, false, s, ep);                                                \
  }                                                                                                         \
  cudaError_t bwd_k##K(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {  \
    return run_fwd_k<K>(c, gy, w, nullptr, gx, true, acc, s, Epi{});                                        \
  }                                                                                                         \
  cudaError_t wgrad_k##K(const Conv& c, const void* x, const void* gy, float* ws, int chunks,              \
                         cudaStream_t s) {                                                                  \
    return run_wgrad_k<K>(c, x, gy, ws, chunks, s);                                                         \
  }                                                                                                         \
  bool wgrad_fits_k##K(const Conv& c) { return plan_wgrad<K>(c, 1, nullptr, nullptr); }

}  // namespace large
}  // namespace dwconv
