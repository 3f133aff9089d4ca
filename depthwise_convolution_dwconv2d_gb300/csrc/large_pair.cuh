// Large-kernel depthwise forward and stride-1 grad-input on packed fp32x2
// fused multiply-adds (square odd K from 7 to 31, stride 1, dilation 1, one
// filter per channel).
//
// The MegEngine large-kernel depthwise article ("DirectConv") blocks the
// output at several levels -- CTA tile, rows, a run of outputs per thread --
// and keeps the filter and input windows on chip. On sm_103a the FP32 pipes
// also take a two-lane instruction (fma.rn.f32x2: two independent IEEE fused
// multiply-adds in one issue slot), and the blocking here is built around it:
//  * A thread computes the same block of outputs -- one output row, V = 8 or
//    16 consecutive columns -- for two planes at once. The two planes of a
//    plane pair are staged interleaved (float2: plane 0, plane 1), so every
//    input value, filter tap and accumulator is a ready-made 64-bit lane pair
//    and one filter tap feeds V packed FMAs. With scalar FMAs this loop is
//    bound by instruction issue; packed, it needs half the issue slots and
//    the FP32 pipe becomes the limit. Each lane of a pair rounds exactly like
//    fmaf; every output adds its taps in (filter row, filter column) order
//    and its bias last.
//  * The filter rows an output row needs are those whose input row is real,
//    a in [max(0, pad - oh), min(K, H + pad - oh)): every lane loops over
//    its own range, so zero-padding rows are never multiplied. The rows of a
//    plane are handed to the lanes in mirror order (0, H-1, 1, H-2, ...): a
//    row and its mirror have ranges of equal length, so the lanes of a warp
//    run nearly equal trip counts.
//  * Per filter row a thread loads the filter row (two taps per 16-byte
//    load) and the input window (V + K - 1 pairs, two per 16-byte load) in
//    the order they are consumed; each window pair then feeds up to V packed
//    FMAs from registers.
//  * Staged rows carry a 16-byte gap after every V pairs, so the windows of
//    neighbouring column blocks start in different shared-memory bank
//    groups; the row and plane-pair strides are padded by the host planner,
//    which simulates the bank groups of every quarter-warp's loads.
//  * A CTA owns units of (plane pairs, band of output rows) in a persistent
//    loop. A unit's input band (with its zero halo, widened to fp32) and its
//    filters are copied in with cp.async, two stages deep when they fit, else
//    one stage with two CTAs per SM taking turns.
// Grad-input at stride 1 is the same computation on grad_out with the filter
// rotated by 180 degrees and padding K - 1 - pad (the adjoint of the forward).
#pragma once

#include <cstdio>
#include <cstdlib>

#include "large_common.cuh"

namespace dwconv {
namespace large {

typedef f32x2 u64;

// d = w * x + d on both 32-bit lanes of the 64-bit operands.
__device__ __forceinline__ void fma2(u64& d, u64 w, u64 x) { fma_f32x2(d, w, x); }
__device__ __forceinline__ void unpack2(u64 v, float& lo, float& hi) { unpack_f32x2(v, lo, hi); }

// Physical pair index of logical pair column q in a staged row: a 16-byte
// gap (two pairs) after every V pairs.
template <int V>
__host__ __device__ __forceinline__ int pphys(int q) {
  return q + 2 * (q / V);
}

// Filter row stride in pairs: K taps plus a zero slot, in whole 16-byte
// chunks, with an odd number of chunks so that consecutive filter rows start
// in different bank groups.
template <int K>
struct FiltGeo {
  static constexpr int kp0 = (K + 2) / 2 * 2;
  static constexpr int KP2 = ((kp0 / 2) % 2 == 0) ? kp0 + 2 : kp0;
};

struct PCfg {
  int ppu;             // plane pairs per unit
  int bo, nbands;      // output rows per band, bands per plane
  int tr, cols, rs;    // staged rows per band, staged logical pair columns, row stride (pairs)
  int fofs;            // filter table offset in a plane-pair block (pairs)
  int blk;             // pairs per plane-pair block
  int stage_elems;     // pairs per stage
  int cb;              // column blocks of V outputs
  int items;           // items per unit (ppu * bo * cb)
  int mirror;          // rows in mirror order (whole plane in one band)
  int pad, Hin, Win, Hout, Wout;
  int flip, dtype, acc, stages;
  int64_t npairs, units;
  FastDiv d_bands, d_tr, d_cb, d_ppu;
};

// Band row handled by slot s of a band of `rows` rows.
__host__ __device__ __forceinline__ int slot_row(int s, int rows, int mirror) {
  if (!mirror) return s;
  return (s & 1) ? rows - 1 - (s >> 1) : (s >> 1);
}

// One filter row: acc[v] += w[b] * x[v + b] over b ascending, for the V
// outputs of the block on both planes. wr: the filter row (16-byte chunks,
// two taps each); xr: the window's first chunk (two input pairs per chunk,
// a gap chunk after every V / 2 chunks).
template <int K, int V>
__device__ __forceinline__ void tap_row(u64 (&acc)[V], const ulonglong2* __restrict__ wr,
                                        const ulonglong2* __restrict__ xr) {
  constexpr int NWP = V + K - 1;  // window pairs (even: V even, K odd)
  constexpr int NCH = NWP / 2;
  u64 xw[NWP];
  u64 wv[K + 1];
#pragma unroll
  for (int s = 0; s < V / 2; ++s) {
    const ulonglong2 t = xr[s + s / (V / 2)];
    xw[2 * s] = t.x;
    xw[2 * s + 1] = t.y;
  }
#pragma unroll
  for (int b = 0; b < K; ++b) {
    if ((b & 1) == 0) {
      const ulonglong2 t = wr[b >> 1];
      wv[b] = t.x;
      wv[b + 1] = t.y;
    } else {
      // pairs b + V - 1 and b + V are first needed at taps b and b + 1
      const int s = (b + V - 1) >> 1;
      if (s < NCH) {
        const ulonglong2 t = xr[s + s / (V / 2)];
        xw[2 * s] = t.x;
        xw[2 * s + 1] = t.y;
      }
    }
#pragma unroll
    for (int v = 0; v < V; ++v) fma2(acc[v], wv[b], xw[v + b]);
  }
}

template <int K, int V>
__global__ void __launch_bounds__(kNT, 2)
pconv_kernel(Conv c, PCfg g, const void* __restrict__ in, const void* __restrict__ w,
             const void* __restrict__ bias, void* out, Epi ep) {
  extern __shared__ __align__(16) float2 smp[];
  constexpr int KP2 = FiltGeo<K>::KP2;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, nw = nt >> 5;
  const int64_t nplanes = c.N * c.C;
  const int es = g.dtype == DWCONV_F32 ? 4 : 2;
  const bool f32 = g.dtype == DWCONV_F32;

  auto split_unit = [&](int64_t u, int64_t& pp0, int& band) {
    uint32_t q;
    band = (int)g.d_bands.divmod((uint32_t)u, q);
    pp0 = (int64_t)q * g.ppu;
  };

  // Copy unit u's input band and filters into the stage at dst (fp32 by
  // cp.async with zero fill, 16-bit widened through registers).
  auto issue = [&](int64_t u, float2* dst) {
    int64_t pp0;
    int band;
    split_unit(u, pp0, band);
    const int npp = (int)((g.npairs - pp0) < g.ppu ? (g.npairs - pp0) : g.ppu);
    const int iy0 = band * g.bo - g.pad;  // input row of staged row 0
    // input rows: a warp per (plane pair, plane, row), its lanes over columns
    const int nrows = npp * 2 * g.tr;
    for (int t = tid >> 5; t < nrows; t += nw) {
      uint32_t ph;
      const int r = (int)g.d_tr.divmod((uint32_t)t, ph);
      const int pp = (int)(ph >> 1), h = (int)(ph & 1);
      const int64_t p = 2 * (pp0 + pp) + h;
      const int iy = iy0 + r;
      const bool rin = p < nplanes && iy >= 0 && iy < g.Hin;
      int64_t pb = 0;
      if (rin) {
        int64_t n, ch;
        c.split(p, n, ch);
        pb = (g.flip ? c.y_base(n, ch) : c.x_base(n, ch)) + (int64_t)iy * g.Win;
      }
      const char* srow = reinterpret_cast<const char*>(in) + pb * es;
      float* drow = reinterpret_cast<float*>(dst + pp * g.blk + r * g.rs) + h;
      for (int col = lane; col < g.cols; col += 32) {
        const int ix = col - g.pad;
        const bool ok = rin && ix >= 0 && ix < g.Win;
        float* d = drow + 2 * pphys<V>(col);
        if (f32) tile::cp_async4(d, reinterpret_cast<const float*>(srow) + (ok ? ix : 0), ok ? 4 : 0);
        else *d = ok ? ld_any(srow, ix, g.dtype) : 0.f;
      }
    }
    // filters: pair (a, b) = taps (a, b) of both planes' filters (rotated
    // for the grad-input), zero past the last tap and for a missing plane
    const int nf = npp * 2 * K * KP2;
    for (int t = tid; t < nf; t += nt) {
      const int b = t % KP2;
      const int r1 = t / KP2;
      const int a = r1 % K;
      const int ph = r1 / K;
      const int pp = ph >> 1, h = ph & 1;
      const int64_t p = 2 * (pp0 + pp) + h;
      const bool ok = b < K && p < nplanes;
      int64_t wi = 0;
      if (ok) {
        int64_t n, ch;
        c.split(p, n, ch);
        const int tap = g.flip ? (K * K - 1 - (a * K + b)) : (a * K + b);
        wi = ch * (K * K) + tap;
      }
      float* d = reinterpret_cast<float*>(dst + pp * g.blk + g.fofs + a * KP2 + b) + h;
      if (f32) tile::cp_async4(d, reinterpret_cast<const float*>(w) + wi, ok ? 4 : 0);
      else *d = ok ? ld_any(w, wi, g.dtype) : 0.f;
    }
  };

  int stage = 0;
  int64_t u = blockIdx.x;
  if (u < g.units) issue(u, smp);
  tile::cp_async_commit();
  for (; u < g.units; u += gridDim.x) {
    const int64_t un = u + gridDim.x;
    float2* cur = smp + stage * g.stage_elems;
    if (g.stages == 2) {
      if (un < g.units) issue(un, smp + (stage ^ 1) * g.stage_elems);
      tile::cp_async_commit();
      tile::cp_async_wait<1>();
    } else {
      tile::cp_async_wait<0>();
    }
    __syncthreads();

    int64_t pp0;
    int band;
    split_unit(u, pp0, band);
    const int rows = (g.Hout - band * g.bo) < g.bo ? (g.Hout - band * g.bo) : g.bo;
    // items ordered (slot, plane pair, column block): the lanes of a warp
    // hold few distinct rows, and rows of equal range length sit together
    for (int it = tid; it < g.items; it += nt) {
      uint32_t cbi, pp, slot;
      const uint32_t rest = g.d_cb.divmod((uint32_t)it, slot);  // slot = it / cb, rest = it % cb
      cbi = rest;
      pp = g.d_ppu.divmod(slot, slot);                            // pp = slot % ppu, slot /= ppu
      const int64_t p0 = 2 * (pp0 + (int64_t)pp);
      if (p0 >= nplanes || (int)slot >= rows) continue;
      const int ohr = slot_row((int)slot, rows, g.mirror);
      const int oh = band * g.bo + ohr;
      int a_lo = g.pad - oh;
      a_lo = a_lo < 0 ? 0 : a_lo;
      int a_hi = g.Hin + g.pad - oh;
      a_hi = a_hi > K ? K : a_hi;
      u64 acc[V];
#pragma unroll
      for (int v = 0; v < V; ++v) acc[v] = 0ull;
      const float2* blk = cur + pp * g.blk;
      const float2* xbase = blk + ohr * g.rs + (V + 2) * (int)cbi;
      const float2* fbase = blk + g.fofs;
      for (int a = a_lo; a < a_hi; ++a)
        tap_row<K, V>(acc, reinterpret_cast<const ulonglong2*>(fbase + a * KP2),
                      reinterpret_cast<const ulonglong2*>(xbase + a * g.rs));
      // bias, epilogue and store, plane by plane
      const int ow0 = V * (int)cbi;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t p = p0 + h;
        if (p >= nplanes) break;
        int64_t n, ch;
        c.split(p, n, ch);
        float o[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
          float lo, hi;
          unpack2(acc[v], lo, hi);
          o[v] = h ? hi : lo;
        }
        if (bias) {
          const float bv = ld_any(bias, ch, g.dtype);
#pragma unroll
          for (int v = 0; v < V; ++v) o[v] += bv;
        }
        if (ep.active()) {
          const float sc = ep.scale ? ld_any(ep.scale, ch, g.dtype) : 1.f;
          const float sh = ep.shift ? ld_any(ep.shift, ch, g.dtype) : 0.f;
#pragma unroll
          for (int v = 0; v < V; ++v) o[v] = epi_act(fmaf(o[v], sc, sh), ep.act);
        }
        const int64_t ob = (g.flip ? c.x_base(n, ch) : c.y_base(n, ch)) + (int64_t)oh * g.Wout + ow0;
        if (f32 && !g.acc && ow0 + V <= g.Wout &&
            (reinterpret_cast<uintptr_t>(reinterpret_cast<float*>(out) + ob) & 15) == 0) {
          float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + ob);
#pragma unroll
          for (int q = 0; q < V / 4; ++q) d[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        } else {
#pragma unroll
          for (int v = 0; v < V; ++v)
            if (ow0 + v < g.Wout) {
              const float val = g.acc ? o[v] + ld_rw_any(out, ob + v, g.dtype) : o[v];
              st_any(out, ob + v, val, g.dtype);
            }
        }
      }
    }
    __syncthreads();
    if (g.stages == 1) {
      if (un < g.units) issue(un, smp);
      tile::cp_async_commit();
    } else {
      stage ^= 1;
    }
  }
  tile::cp_async_wait<0>();
}

// ---- host planner -----------------------------------------------------------
// Bank-group conflict degree of the first window and filter loads of the
// CTA's first quarter-warps (the lanes' later loads keep the same offsets
// from one another): per quarter-warp, the most distinct 16-byte chunks that
// fall in one bank group, summed.
template <int K, int V>
int pair_conflicts(const PCfg& g, int threads) {
  constexpr int KP2 = FiltGeo<K>::KP2;
  const int rows = g.bo < g.Hout ? g.bo : g.Hout;
  const int lanes = threads < 128 ? threads : 128;
  int total = 0;
  for (int q0 = 0; q0 < lanes; q0 += 8) {
    int wq[8], fq[8], n = 0;
    for (int l = 0; l < 8; ++l) {
      const int it = q0 + l;
      if (it >= g.items) break;
      const int cbi = it % g.cb, slot0 = it / g.cb, pp = slot0 % g.ppu, slot = slot0 / g.ppu;
      if (slot >= rows) break;
      const int ohr = slot_row(slot, rows, g.mirror);
      int a_lo = g.pad - ohr;  // first band
      a_lo = a_lo < 0 ? 0 : a_lo;
      wq[n] = (pp * g.blk + (ohr + a_lo) * g.rs + (V + 2) * cbi) / 2;
      fq[n] = (pp * g.blk + g.fofs + a_lo * KP2) / 2;
      ++n;
    }
    for (int pass = 0; pass < 2; ++pass) {
      const int* q = pass ? fq : wq;
      int cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      for (int i = 0; i < n; ++i) {
        bool dup = false;
        for (int j = 0; j < i; ++j) dup |= q[j] == q[i];
        if (!dup) ++cnt[q[i] & 7];
      }
      int worst = 0;
      for (int b = 0; b < 8; ++b) worst = cnt[b] > worst ? cnt[b] : worst;
      total += worst;
    }
  }
  return total;
}

// Share of the filter-row iterations a unit's warps issue that some lane
// needs: a warp runs as many iterations as its longest lane.
template <int K>
double pair_rowfill(const PCfg& g, int threads) {
  double need = 0.0, run = 0.0;
  for (int band = 0; band < g.nbands; ++band) {
    const int rows = (g.Hout - band * g.bo) < g.bo ? (g.Hout - band * g.bo) : g.bo;
    for (int w0 = 0; w0 < g.items; w0 += 32) {
      int most = 0, active = 0;
      for (int it = w0; it < w0 + 32 && it < g.items; ++it) {
        const int slot = it / g.cb / g.ppu;
        if (slot >= rows) continue;
        const int oh = band * g.bo + slot_row(slot, rows, g.mirror);
        int lo = g.pad - oh, hi = g.Hin + g.pad - oh;
        lo = lo < 0 ? 0 : lo;
        hi = hi > K ? K : hi;
        const int n = hi > lo ? hi - lo : 0;
        need += n;
        most = n > most ? n : most;
        ++active;
      }
      run += 32.0 * most;
      (void)active;
    }
    if (band >= 2 && band + 2 < g.nbands) band = g.nbands - 3;  // interior bands repeat band 1
  }
  (void)threads;
  return run > 0 ? need / run : 1.0;
}

// Strides of a plan with row and block padding (pairs, even).
template <int K>
void pair_strides(PCfg& t, int rs0, int rpad, int bpad) {
  constexpr int KP2 = FiltGeo<K>::KP2;
  t.rs = rs0 + rpad;
  t.fofs = t.tr * t.rs;
  t.blk = (t.fofs + K * KP2 + bpad + 1) / 2 * 2;
  t.stage_elems = t.ppu * t.blk;
}

// Plan for output blocks of V columns: bands, plane pairs per unit, stages,
// strides. Returns false if not even one plane-pair band fits.
// A plan may be pinned (force_bo / force_ppu / force_stages > 0) for tuning.
template <int K, int V>
bool plan_pair(const Conv& c, bool flip, PCfg* out_cfg, int* threads_out, double* score_out,
               int force_bo = 0, int force_ppu = 0, int force_stages = 0) {
  PCfg g{};
  g.flip = flip;
  g.dtype = c.dtype;
  g.Hin = (int)(flip ? c.Ho : c.H);
  g.Win = (int)(flip ? c.Wo : c.W);
  g.Hout = (int)(flip ? c.H : c.Ho);
  g.Wout = (int)(flip ? c.W : c.Wo);
  g.pad = flip ? K - 1 - c.ph : c.ph;
  g.cb = (g.Wout + V - 1) / V;
  int cols = g.cb * V + K - 1;  // the last block's window ends at column cols - 1
  if (cols < g.Win + g.pad) cols = g.Win + g.pad;
  cols = (cols + 1) / 2 * 2;
  g.cols = cols;
  const int rs0 = (pphys<V>(cols - 1) + 2) / 2 * 2;
  g.npairs = (c.N * c.C + 1) / 2;
  const int64_t sm_bytes = 228 * 1024;  // shared memory per SM
  const int64_t cta_max = 227 * 1024;   // per CTA
  double best = -1.0;
  PCfg bestg{};
  int best_threads = 0;
  // Measured on the 64 x 384 large-kernel layers (every band height, plane
  // pairs per unit and stage count): the whole plane as one band, one stage
  // with two CTAs per SM taking turns (a second stage where it still leaves
  // two CTAs per SM), and enough plane pairs per unit for about 256 threads.
  // Bands of rows are used only where one plane pair does not fit half an SM.
  const int64_t half_sm = sm_bytes / 2 - 1024;
  int bos[32], nbo = 0;
  if (force_bo > 0) bos[nbo++] = force_bo < g.Hout ? force_bo : g.Hout;
  else
    for (int bo = g.Hout; bo >= 1 && nbo < 32; bo = (bo > 8 ? (bo + 1) / 2 : 0)) bos[nbo++] = bo;
  // first pass: units that leave room for two CTAs per SM; second pass (only
  // if nothing fits that way): one CTA per SM
  for (int pass = 0; pass < 2 * nbo && best < 0; ++pass) {
    const int bi = pass % nbo;
    const int64_t limit = pass < nbo ? half_sm : cta_max - 1024;
    const int bo = bos[bi];
    PCfg t = g;
    t.bo = bo;
    t.nbands = (g.Hout + bo - 1) / bo;
    t.mirror = t.nbands == 1;
    t.tr = bo + K - 1;
    const int64_t ipb = (int64_t)bo * g.cb;  // items per plane-pair band
    t.ppu = 1;
    pair_strides<K>(t, rs0, 0, 0);
    const int64_t blk0 = (int64_t)t.blk * 8;
    int64_t ppu = (kNT + ipb - 1) / ipb;
    if (ppu * blk0 > limit) ppu = limit / blk0;
    if (ppu > g.npairs) ppu = g.npairs;
    if (force_ppu > 0) ppu = force_ppu;
    if (ppu < 1) continue;
    t.ppu = (int)ppu;
    t.items = (int)(ppu * ipb);
    // rows in mirror order (a warp's lanes then share equal filter-row
    // ranges) unless a quarter-warp's items wrap from one row to the next
    // and the filter is long: a mirror partner sits at a row distance that
    // changes from one quarter-warp to the next, so no row stride keeps
    // their window loads apart (at 48 columns a third of the shared-memory
    // wavefronts were conflicts), while the next row in plain order is
    // always one stride away. Measured on the 64 x 384 layers: plain order
    // 2-5 % faster at 48 rows for 21..31 taps, 2-4 % slower at 13 taps,
    // where the unequal ranges at the plane edges weigh more.
    if (((int64_t)t.ppu * g.cb) % 8 != 0 && K >= 21) t.mirror = 0;
    const int threads = ((t.items < kNT ? t.items : kNT) + 31) / 32 * 32;
    // strides with the fewest bank-group conflicts among those that keep the
    // unit within the limit: row stride first, then the block stride
    int rbest = 0, bbest = 0, cbest = 1 << 30;
    for (int rpad = 0; rpad < 16; rpad += 2) {
      PCfg u = t;
      pair_strides<K>(u, rs0, rpad, 0);
      if ((int64_t)u.stage_elems * 8 > limit) break;
      const int conf = pair_conflicts<K, V>(u, threads);
      if (conf < cbest) {
        cbest = conf;
        rbest = rpad;
      }
    }
    for (int bpad = 2; bpad < 16; bpad += 2) {
      PCfg u = t;
      pair_strides<K>(u, rs0, rbest, bpad);
      if ((int64_t)u.stage_elems * 8 > limit) break;
      const int conf = pair_conflicts<K, V>(u, threads);
      if (conf < cbest) {
        cbest = conf;
        bbest = bpad;
      }
    }
    pair_strides<K>(t, rs0, rbest, bbest);
    t.stages = 2 * (int64_t)t.stage_elems * 8 <= limit ? 2 : 1;
    if (force_stages > 0) t.stages = force_stages;
    if ((int64_t)t.stages * t.stage_elems * 8 > cta_max) continue;
    best_threads = threads;
    best = pair_rowfill<K>(t, threads);
    bestg = t;
  }
  if (best < 0) return false;
  const int64_t groups = (bestg.npairs + bestg.ppu - 1) / bestg.ppu;
  bestg.units = groups * bestg.nbands;
  bestg.d_bands = FastDiv((uint32_t)bestg.nbands);
  bestg.d_tr = FastDiv((uint32_t)bestg.tr);
  bestg.d_cb = FastDiv((uint32_t)bestg.cb);
  bestg.d_ppu = FastDiv((uint32_t)bestg.ppu);
  if (out_cfg) *out_cfg = bestg;
  if (threads_out) *threads_out = best_threads;
  if (score_out) *score_out = best;
  return true;
}

template <int K, int V>
cudaError_t launch_pair(const Conv& c, const PCfg& g0, int threads, const void* in, const void* w,
                        const void* bias, void* out, bool acc, cudaStream_t s, const Epi& ep) {
  PCfg g = g0;
  g.acc = acc;
  auto kern = pconv_kernel<K, V>;
  const size_t smem = (size_t)g.stages * g.stage_elems * 8;
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

// DWCONV_LARGE_FWD_PLAN="V:bo:ppu:stages" pins a plan (a
// tuning aid; 0 leaves a field to the planner).
template <int K>
cudaError_t run_fwd_k(const Conv& c, const void* in, const void* w, const void* bias, void* out, bool flip,
                      bool acc, cudaStream_t s, const Epi& ep) {
  int fv = 0, fbo = 0, fppu = 0, fst = 0;
  if (const char* e = std::getenv("DWCONV_LARGE_FWD_PLAN"))
    if (std::sscanf(e, "%d:%d:%d:%d", &fv, &fbo, &fppu, &fst) != 4) fv = fbo = fppu = fst = 0;
  PCfg g8, g16;
  int t8 = 0, t16 = 0;
  double s8 = 0, s16 = 0;
  const bool ok16 = fv != 8 && plan_pair<K, 16>(c, flip, &g16, &t16, &s16, fbo, fppu, fst);
  const bool ok8 = fv != 16 && plan_pair<K, 8>(c, flip, &g8, &t8, &s8, fbo, fppu, fst);
  if (!ok8 && !ok16) return cudaErrorInvalidConfiguration;
  // 8-wide column blocks measured faster for 31 x 31 filters and on planes
  // up to 32 columns wide, 16-wide blocks for the rest
  const int wout = (int)(flip ? c.W : c.Wo);
  const bool want8 = fv == 8 || (fv == 0 && (K >= 29 || wout <= 32));
  if ((!want8 && ok16) || !ok8) return launch_pair<K, 16>(c, g16, t16, in, w, bias, out, acc, s, ep);
  return launch_pair<K, 8>(c, g8, t8, in, w, bias, out, acc, s, ep);
}

}  // namespace large
}  // namespace dwconv
