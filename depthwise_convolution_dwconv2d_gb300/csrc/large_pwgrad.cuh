// Large-kernel depthwise weight gradient on packed fp32x2 FMAs (square odd K
// from 7 to 31, stride 1, dilation 1, one filter per channel):
//   gw[c, a, b] = sum_{n, oh, ow} gy[n, c, oh, ow] * x[n, c, oh + a - p, ow + b - p]
// for one chunk of samples and one band of output rows per unit; every unit
// writes one fp32 partial per channel (taps and bias), and the second pass
// adds the partials in index order.
//
// It is a correlation of the zero-padded x plane with the grad_out plane that
// yields a K x K result. A CTA owns (channel, sample chunk, band of output
// rows) units and walks the chunk's samples two at a time: the two samples'
// x bands and grad_out bands are staged interleaved (float2: sample n,
// sample n + 1), so every operand is a ready-made lane pair for
// fma.rn.f32x2 and the two lanes accumulate the two samples' sums.
//  * A thread owns RA filter rows x 8 filter columns of taps. Its threads
//    for every tap block form a group, and group g takes the output rows
//    oh = g, g + G, ... of the band. Per output row the thread walks grad_out
//    two columns at a time -- one 16-byte load of two grad_out pairs, the
//    same address for the whole group -- against a ring of five 16-byte
//    chunks of each of its x rows: each grad_out pair feeds RA x 8 packed
//    FMAs from registers, the operand pattern that keeps the FP32 pipe near
//    its peak.
//  * Output rows whose x rows are all zero padding for the thread's filter
//    rows are skipped (the threads of a warp hold one or two filter-row
//    blocks, so their ranges nearly agree).
//  * The threads of a quarter-warp read two tap-column blocks' windows of
//    four consecutive output rows; the x row stride is an odd number of
//    16-byte chunks (chosen by the host planner, which simulates the bank
//    groups of every quarter-warp's loads), so those loads do not collide.
//  * At the end of a unit each thread adds its two lanes, the groups' sums
//    are added in a fixed order and written as the unit's partial; results
//    are bitwise reproducible.
#pragma once

#include "large_pair.cuh"

namespace dwconv {
namespace large {

template <int K>
struct PWGeo {
  // three filter rows per thread where three divide K (no empty rows in
  // the last block), else two (measured at 13, 21, 27 and 31 taps: two rows
  // are 2-8 % slower at 21 and 27, three rows 11-16 % slower at 31, where
  // the last block holds one row of three and only five row groups fit a
  // CTA; four rows with one CTA per SM were slower still); two CTAs per SM
  static constexpr int RA = K % 3 == 0 ? 3 : 2, VB = 8;
  static constexpr int min_ctas = RA == 4 ? 1 : 2;
  static constexpr int NA = (K + RA - 1) / RA, NB = (K + VB - 1) / VB;
  static constexpr int items = NA * NB;
  static constexpr int G = kNT / items;
  static constexpr int threads = (items * G + 31) / 32 * 32;
  // Thread t -> (tap-column block ib, group grp, tap-row block ia). With an
  // even number of column blocks a quarter-warp holds two column blocks
  // (windows 64 bytes apart) of four consecutive groups (rows one row stride
  // apart): with a row stride of an odd number of 16-byte chunks its eight
  // loads fall in eight bank groups. The threads of a warp share one or two
  // tap-row blocks.
  __host__ __device__ static void split(int t, int& ib, int& grp, int& ia) {
    if constexpr (NB % 2 == 0) {
      const int r1 = t >> 1;
      grp = r1 % G;
      const int r2 = r1 / G;
      ib = (t & 1) + 2 * (r2 % (NB / 2));
      ia = r2 / (NB / 2);
    } else {
      ib = t % NB;
      const int r1 = t / NB;
      grp = r1 % G;
      ia = r1 / G;
    }
  }
};

struct PWCfg {
  int nb, chunks, bands, bo;  // samples per chunk, chunks, bands of output rows, rows per band
  int xrows, xcols, xrs;      // x tile: rows, staged logical pair columns, row stride (pairs)
  int gcols, grs;             // grad_out tile: staged pair columns (even, >= Wo), row stride (pairs)
  int x_elems, stage_elems;   // pairs
  int stages, pad, dtype;
  FastDiv d_xrows, d_bo, d_parts;
};

template <int K>
__global__ void __launch_bounds__(kNT, PWGeo<K>::min_ctas)
pwgrad_kernel(Conv c, PWCfg g, const void* __restrict__ x, const void* __restrict__ gy, float* __restrict__ ws) {
  using Gm = PWGeo<K>;
  constexpr int RA = Gm::RA, VB = Gm::VB, G = Gm::G;
  extern __shared__ __align__(16) float2 smp[];
  const int tid = threadIdx.x, lane = tid & 31, nw = blockDim.x >> 5, nt = blockDim.x;
  const int64_t units = c.C * g.chunks * g.bands;
  const int H = (int)c.H, W = (int)c.W, Ho = (int)c.Ho, Wo = (int)c.Wo;
  const int es = g.dtype == DWCONV_F32 ? 4 : 2;
  const bool f32 = g.dtype == DWCONV_F32;

  // unit u = part * C + channel, part = chunk * bands + band
  struct Unit {
    int64_t ch, n0, n1;  // channel, samples [n0, n1)
    int oh0, rows;       // output rows [oh0, oh0 + rows)
    int64_t part;
  };
  auto unit_of = [&](int64_t u) {
    Unit r;
    uint32_t part;
    r.ch = c.dC.divmod((uint32_t)u, part);
    uint32_t chunk;
    const int band = (int)g.d_parts.divmod(part, chunk);
    r.part = part;
    r.n0 = (int64_t)chunk * g.nb;
    r.n1 = r.n0 + g.nb < c.N ? r.n0 + g.nb : c.N;
    r.oh0 = band * g.bo;
    r.rows = Ho - r.oh0 < g.bo ? Ho - r.oh0 : g.bo;
    return r;
  };
  auto unit_steps = [&](const Unit& r) {
    const int64_t ns = r.n1 - r.n0;
    return ns > 0 ? (int)((ns + 1) / 2) : 1;  // an empty unit still writes its zero partial
  };

  // Stage sample pair sp of unit r: x rows oh0 - p .. (band + halo), grad_out rows of the band.
  auto issue = [&](const Unit& r, int sp, float2* dst) {
    for (int t = tid >> 5; t < 2 * g.xrows; t += nw) {
      uint32_t h;
      const int rr = (int)g.d_xrows.divmod((uint32_t)t, h);
      const int64_t n = r.n0 + 2 * sp + h;
      const int iy = r.oh0 + rr - g.pad;
      const bool rin = n < r.n1 && iy >= 0 && iy < H;
      const char* srow = reinterpret_cast<const char*>(x) + (rin ? c.x_base(n, r.ch) + (int64_t)iy * W : 0) * es;
      float* drow = reinterpret_cast<float*>(dst + rr * g.xrs) + h;
      for (int col = lane; col < g.xcols; col += 32) {
        const int ix = col - g.pad;
        const bool ok = rin && ix >= 0 && ix < W;
        float* d = drow + 2 * col;
        if (f32) tile::cp_async4(d, reinterpret_cast<const float*>(srow) + (ok ? ix : 0), ok ? 4 : 0);
        else *d = ok ? ld_any(srow, ix, g.dtype) : 0.f;
      }
    }
    float2* gdst = dst + g.x_elems;
    for (int t = tid >> 5; t < 2 * g.bo; t += nw) {
      uint32_t h;
      const int rr = (int)g.d_bo.divmod((uint32_t)t, h);
      if (rr >= r.rows) continue;  // past the last band's rows
      const int64_t n = r.n0 + 2 * sp + h;
      const bool rin = n < r.n1;
      const char* srow =
          reinterpret_cast<const char*>(gy) + (rin ? c.y_base(n, r.ch) + (int64_t)(r.oh0 + rr) * Wo : 0) * es;
      float* drow = reinterpret_cast<float*>(gdst + rr * g.grs) + h;
      for (int col = lane; col < g.grs; col += 32) {
        const bool ok = rin && col < Wo;
        float* d = drow + 2 * col;
        if (f32) tile::cp_async4(d, reinterpret_cast<const float*>(srow) + (ok ? col : 0), ok ? 4 : 0);
        else *d = ok ? ld_any(srow, col, g.dtype) : 0.f;
      }
    }
  };

  // this thread's taps: filter rows a0 .. a0 + RA - 1, columns b0 .. b0 + 7
  int ib, grp, ia;
  Gm::split(tid, ib, grp, ia);
  const bool active = ia < Gm::NA;
  const int a0 = RA * ia, b0 = VB * ib;
  u64 acc[RA][VB];
#pragma unroll
  for (int r = 0; r < RA; ++r)
#pragma unroll
    for (int v = 0; v < VB; ++v) acc[r][v] = 0ull;
  float bsum = 0.f;

  auto compute = [&](const Unit& r, const float2* xs, const float2* gs) {
    // bias: every staged grad_out value (padding columns are zero)
    for (int e = tid; e < r.rows * g.grs; e += nt) {
      const float2 v = gs[e];
      bsum += v.x + v.y;
    }
    if (!active) return;
    // band rows whose x rows (tile rows oh + a0 .. oh + a0 + RA - 1) meet a real input row
    int lo = g.pad - r.oh0 - a0 - (RA - 1);
    int hi = g.pad + H - r.oh0 - a0;
    lo = lo < 0 ? 0 : lo;
    hi = hi > r.rows ? r.rows : hi;
    int oh = grp;
    if (oh < lo) oh += (lo - oh + G - 1) / G * G;
    const int nst = g.gcols / 2;
    for (; oh < hi; oh += G) {
      // window chunk m of x row ra: pairs b0 + 2m, b0 + 2m + 1
      const ulonglong2* xrow[RA];
#pragma unroll
      for (int ra = 0; ra < RA; ++ra)
        xrow[ra] = reinterpret_cast<const ulonglong2*>(xs + (oh + a0 + ra) * g.xrs + b0);
      const ulonglong2* grow = reinterpret_cast<const ulonglong2*>(gs + oh * g.grs);
      // ring of five chunks per x row: chunk m in slot m % 5
      u64 xw[RA][10];
      auto ldx = [&](int ra, int slot, const ulonglong2* p) {
        const ulonglong2 t = *p;
        xw[ra][2 * slot] = t.x;
        xw[ra][2 * slot + 1] = t.y;
      };
#pragma unroll
      for (int ra = 0; ra < RA; ++ra)
#pragma unroll
        for (int m = 0; m < 4; ++m) ldx(ra, m, xrow[ra] + m);
      for (int s0 = 0; s0 < nst; s0 += 5) {
#pragma unroll
        for (int ss = 0; ss < 5; ++ss) {
          const int s = s0 + ss;
          if (s >= nst) break;
#pragma unroll
          for (int ra = 0; ra < RA; ++ra) ldx(ra, (ss + 4) % 5, xrow[ra] + s + 4);
          const ulonglong2 gg = grow[s];  // grad_out pairs at columns 2s, 2s + 1
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const u64 gv = j ? gg.y : gg.x;
#pragma unroll
            for (int ra = 0; ra < RA; ++ra)
#pragma unroll
              for (int v = 0; v < VB; ++v) {
                const int idx = j + v;  // window pair 2s + idx
                const int slot = (ss + (idx >> 1)) % 5;
                fma2(acc[ra][v], gv, xw[ra][2 * slot + (idx & 1)]);
              }
          }
        }
      }
    }
  };

  // end of a unit: lanes added, groups' sums added in a fixed order (in the
  // consumed stage buffer), one partial per (part, channel)
  auto finish_unit = [&](const Unit& r, float* red) {
    if (active) {
#pragma unroll
      for (int ra = 0; ra < RA; ++ra)
#pragma unroll
        for (int v = 0; v < VB; ++v) {
          const int a = a0 + ra, b = b0 + v;
          float lo, hi;
          unpack2(acc[ra][v], lo, hi);
          if (a < K && b < K) red[grp * (K * K) + a * K + b] = lo + hi;
        }
    }
#pragma unroll
    for (int ra = 0; ra < RA; ++ra)
#pragma unroll
      for (int v = 0; v < VB; ++v) acc[ra][v] = 0ull;
    float bv = bsum;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bv += __shfl_xor_sync(0xffffffffu, bv, o);
    bsum = 0.f;
    float* wred = red + G * (K * K);
    if (lane == 0) wred[tid >> 5] = bv;
    __syncthreads();
    float* dstp = ws + (r.part * c.OC() + r.ch) * (K * K + 1);
    for (int t = tid; t < K * K; t += nt) {
      float sum = 0.f;
      for (int gi = 0; gi < G; ++gi) sum += red[gi * (K * K) + t];
      dstp[t] = sum;
    }
    if (tid == 0) {
      float sum = 0.f;
      for (int wi = 0; wi < nw; ++wi) sum += wred[wi];
      dstp[K * K] = sum;
    }
    __syncthreads();
  };

  // (unit, sample pair) steps of this CTA, flattened; a stage per step
  int64_t u = blockIdx.x;
  if (u >= units) return;
  Unit cu = unit_of(u);
  int sp = 0;
  issue(cu, sp, smp);
  tile::cp_async_commit();
  for (int k = 0;; ++k) {
    // next step
    int64_t un = u;
    Unit nu = cu;
    int spn = sp + 1;
    if (spn >= unit_steps(cu)) {
      spn = 0;
      un = u + gridDim.x;
      if (un < units) nu = unit_of(un);
    }
    float2* cur = smp + (g.stages == 2 ? (k & 1) : 0) * g.stage_elems;
    if (g.stages == 2) {
      if (un < units) issue(nu, spn, smp + ((k + 1) & 1) * g.stage_elems);
      tile::cp_async_commit();
      tile::cp_async_wait<1>();
    } else {
      tile::cp_async_wait<0>();
    }
    __syncthreads();
    compute(cu, cur, cur + g.x_elems);
    __syncthreads();
    if (un != u) finish_unit(cu, reinterpret_cast<float*>(cur));
    if (g.stages == 1) {
      if (un < units) issue(nu, spn, smp);
      tile::cp_async_commit();
    }
    if (un >= units) break;
    u = un;
    cu = nu;
    sp = spn;
  }
  tile::cp_async_wait<0>();
}

// ---- host planner ----------------------------------------------------------
// Bank-group conflicts of the first x-window and grad_out loads of the CTA's
// quarter-warps (per quarter-warp, the most distinct 16-byte chunks in one
// bank group), summed.
template <int K>
int pw_conflicts(const PWCfg& g, int threads) {
  using Gm = PWGeo<K>;
  int total = 0;
  for (int q0 = 0; q0 < threads; q0 += 8) {
    int xq[8], gq[8], n = 0;
    for (int l = 0; l < 8; ++l) {
      const int t = q0 + l;
      int ib, grp, ia;
      Gm::split(t, ib, grp, ia);
      if (ia >= Gm::NA) break;
      xq[n] = ((grp + Gm::RA * ia) * g.xrs + Gm::VB * ib) / 2;
      gq[n] = (grp * g.grs) / 2;
      ++n;
    }
    for (int pass = 0; pass < 2; ++pass) {
      const int* q = pass ? gq : xq;
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

// Samples per chunk of the sample axis: about eight (channel, chunk) units
// per resident CTA (two per SM), so the persistent CTAs end close together,
// rounded up to an even count so that only the batch's last sample can sit
// in a half-empty pair (a chunk of 3 samples would spend a quarter of its
// FMAs on the zero second lane of its last pair).
inline int64_t pw_chunk_samples(const Conv& c) {
  int64_t chunks = (152 * 2 * 8 + c.C - 1) / c.C;
  if (chunks > c.N) chunks = c.N;
  if (chunks < 1) chunks = 1;
  const int64_t nb = (c.N + chunks - 1) / chunks;
  return nb + (nb & 1);
}

inline int pw_chunks(const Conv& c) {
  const int64_t nb = pw_chunk_samples(c);
  return (int)(c.N > 0 ? (c.N + nb - 1) / nb : 1);
}

// Plan: the fewest bands of output rows whose stage (x band with its halo
// and the grad_out band, both for two samples) leaves room for two CTAs per
// SM; a second stage where it still does. Depends on the descriptor alone.
template <int K>
bool plan_pwgrad(const Conv& c, PWCfg* out_cfg, size_t* smem_out) {
  using Gm = PWGeo<K>;
  // per-CTA budget: half an SM where two CTAs are resident, else one CTA
  const int64_t half_sm = Gm::min_ctas == 2 ? 228 * 1024 / 2 - 1024 : 227 * 1024 - 1024;
  const int Ho = (int)c.Ho, Wo = (int)c.Wo;
  PWCfg g{};
  g.chunks = pw_chunks(c);
  g.nb = (int)(c.N > 0 ? pw_chunk_samples(c) : 1);
  g.pad = c.ph;
  g.dtype = c.dtype;
  g.gcols = (Wo + 1) / 2 * 2;
  g.grs = (g.gcols / 2) % 2 == 0 ? g.gcols + 2 : g.gcols;  // odd number of chunks per row
  // window chunks reach logical pair b0 + 2 (nst + 3) + 1 <= 8 (NB - 1) + gcols + 7
  g.xcols = g.gcols + 8 * Gm::NB;
  const int xrs0 = (g.xcols + 1) / 2 * 2;
  for (int bands = 1; bands <= Ho; ++bands) {
    PWCfg t = g;
    t.bands = bands;
    t.bo = (Ho + bands - 1) / bands;
    t.xrows = t.bo + Gm::RA * Gm::NA - 1;
    int best = 1 << 30, bestpad = 0;
    for (int pad2 = 0; pad2 < 16; pad2 += 2) {
      PWCfg u = t;
      u.xrs = xrs0 + pad2;
      const int conf = pw_conflicts<K>(u, Gm::threads);
      if (conf < best) {
        best = conf;
        bestpad = pad2;
      }
    }
    t.xrs = xrs0 + bestpad;
    t.x_elems = t.xrows * t.xrs;
    int64_t stage = (int64_t)t.x_elems + (int64_t)t.bo * t.grs;
    const int64_t red_pairs = ((int64_t)Gm::G * K * K + kNT / 32 + 1) / 2;
    if (stage < red_pairs) stage = red_pairs;
    stage = (stage + 1) / 2 * 2;
    if (stage * 8 > half_sm && bands < Ho) continue;
    if (stage * 8 > 227 * 1024 - 1024) return false;
    t.stage_elems = (int)stage;
    t.stages = 2 * stage * 8 <= half_sm ? 2 : 1;
    t.d_xrows = FastDiv((uint32_t)t.xrows);
    t.d_bo = FastDiv((uint32_t)t.bo);
    t.d_parts = FastDiv((uint32_t)t.bands);
    if (out_cfg) *out_cfg = t;
    if (smem_out) *smem_out = (size_t)t.stages * t.stage_elems * 8;
    return true;
  }
  return false;
}

// Partials the weight gradient writes per channel (sample chunks x bands).
template <int K>
int pwgrad_parts(const Conv& c) {
  PWCfg g;
  if (!plan_pwgrad<K>(c, &g, nullptr)) return 0;
  return g.chunks * g.bands;
}

template <int K>
cudaError_t run_pwgrad_k(const Conv& c, const void* x, const void* gy, float* ws, int parts, cudaStream_t s) {
  PWCfg g;
  size_t smem = 0;
  if (!plan_pwgrad<K>(c, &g, &smem) || g.chunks * g.bands != parts) return cudaErrorInvalidConfiguration;
  auto kern = pwgrad_kernel<K>;
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 152, per_sm = 1;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, PWGeo<K>::threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t units = c.C * parts;
  const int64_t cap = (int64_t)sms * per_sm;
  const int grid = (int)(units < cap ? units : cap);
  kern<<<grid, PWGeo<K>::threads, smem, s>>>(c, g, x, gy, ws);
  return cudaGetLastError();
}

}  // namespace large
}  // namespace dwconv
