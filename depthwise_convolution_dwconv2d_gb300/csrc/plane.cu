// Small-plane depthwise kernels (3x3 filters, stride 1 or 2, rows of at most
// 32 elements), one warp per group of whole planes.
//
// The "Spatial Depthwise Convolution on the GPU #3057" kernels compute one
// output per thread straight from global memory; the tile kernels stage bands
// of many planes per CTA. For the small MobileNet planes (7², 14², 28²) both
// spend most of their instructions on indexing and staging, so here a warp
// works alone on a few whole planes of one channel (P samples at a time):
//  * it copies the planes (coalesced rows, 8-byte granules where aligned)
//    into its own double-buffered, zero-haloed tile in shared memory (plane
//    slots offset so that the planes' lanes read disjoint banks), with what the
//    compute needs next to them (the channel's filter taps and bias; for the
//    weight gradient the grad_out planes), all with asynchronous copies
//    issued one work item ahead -- no CTA barrier and no global load on the
//    compute path;
//  * each lane owns one output column of one plane (two, four or eight
//    planes per warp as the rows narrow) and walks the output rows with the
//    K x K window held in registers (a stride-1 step loads one new row of
//    K values), so an output costs K shared loads, K*K FMAs and a store;
//    the walk is unrolled (fully for the common plane heights), with 32-bit
//    shared offsets and running pointers, so almost no integer work is left
//    per output row.
// The same correlation kernel serves the forward and the stride-1
// grad-input (grad_out correlated with the filter rotated by 180 degrees,
// padding K-1-p). In the weight-gradient first pass each warp owns whole
// (chunk, channel) units: its lanes accumulate K*K + 1 sums over the unit's
// sample groups, and at the end of a unit a butterfly reduces them into the
// unit's partial; the walk (and its copies) runs on across unit boundaries.
// Measured against the tile kernels on the MobileNet layers, these win for
// the forward and stride-1 grad-input on rows of 9..16 elements and for the
// weight gradient on output rows of at most 16; the planner uses them there
// only.
#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "plan.h"
#include "tile.cuh"

namespace dwconv {
namespace plane {
namespace {

constexpr int kWarps = 8;  // warps per CTA of the correlation kernels
constexpr int kThreads = kWarps * 32;
constexpr int kMaxW = 32;  // widest input / output row (one lane per column)
constexpr int kRB = 16;    // output rows per unrolled block of a lane's walk
constexpr int kCO = 2;     // tile column of input column 0 (even: 8-byte copies land aligned)

struct PCfg {
  int Hin, Win, Hout, Wout;  // planes read / written
  int pad;                   // padding of the evaluated correlation
  int L, P;                  // lanes per plane (power of two >= output columns), planes per warp (32 / L)
  int gran;                  // floats per plane copy granule: 2 (8-byte fp32 copies) or 1
  int ggran;                 // floats per grad_out copy granule (weight gradient): 4 (16-byte) or 1
  int Lw;                    // lanes per row when copying (power of two >= granules per row)
  int TR, TP, TS;            // tile rows, pitch (even), floats per plane slot
  int GS;                    // weight gradient: floats per staged grad_out plane slot
  int XO;                    // floats of a buffer before its filter taps / grad_out planes
  int BS;                    // floats per tile buffer (two per warp; a multiple of 4)
  int gpc;                   // sample groups per channel (ceil(N / P))
  int nb, G;                 // weight gradient: samples per chunk, sample groups per chunk
  int klast;                 // weight gradient: group holding the last chunk's last sample
};

int pow2_at_least(int v) {
  int p = 1;
  while (p < v) p *= 2;
  return p;
}

// smallest v' >= v with v' = r (mod 32)
int round_to_residue(int v, int r) {
  r &= 31;
  return v + ((r - v) % 32 + 32) % 32;
}

// asynchronous copies to a 32-bit shared-memory byte address
__device__ __forceinline__ void cp4(uint32_t s, const void* g) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, 4;\n" ::"r"(s), "l"(g) : "memory");
}
__device__ __forceinline__ void cp8(uint32_t s, const void* g) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, 8;\n" ::"r"(s), "l"(g) : "memory");
}
__device__ __forceinline__ void cp16(uint32_t s, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, 16;\n" ::"r"(s), "l"(g) : "memory");
}

// Copies of a group of np <= P planes into tile slots slot0 + q*TS: plane q
// is read at src0 + q*pstride (rows Win elements apart); its input row r
// lands on tile row r + pad and input column j on tile column kCO + j; the
// rest of a slot (the zero halo) is never written. The warp walks the
// group's rows flattened over the planes: lane (lr, lc) copies granule lc of
// rows lr, lr + rstep, ..., advancing its (plane, row) cursor by a constant
// step (no per-plane setup, no division); tall planes (about 16 rows or
// more) are walked one by one instead. fp32 goes by asynchronous copies
// (completed by the caller's wait), 16-bit types are widened through
// registers.
struct RowCopier {
  int lr, lc, rstep;  // lane's first row and granule, rows per warp step
  int q0, r0;         // lr as (plane, row)
  int dq, dr;         // rstep as (planes, rows)
  __device__ RowCopier(const PCfg& g, int lane) {
    lr = lane / g.Lw;
    lc = lane - lr * g.Lw;
    rstep = 32 / g.Lw;
    q0 = lr / g.Hin;
    r0 = lr - q0 * g.Hin;
    dq = rstep / g.Hin;
    dr = rstep - dq * g.Hin;
  }
  // TALL: 1 = per-plane loops, 0 = flattened walk, -1 = choose by the plane
  // height at run time
  template <int TALL, typename T>
  __device__ __forceinline__ void run(float* psm, int slot0, const T* __restrict__ src0, int64_t pstride, int np,
                                      const PCfg& g) const {
    const int cw = (sizeof(T) == 4 ? g.gran : 1) * lc;
    if (cw >= g.Win) return;
    const int rend = min(g.Hin, g.TR - g.pad);
    const uint32_t sb = (uint32_t)__cvta_generic_to_shared(psm);
    if (TALL == 1 || (TALL < 0 && g.Hin >= 16)) {
      // tall planes: a plain unrolled row loop per plane (its setup is paid
      // over many rows)
      for (int q = 0; q < np; ++q) {
        int di = slot0 + q * g.TS + (g.pad + lr) * g.TP + kCO + cw;
        const T* sp = src0 + q * pstride + lr * g.Win + cw;
#pragma unroll 4
        for (int r = lr; r < rend; r += rstep, di += rstep * g.TP, sp += rstep * g.Win) {
          if (sizeof(T) != 4) psm[di] = ld(sp);
          else if (g.gran == 2) cp8(sb + 4u * di, sp);
          else cp4(sb + 4u * di, sp);
        }
      }
      return;
    }
    int q = q0, r = r0;
    int di = slot0 + q * g.TS + (r + g.pad) * g.TP + kCO + cw;
    const T* sp = src0 + q * pstride + r * g.Win + cw;
    const int dstep = dq * g.TS + dr * g.TP, dwrap = g.TS - g.Hin * g.TP;
    const int64_t sstep = dq * pstride + dr * g.Win, swrap = pstride - (int64_t)g.Hin * g.Win;
    while (q < np) {
      if (r < rend) {
        if (sizeof(T) != 4) psm[di] = ld(sp);
        else if (g.gran == 2) cp8(sb + 4u * di, sp);
        else cp4(sb + 4u * di, sp);
      }
      r += dr;
      q += dq;
      di += dstep;
      sp += sstep;
      if (r >= g.Hin) {
        r -= g.Hin;
        ++q;
        di += dwrap;
        sp += swrap;
      }
    }
  }
};

// Zero a warp's two tile buffers (2 * BS floats from float index b0, a
// multiple of 4) with 16-byte stores.
__device__ __forceinline__ void zero_buffers(float* psm, int b0, int BS, int lane) {
  float4* z = reinterpret_cast<float4*>(psm + b0);
  for (int i = lane; i < BS / 2; i += 32) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  __syncwarp();
}

// One warp's run over its work items [ia, ib): item i+1 is copied into the
// other tile buffer while item i is computed. issue(buf) and compute(buf)
// are called once per item, in item order (each keeps its own cursor).
template <typename Issue, typename Compute>
__device__ __forceinline__ void warp_run(int ia, int ib, int buf0, int buf1, Issue issue, Compute compute) {
  if (ia < ib) issue(buf0);
  tile::cp_async_commit();
  for (int it = ia; it < ib; ++it) {
    const int cur = ((it - ia) & 1) ? buf1 : buf0;
    if (it + 1 < ib) issue(cur == buf0 ? buf1 : buf0);
    tile::cp_async_commit();
    tile::cp_async_wait<1>();
    __syncwarp();
    compute(cur);
    __syncwarp();
  }
  tile::cp_async_wait<0>();
}

// A lane's walk down its output column. t0 is the shared-memory float index
// of its window's top-left element for output row 0 (tile rows TP floats
// apart); row(win) is called for output rows 0, 1, ... in order with the
// K x K window. Addresses are 32-bit shared offsets advanced by constant
// strides, and the window's row shifts are register renames: rows run fully
// unrolled when the height HB is a compile-time constant, else in unrolled
// blocks of kRB with a bound check per row.
template <int K, int S, int HB, typename Row>
__device__ __forceinline__ void walk_rows(const float* __restrict__ sm, int t0, int TP, int Hout, Row row) {
  float win[K][K];
#pragma unroll
  for (int a = 0; a < K - S; ++a)
#pragma unroll
    for (int b = 0; b < K; ++b) win[a + S][b] = sm[t0 + a * TP + b];
  int t = t0 + (K - S) * TP;  // first tile row not yet in the window
  auto step = [&]() {
#pragma unroll
    for (int a = 0; a < K - S; ++a)
#pragma unroll
      for (int b = 0; b < K; ++b) win[a][b] = win[a + S][b];
#pragma unroll
    for (int a = K - S; a < K; ++a)
#pragma unroll
      for (int b = 0; b < K; ++b) win[a][b] = sm[t + (a - (K - S)) * TP + b];
    t += S * TP;
    row(win);
  };
  if (HB > 0) {
#pragma unroll
    for (int oy = 0; oy < HB; ++oy) step();
  } else {
    for (int ob = 0; ob < Hout; ob += kRB) {
#pragma unroll
      for (int u = 0; u < kRB; ++u) {
        if (ob + u >= Hout) break;
        step();
      }
    }
  }
}

// Cursor over (channel, index within channel) with a fixed count per channel.
struct Cursor {
  int ch, j;
  __device__ __forceinline__ void next(int per) {
    if (++j == per) {
      j = 0;
      ++ch;
    }
  }
};

// out[oy][ox] = bias + sum_{a,b} w'[a][b] in[oy*S - pad + a][ox*S - pad + b]
// MODE 0: forward (in = x, out = y slice)
// MODE 1: stride-1 grad-input (in = grad_out slice, w' = rot180(w), out = gx;
//         ACC adds to gx instead of overwriting it)
// Work item i = (channel ch, sample group k): the planes (n, ch) for n in
// [k*P, k*P + P), channel-major, so a warp's consecutive items share their
// filter. A tile buffer holds the group's P plane slots (TS floats each) and
// then the channel's K*K filter taps and bias (zero when absent). Global warp
// w runs items [I*w/Wt, I*(w+1)/Wt) of the I = C * gpc items. HB > 0: every
// output plane has HB rows.
template <typename T, int K, int S, int MODE, bool ACC, int HB>
__global__ void __launch_bounds__(kThreads, 4)
conv_kernel(Conv c, PCfg g, const T* __restrict__ in, const T* __restrict__ w, const T* __restrict__ bias,
            T* __restrict__ out) {
  constexpr int KK = K * K;
  extern __shared__ __align__(16) float psm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b0 = warp * 2 * g.BS;
  zero_buffers(psm, b0, g.BS, lane);  // the halo (and an absent bias) stays zero
  const int pl = lane / g.L, ox = lane - pl * g.L;
  const RowCopier rc(g, lane);
  const int N = (int)c.N;
  const int items = (int)c.C * g.gpc;
  // consecutive samples of one channel are this far apart in `in`
  const int64_t pstride = MODE == 0 ? c.x_base(1, 0) : c.y_base(1, 0) - c.y_base(0, 0);
  const uint32_t nw = gridDim.x * kWarps, wi = blockIdx.x * kWarps + warp;
  const int ia = (int)((uint64_t)items * wi / nw), ib = (int)((uint64_t)items * (wi + 1) / nw);
  auto in_base = [&](int n, int ch) -> int64_t { return MODE == 0 ? c.x_base(n, ch) : c.y_base(n, ch); };
  auto out_base = [&](int n, int ch) -> int64_t { return MODE == 0 ? c.y_base(n, ch) : c.x_base(n, ch); };
  Cursor ci{g.gpc > 0 ? ia / g.gpc : 0, g.gpc > 0 ? ia % g.gpc : 0}, cc = ci;
  auto issue = [&](int buf) {
    const int n0 = ci.j * g.P;
    rc.run<HB == 0 ? -1 : (HB * S >= 16 ? 1 : 0)>(psm, buf, in + in_base(n0, ci.ch), pstride, min(g.P, N - n0), g);
    if (lane < KK) {
      if (sizeof(T) == 4) cp4((uint32_t)__cvta_generic_to_shared(psm + buf + g.XO + lane), w + ci.ch * KK + lane);
      else psm[buf + g.XO + lane] = ld(w + ci.ch * KK + lane);
    } else if (lane == KK && MODE == 0 && bias != nullptr) {
      if (sizeof(T) == 4) cp4((uint32_t)__cvta_generic_to_shared(psm + buf + g.XO + KK), bias + ci.ch);
      else psm[buf + g.XO + KK] = ld(bias + ci.ch);
    }
    ci.next(g.gpc);
  };
  auto compute = [&](int buf) {
    const int ch = cc.ch, n = cc.j * g.P + pl;
    cc.next(g.gpc);
    if (ox >= g.Wout || n >= N) return;
    const float* const wt = psm + buf + g.XO;
    float wr[KK];
#pragma unroll
    for (int i = 0; i < KK; ++i) wr[i] = wt[MODE == 1 ? KK - 1 - i : i];
    const float bv = wt[KK];
    T* op = out + out_base(n, ch) + ox;
    const int wo = g.Wout;
    walk_rows<K, S, HB>(psm, buf + pl * g.TS + (kCO - g.pad) + ox * S, g.TP, g.Hout, [&](float (&win)[K][K]) {
      float acc = bv;
#pragma unroll
      for (int a = 0; a < K; ++a)
#pragma unroll
        for (int b = 0; b < K; ++b) acc = fmaf(wr[a * K + b], win[a][b], acc);
      *op = from_f<T>(ACC ? acc + ld_rw(op) : acc);
      op += wo;
    });
  };
  warp_run(ia, ib, b0, b0 + g.BS, issue, compute);
}

// Weight-gradient first pass: for unit (chunk cq, channel c),
// partial[cq, c, a*K + b] = sum over the chunk's samples of sum_{oy,ox} gy*x̃,
// partial[cq, c, K*K] = sum of gy. Units are ordered channel-major
// (u = c*chunks + cq); global warp w owns units [U*w/Wt, U*(w+1)/Wt) and
// walks their G sample groups each (P samples per group, one per lane group)
// as one run of work items. A tile buffer holds the group's P zero-haloed x
// plane slots and then its P grad_out planes (GS floats apart). Each lane
// keeps K*K + 1 sums; at the end of a unit a butterfly adds them over the
// warp in a fixed order and lanes 0..K*K write the unit's partial. HB > 0:
// every output plane has HB rows.
template <typename T, int K, int S, int HB>
__global__ void __launch_bounds__(kThreads, 3)
wgrad_kernel(Conv c, PCfg g, const T* __restrict__ x, const T* __restrict__ gy, float* __restrict__ ws,
             int chunks) {
  extern __shared__ __align__(16) float psm[];
  constexpr int NV = K * K + 1;
  const int nwarps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b0 = warp * 2 * g.BS;
  zero_buffers(psm, b0, g.BS, lane);
  const int pl = lane / g.L, ox = lane - pl * g.L;
  const RowCopier rc(g, lane);
  // (N * C < 2^31, so units, items and samples all fit 32 bits)
  const int N = (int)c.N, G = g.G;
  const int units = (int)c.C * chunks;
  const uint32_t nw = gridDim.x * nwarps, wi = blockIdx.x * nwarps + warp;
  const int ua = (int)((uint64_t)units * wi / nw), ub = (int)((uint64_t)units * (wi + 1) / nw);
  const int64_t xstride = c.x_base(1, 0), gstride = c.y_base(1, 0) - c.y_base(0, 0);
  // grad_out planes are copied as chunks of ggran floats, flattened over the
  // group's planes: lane's chunks lane, lane + 32, ... as (plane, chunk)
  const int ghw = g.Hout * g.Wout, cpp = ghw / g.ggran;
  const int gq0 = lane / cpp, gc0 = lane - gq0 * cpp, gdq = 32 / cpp, gdc = 32 - gdq * cpp;
  // unit cursor: channel ch, chunk cq, sample group k (samples
  // [cq*nb + k*P, min(cq*nb + k*P + P, chunk end)))
  struct UCur {
    int ch, cq, k;
  };
  auto next = [&](UCur& u) {
    if (++u.k == G) {
      u.k = 0;
      if (++u.cq == chunks) {
        u.cq = 0;
        ++u.ch;
      }
    }
  };
  float acc[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) acc[i] = 0.f;
  UCur ci{ua / chunks, ua % chunks, 0}, cc = ci;
  auto issue = [&](int buf) {
    const int c0 = ci.cq * g.nb, s0 = c0 + ci.k * g.P, np = min(g.P, min(c0 + g.nb, N) - s0);
    if (np > 0) {
      rc.run<HB == 0 ? -1 : (HB * S >= 16 ? 1 : 0)>(psm, buf, x + c.x_base(s0, ci.ch), xstride, np, g);
      const T* gp0 = gy + c.y_base(s0, ci.ch);
      const uint32_t sb = (uint32_t)__cvta_generic_to_shared(psm);
      for (int q = gq0, cc4 = gc0; q < np;) {
        const int di = buf + g.XO + q * g.GS + cc4 * g.ggran;
        const T* sp = gp0 + q * gstride + cc4 * g.ggran;
        if (sizeof(T) != 4) psm[di] = ld(sp);
        else if (g.ggran == 4) cp16(sb + 4u * di, sp);
        else cp4(sb + 4u * di, sp);
        cc4 += gdc;
        q += gdq;
        if (cc4 >= cpp) {
          cc4 -= cpp;
          ++q;
        }
      }
    }
    next(ci);
  };
  auto compute = [&](int buf) {
    const int ch = cc.ch, cq = cc.cq, k = cc.k;
    next(cc);
    const int c0 = cq * g.nb, s0 = c0 + k * g.P, s1 = min(c0 + g.nb, N);
    // an item with fewer than P samples (end of the last chunk) leaves some
    // lane groups idle; items past that end are empty. A unit flushes once,
    // at the item holding its last sample (item 0 when the batch is empty:
    // the partial is then zero).
    const bool last = k == (cq == chunks - 1 ? g.klast : G - 1);
    if (ox < g.Wout && s0 + pl < s1) {
      int gi = buf + g.XO + pl * g.GS + ox;
      const int wo = g.Wout;
      walk_rows<K, S, HB>(psm, buf + pl * g.TS + (kCO - g.pad) + ox * S, g.TP, g.Hout, [&](float (&win)[K][K]) {
        const float gv = psm[gi];
        gi += wo;
#pragma unroll
        for (int a = 0; a < K; ++a)
#pragma unroll
          for (int b = 0; b < K; ++b) acc[a * K + b] = fmaf(gv, win[a][b], acc[a * K + b]);
        acc[K * K] += gv;
      });
    }
    if (last) {
      float mine = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        float v = acc[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == i) mine = v;
        acc[i] = 0.f;
      }
      if (lane < NV) ws[((int64_t)cq * c.OC() + ch) * NV + lane] = mine;
    }
  };
  warp_run(ua * G, ub * G, b0, b0 + g.BS, issue, compute);
}

// Shapes served here: 3x3, stride 1 or 2, dilation 1, one filter per channel,
// input and output rows of at most 32, planes of at most 64 rows.
bool shape_ok(const Conv& c) {
  if (!c.planes32() || c.m != 1) return false;
  if (c.kh != 3 || c.kw != 3 || c.sh != c.sw || (c.sh != 1 && c.sh != 2) || c.dh != 1 || c.dw != 1) return false;
  if (c.ph != c.pw || c.ph > 2) return false;
  if (c.W > kMaxW || c.Wo > kMaxW || c.H > 64 || c.Ho > 64) return false;
  return true;
}

size_t smem_of(const PCfg& g, int warps) { return (size_t)warps * 2 * g.BS * sizeof(float); }

// dynamic shared memory a CTA may use (227 KB on this GPU)
constexpr size_t kSmemMax = 227 * 1024;

int resident(const void* kern, int threads, size_t smem) {
  int per = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, threads, smem) != cudaSuccess || per < 1) per = 1;
  return per;
}

int grid_of(const void* kern, int threads, size_t smem, int64_t work) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t cap = (int64_t)sms * resident(kern, threads, smem);
  return (int)(work < cap ? (work > 0 ? work : 1) : cap);
}

// Correlation geometry for MODE 0 / 1 (and the weight gradient's x planes);
// src is the first plane read, for the 8-byte copy alignment test.
PCfg conv_cfg(const Conv& c, bool grad, const void* src) {
  PCfg g{};
  g.Hin = grad ? (int)c.Ho : (int)c.H;
  g.Win = grad ? (int)c.Wo : (int)c.W;
  g.Hout = grad ? (int)c.H : (int)c.Ho;
  g.Wout = grad ? (int)c.W : (int)c.Wo;
  g.pad = grad ? c.kh - 1 - c.ph : c.ph;
  const int S = grad ? 1 : c.sh, K = c.kh;
  g.L = pow2_at_least(g.Wout);
  g.P = 32 / g.L;
  // 8-byte copies when every plane row starts 8-byte aligned
  const int64_t hw_in = (int64_t)g.Hin * g.Win;
  g.gran = (c.dtype == DWCONV_F32 && g.Win % 2 == 0 && hw_in % 2 == 0 && ((uintptr_t)src & 7) == 0) ? 2 : 1;
  g.Lw = pow2_at_least(g.gran == 2 ? g.Win / 2 : g.Win);
  g.TR = (g.Hout - 1) * S + K;
  g.TP = std::max(kCO + g.Win, kCO - g.pad + (g.Wout - 1) * S + K);
  g.TP += g.TP & 1;
  g.TS = g.TR * g.TP;
  // stride 1: the P planes' lanes read P disjoint bank ranges
  if (S == 1 && g.L >= 2) g.TS = round_to_residue(g.TS, g.L);
  g.XO = (g.P * g.TS + 3) / 4 * 4;
  g.GS = g.L >= 2 ? round_to_residue(g.Hout * g.Wout, g.L) : g.Hout * g.Wout;
  g.BS = (g.XO + K * K + 1 + 3) / 4 * 4;
  g.gpc = (int)((c.N + g.P - 1) / g.P);
  return g;
}

// Plane heights with fully unrolled row walks (the fp32 MobileNet planes:
// 14 and 7 rows, and 4 for the 7x7 stride-2 weight gradient); 0 = any height.
template <typename T, typename F>
cudaError_t with_height(int h, F f) {
  if (sizeof(T) == 4) {
    if (h == 14) return f(std::integral_constant<int, 14>());
    if (h == 7) return f(std::integral_constant<int, 7>());
    if (h == 4) return f(std::integral_constant<int, 4>());
  }
  return f(std::integral_constant<int, 0>());
}

template <typename T, int S, int HB>
cudaError_t fwd_h(const Conv& c, const PCfg& g, const void* x, const void* w, const void* b, void* y,
                  cudaStream_t s) {
  auto kern = conv_kernel<T, 3, S, 0, false, HB>;
  const size_t smem = smem_of(g, kWarps);
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_of((const void*)kern, kThreads, smem, (c.C * g.gpc + kWarps - 1) / kWarps);
  kern<<<grid, kThreads, smem, s>>>(c, g, (const T*)x, (const T*)w, (const T*)b, (T*)y);
  return cudaGetLastError();
}

template <typename T, int S>
cudaError_t fwd_t(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s) {
  const PCfg g = conv_cfg(c, false, x);
  return with_height<T>(g.Hout, [&](auto hb) { return fwd_h<T, S, decltype(hb)::value>(c, g, x, w, b, y, s); });
}

template <typename T, bool ACC, int HB>
cudaError_t bwd1_h(const Conv& c, const PCfg& g, const void* gy, const void* w, void* gx, cudaStream_t s) {
  auto kern = conv_kernel<T, 3, 1, 1, ACC, HB>;
  const size_t smem = smem_of(g, kWarps);
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_of((const void*)kern, kThreads, smem, (c.C * g.gpc + kWarps - 1) / kWarps);
  kern<<<grid, kThreads, smem, s>>>(c, g, (const T*)gy, (const T*)w, nullptr, (T*)gx);
  return cudaGetLastError();
}

template <typename T, bool ACC>
cudaError_t bwd1_t(const Conv& c, const void* gy, const void* w, void* gx, cudaStream_t s) {
  const T* first = (const T*)gy + c.y_base(0, 0);
  const PCfg g = conv_cfg(c, true, first);
  return with_height<T>(g.Hout, [&](auto hb) { return bwd1_h<T, ACC, decltype(hb)::value>(c, g, gy, w, gx, s); });
}

template <typename T, int S, int HB>
cudaError_t wgrad_h(const Conv& c, const PCfg& g, const void* x, const void* gy, float* ws, int chunks,
                    cudaStream_t s) {
  auto kern = wgrad_kernel<T, 3, S, HB>;
  // warps are independent: take the CTA size (8 or 4 warps) that keeps more
  // warps resident under the tile buffers' shared memory
  // (4 warps when 8 warps' buffers exceed a CTA's shared memory; the
  // planner only routes shapes whose 4-warp buffers fit)
  int warps = kWarps;
  {
    const size_t s8 = smem_of(g, 8), s4 = smem_of(g, 4);
    const bool eight = s8 <= kSmemMax;
    cudaError_t e = tile::set_smem(kern, eight ? s8 : s4);
    if (e != cudaSuccess) return e;
    if (!eight || 4 * resident((const void*)kern, 128, s4) > 8 * resident((const void*)kern, 256, s8)) warps = 4;
  }
  const size_t smem = smem_of(g, warps);
  const int64_t units = c.C * chunks;
  const int grid = grid_of((const void*)kern, warps * 32, smem, (units + warps - 1) / warps);
  kern<<<grid, warps * 32, smem, s>>>(c, g, (const T*)x, (const T*)gy, ws, chunks);
  return cudaGetLastError();
}

// Weight-gradient geometry: x plane slots, then the P grad_out planes.
PCfg wgrad_cfg(const Conv& c, const void* x) {
  PCfg g = conv_cfg(c, false, x);
  g.BS = (g.XO + g.P * g.GS + 3) / 4 * 4;
  return g;
}

template <typename T, int S>
cudaError_t wgrad_t(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
  PCfg g = wgrad_cfg(c, x);
  g.ggran = (c.dtype == DWCONV_F32 && (g.Hout * g.Wout) % 4 == 0 && g.GS % 4 == 0 && ((uintptr_t)gy & 15) == 0)
                ? 4 : 1;
  g.nb = (int)wgrad_nb(c);
  g.G = (g.nb + g.P - 1) / g.P;
  g.klast = c.N > 0 ? (int)((c.N - (int64_t)(chunks - 1) * g.nb - 1) / g.P) : 0;
  if (c.N > 0 && (c.N + g.nb - 1) / g.nb != chunks) return cudaErrorInvalidConfiguration;
  return with_height<T>(g.Hout, [&](auto hb) { return wgrad_h<T, S, decltype(hb)::value>(c, g, x, gy, ws, chunks, s); });
}

}  // namespace

// A shape is served only when its warps' tile buffers fit a CTA's shared
// memory (8 warps for the correlation kernels, at least 4 for the weight
// gradient); taller planes go to the tile kernels.
bool fwd_supported(const Conv& c) {
  return shape_ok(c) && c.W > 8 && c.W <= 16 && smem_of(conv_cfg(c, false, nullptr), kWarps) <= kSmemMax;
}
bool bwd_data_supported(const Conv& c) {
  return shape_ok(c) && c.sh == 1 && c.W > 8 && c.W <= 16 && smem_of(conv_cfg(c, true, nullptr), kWarps) <= kSmemMax;
}
bool wgrad_supported(const Conv& c) {
  return shape_ok(c) && c.Wo <= 16 && smem_of(wgrad_cfg(c, nullptr), 4) <= kSmemMax;
}

int64_t wgrad_nb(const Conv& c) {
  // A warp owns whole (chunk, channel) units of G sample groups (P samples
  // each): take the G whose busiest warp -- ceil(units / warps) units, each
  // G groups plus one warp reduction (about a third of a group) -- is
  // shortest, for about 3 x 8 resident warps per SM on 152 SMs.
  const int64_t P = 32 / pow2_at_least((int)c.Wo);
  const int64_t warps = 152 * 24;
  int64_t best = P;
  double best_cost = 0.0;
  for (int64_t G = 1; G <= 8; ++G) {
    const int64_t nb = G * P;
    const int64_t units = c.C * ((c.N + nb - 1) / nb);
    const double cost = (double)((units + warps - 1) / warps) * ((double)G + 0.35);
    if (G == 1 || cost < best_cost - 1e-9) {
      best_cost = cost;
      best = nb;
    }
    if (nb >= c.N) break;
  }
  if (best > c.N) best = c.N > 0 ? c.N : 1;
  return best;
}

int wgrad_chunks(const Conv& c) {
  const int64_t nb = wgrad_nb(c);
  return c.N > 0 ? (int)((c.N + nb - 1) / nb) : 1;
}

cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  if (c.sh == 1) {
    DWCONV_DISPATCH_DTYPE(c.dtype, T, e = (fwd_t<T, 1>(c, x, w, b, y, s)));
  } else {
    DWCONV_DISPATCH_DTYPE(c.dtype, T, e = (fwd_t<T, 2>(c, x, w, b, y, s)));
  }
  return e;
}

cudaError_t bwd_data(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  if (c.sh != 1) return e;
  if (acc) {
    DWCONV_DISPATCH_DTYPE(c.dtype, T, e = (bwd1_t<T, true>(c, gy, w, gx, s)));
  } else {
    DWCONV_DISPATCH_DTYPE(c.dtype, T, e = (bwd1_t<T, false>(c, gy, w, gx, s)));
  }
  return e;
}

cudaError_t wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  if (c.sh == 1) {
    DWCONV_DISPATCH_DTYPE(c.dtype, T, e = (wgrad_t<T, 1>(c, x, gy, ws, chunks, s)));
  } else {
    DWCONV_DISPATCH_DTYPE(c.dtype, T, e = (wgrad_t<T, 2>(c, x, gy, ws, chunks, s)));
  }
  return e;
}

}  // namespace plane
}  // namespace dwconv
