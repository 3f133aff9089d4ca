// Kernel-im2col cache for the tensor-core large-kernel forward / stride-1
// grad-input: the expanded filter is prepared once, in global memory, and
// each call stages it with the tensor memory accelerator instead of
// synthesising it per tile.
//
// The MegEngine large-kernel depthwise article (section on the
// implicit-batched-GEMM algorithm) runs each channel as a GEMM whose A
// operand is the im2col of the *filter*,
//   T_c[f, g] = w_c[ih - oh + ph][iw - ow + pw]
// (f = oh*Wo + ow output positions, g = ih*Wi + iw input positions), and
// remarks that when shapes do not change between inference calls this
// filter-side im2col can be done ahead of time. The uncached kernel
// (ibgemm.cu) rebuilds every 128 x 128 block of T_c for every tile; here the
// blocks come from a cache built once per filter.
//
// Which shapes have a compact cache. With equal input and output row widths
// W (Wi == Wo, i.e. "same" padding across the row) and W dividing 64, a
// 128-position M tile is R = 128 / W whole output rows and a 64-position K
// atom is h = 64 / W whole input rows. Then the rows of T_c that belong to
// output row oh, restricted to the h input rows of one atom starting at ih,
// form a W x 64 matrix that depends only on j = ih - oh + ph:
//   S_j[ow][k] = w_c[j + k / W][k % W - ow + pw]   (0 outside the filter)
// and the 128 x 64 A operand of atom a of K step kc in tile t is the stack
// S_{j0}, S_{j0-1}, ..., S_{j0-R+1} with j0 = R*(kc - t) + h*a + ph. Stored
// in descending j, every A operand is 128 consecutive rows of the strip
// array. The cache holds, per channel, the NS strips with j in
// [jmin, jmax] (every j some nonzero block needs), rows of 64 16-bit elements
// (128 bytes), plain row-major: [C][NS][W][64]. A tensor-map copy with
// 128-byte swizzle puts it into the K-major shared layout the MMA reads, and
// an operand that starts at strip q is the same layout q * W * 128 bytes
// further on (W >= 8 rows keeps every strip on a 1024-byte swizzle-period
// boundary). A shape has a cached form when one channel's strips fit in
// shared memory beside two B stages.
//
// Kernel (persistent CTAs over units = (channel, group of G M tiles, chunk of
// up to 64 samples) in channel order; warp roles hand work over through
// mbarriers only):
//  * producer (warp 8, one lane): when the channel changes, copies the
//    channel's strips into shared memory once the MMAs of the previous
//    channel are done; per K step of the unit, copies the 128-position x
//    64-sample block of X_c into a stage, once for all tiles of the group;
//  * MMA issuer (warp 9, one lane): per K step, eight K=16 tcgen05.mma into
//    every tile of the group that the step reaches, interleaved across the
//    tiles so that consecutive MMAs go to different accumulators (a chain
//    into one 128 x 64 accumulator waits on each previous MMA); operands
//    from shared memory, one fp32 accumulator slot per tile in tensor memory;
//  * epilogue (warps 0-7): as each tile's last K step completes,
//    tcgen05.ld of its accumulator, bias, store.
// Only the K steps whose A operand has a nonzero tap are visited; each
// tile's sum runs over K steps, atoms and K slices in the same order as the
// uncached kernel's.
//
// Every wait is bounded; a wait that gives up counts in the library's
// timeout counter and raises the CTA's abort flag, after which no role
// waits or issues again, the producer and issuer wait (bounded) for their
// copies and MMAs in flight, and the CTA frees its tensor memory and
// returns.
#include <cstdlib>
#include <type_traits>

#include "plan.h"
#include "tc.cuh"
#include "tile.cuh"
#include "tma.cuh"

namespace dwconv {
namespace ibc {
namespace {

constexpr int kM = 128;     // M tile (output positions)
constexpr int kAtom = 64;   // K positions per 128-byte swizzle atom
constexpr int kAtoms = 2;   // atoms per K step
constexpr int kKs = kAtom * kAtoms;
constexpr int kMaxStages = 6;
constexpr int kNChunk = 64;  // samples per unit (MMA N at most 64)
constexpr unsigned kSleepNs = 64;
constexpr size_t kSmemLimit = 226 * 1024;  // dynamic shared memory; 1 KB left for the static part

__host__ __device__ inline int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Geometry of the correlation the kernel runs (the forward as given; the
// grad-input as a correlation of grad_out with the rotated filter and
// padding k - 1 - p) and of its strip cache.
struct Geo {
  int Hi, Wi, Ho, Wo, ph, pw, kh, kw;
  int flip;
  int R, h;          // output rows per M tile, input rows per K atom
  int dmin, dmax;    // K step minus tile, over the blocks with a nonzero tap
  int jmin, jmax;    // strip range
  int NS;            // strips per channel
  int T, KB;         // M tiles, K steps per plane
};

bool make_geo(const Conv& c, bool flip, Geo* out) {
  if (c.dtype != DWCONV_F16 && c.dtype != DWCONV_BF16) return false;
  if (c.sh != 1 || c.sw != 1 || c.dh != 1 || c.dw != 1 || c.m != 1) return false;
  if (c.ph > c.kh - 1 || c.pw > c.kw - 1) return false;
  Geo g{};
  g.kh = c.kh;
  g.kw = c.kw;
  g.flip = flip ? 1 : 0;
  if (!flip) {
    g.Hi = (int)c.H; g.Wi = (int)c.W; g.Ho = (int)c.Ho; g.Wo = (int)c.Wo; g.ph = c.ph; g.pw = c.pw;
  } else {
    g.Hi = (int)c.Ho; g.Wi = (int)c.Wo; g.Ho = (int)c.H; g.Wo = (int)c.W; g.ph = c.kh - 1 - c.ph;
    g.pw = c.kw - 1 - c.pw;
  }
  if (g.Wi != g.Wo || g.Wo < 8 || 64 % g.Wo != 0) return false;
  g.R = kM / g.Wo;
  g.h = kAtom / g.Wo;
  // nonzero blocks: filter rows R*d + ph - (R-1) .. R*d + ph + (R-1) meet 0..kh-1
  g.dmin = -floor_div(g.ph + g.R - 1, g.R);
  g.dmax = floor_div(g.kh - 1 + g.R - 1 - g.ph, g.R);
  g.jmin = g.R * g.dmin + g.ph - (g.R - 1);
  g.jmax = g.R * g.dmax + g.h + g.ph;
  g.NS = g.jmax - g.jmin + 1;
  if (c.C * g.NS * g.Wo >= (int64_t(1) << 31)) return false;  // strip rows are 32-bit copy coordinates
  g.T = (g.Ho * g.Wo + kM - 1) / kM;
  g.KB = (g.Hi * g.Wi + kKs - 1) / kKs;
  *out = g;
  return true;
}

size_t cache_bytes_of(const Conv& c, const Geo& g) { return (size_t)c.C * g.NS * g.Wo * kAtom * 2; }

// K steps of tile t: those whose A operand has a nonzero tap, inside the plane.
__host__ __device__ __forceinline__ void k_range(int T_dmin, int T_dmax, int KB, int t, int& lo, int& hi) {
  lo = t + T_dmin;
  hi = t + T_dmax + 1;
  if (lo < 0) lo = 0;
  if (hi > KB) hi = KB;
}

// First strip (index into the descending-j array) of atom a of the K step
// kc - t = d.
__host__ __device__ __forceinline__ int strip_of(int jmax, int R, int h, int ph, int d, int a) {
  return jmax - (R * d + h * a + ph);
}

// Filter tap of strip element (q, ow, k) of one channel's cache: the index
// into that channel's kh x kw filter as stored (rotated for the
// grad-input), or -1 where the element is zero.
__host__ __device__ __forceinline__ int strip_tap(int kh, int kw, int pw, int flip, int W, int jmax, int q, int ow,
                                                  int k) {
  const int dy = jmax - q + k / W;
  const int dx = k % W - ow + pw;
  if (dy < 0 || dy >= kh || dx < 0 || dx >= kw) return -1;
  return flip ? (kh - 1 - dy) * kw + (kw - 1 - dx) : dy * kw + dx;
}

struct BCfg {
  int kh, kw, pw, flip, W, jmax, NS;
  int64_t C;
};

// Cache build: one thread per 8 elements (16 bytes) of the [C][NS][W][64] array.
template <typename T>
__global__ void __launch_bounds__(256) build_kernel(BCfg b, const T* __restrict__ w, T* __restrict__ cache) {
  const int64_t total = b.C * b.NS * b.W * (kAtom / 8);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i >> 3;
    const int k0 = (int)(i & 7) * 8;
    const int ow = (int)(row % b.W);
    const int64_t cq = row / b.W;
    const int q = (int)(cq % b.NS);
    const int64_t c = cq / b.NS;
    const T* wc = w + c * b.kh * b.kw;
    union {
      T e[8];
      uint4 v;
    } u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int tap = strip_tap(b.kh, b.kw, b.pw, b.flip, b.W, b.jmax, q, ow, k0 + e);
      u.e[e] = tap >= 0 ? wc[tap] : from_f<T>(0.f);
    }
    *reinterpret_cast<uint4*>(cache + i * 8) = u.v;
  }
}

struct KCfg {
  int T, KB, R, h, ph, dmin, dmax, jmax, NS, W;
  int Ho, Wo;
  int G, NG;      // M tiles per unit, tile groups per channel
  int NCH;        // sample chunks per channel
  int nsets;      // accumulator sets (2: a unit's epilogue overlaps the next unit's MMAs)
  int nb;         // MMA N (samples per chunk rounded up to 16, at most 64)
  int acc_cols;   // tensor-memory columns per accumulator
  int ncols;      // tensor-memory columns allocated
  int stages;     // B stages in shared memory
  uint32_t idesc;
  uint32_t bbytes;        // one B atom (nb x 128 bytes)
  uint32_t stage_bytes;   // kAtoms * bbytes
  uint32_t strip_bytes;   // W * 128
  uint32_t strips_bytes;  // NS * strip_bytes
  int64_t N, C;
  int64_t in_off, out_ctot, out_off;
  int64_t units;  // C * NG * NCH
};

// Walk over this CTA's units u0..u1-1 as (channel c, tile group g, sample chunk n).
struct Units {
  int64_t c, u, u1;
  int g, n, NG, NCH;
  __device__ __forceinline__ Units(int64_t u0_, int64_t u1_, int NG_, int NCH_)
      : u(u0_), u1(u1_), NG(NG_), NCH(NCH_) {
    c = u0_ / ((int64_t)NG_ * NCH_);
    const int r = (int)(u0_ - c * NG_ * NCH_);
    g = r / NCH_;
    n = r - g * NCH_;
  }
  __device__ __forceinline__ bool more() const { return u < u1; }
  __device__ __forceinline__ void next() {
    ++u;
    if (++n == NCH) {
      n = 0;
      if (++g == NG) { g = 0; ++c; }
    }
  }
};

struct Ring {
  int s = 0, n = 1;
  uint32_t ph = 0;
  bool wrapped = false;
  __device__ __forceinline__ explicit Ring(int n_) : n(n_) {}
  __device__ __forceinline__ void next() {
    if (++s == n) { s = 0; ph ^= 1; wrapped = true; }
  }
};

// K steps of a unit with tiles t0..t1-1: the union of its tiles' ranges.
__host__ __device__ __forceinline__ void unit_range(const KCfg& g, int t0, int t1, int& lo, int& hi) {
  lo = t0 + g.dmin;
  hi = t1 - 1 + g.dmax + 1;
  if (lo < 0) lo = 0;
  if (hi > g.KB) hi = g.KB;
}

constexpr int kEpiThreads = 256;  // warps 0-7: epilogue; warp w reads lanes 32*(w%4).., column chunks of parity w/4
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr int kMaxSlots = 16;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
cached_kernel(KCfg g, const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap amap,
              unsigned int* timeouts, const T* __restrict__ bias, T* __restrict__ y, int accumulate_out) {
  extern __shared__ __align__(1024) unsigned char smdyn[];
  // fullS[s]: the producer's expect_tx arrival and the stage's bytes;
  // freeS[s]: the MMAs that read stage s are done; accfull / accfree per
  // accumulator slot; sfull: the channel's strips have landed; sfree: the
  // MMAs of the previous channel are done
  __shared__ __align__(8) uint64_t fullS[kMaxStages], freeS[kMaxStages], accfull[kMaxSlots], accfree[kMaxSlots],
      sfull, sfree, done;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  unsigned char* base = smdyn + ((1024 - (tma::smem_u32(smdyn) & 1023)) & 1023);
  unsigned char* strips = base;                   // the channel's strips (strips_bytes)
  unsigned char* stage0 = base + g.strips_bytes;  // B stages
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nslots = g.nsets * g.G;
  if (tid == 0) {
    for (int s = 0; s < g.stages; ++s) {
      tma::mbar_init(&fullS[s], 1);
      tma::mbar_init(&freeS[s], 1);
    }
    for (int s = 0; s < nslots; ++s) {
      tma::mbar_init(&accfull[s], 1);
      tma::mbar_init(&accfree[s], kEpiThreads);
    }
    tma::mbar_init(&sfull, 1);
    tma::mbar_init(&sfree, 1);
    tma::mbar_init(&done, 1);
    tma::fence_init();
    abort_s = 0;
  }
  if (warp == 0) tc::alloc(&tmem_base_s, g.ncols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base_s;
  volatile int* abortp = &abort_s;
  const int64_t u0 = (int64_t)blockIdx.x * g.units / gridDim.x;
  const int64_t u1 = (int64_t)(blockIdx.x + 1) * g.units / gridDim.x;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      Ring r(g.stages);
      uint32_t issued = 0, nload = 0;
      int64_t cur_c = -1;
      for (Units w(u0, u1, g.NG, g.NCH); w.more() && !*abortp; w.next()) {
        const int64_t c = w.c;
        const int t0 = w.g * g.G, t1 = min(g.T, t0 + g.G);
        if (c != cur_c) {
          // the previous channel's MMAs must be done before its strips are overwritten
          if (nload > 0 && !tc::wait(&sfree, (nload - 1) & 1, timeouts, abortp, kSleepNs)) { *abortp = 1; break; }
          tma::mbar_expect_tx(&sfull, g.strips_bytes);
          for (int q = 0; q < g.NS; ++q)
            tma::load_3d(strips + (size_t)q * g.strip_bytes, &amap, 0, (int)((c * g.NS + q) * g.W), 0, &sfull);
          ++nload;
          cur_c = c;
        }
        int lo, hi;
        unit_range(g, t0, t1, lo, hi);
        for (int kc = lo; kc < hi && !*abortp; ++kc, r.next()) {
          if (r.wrapped && !tc::wait(&freeS[r.s], r.ph ^ 1, timeouts, abortp, kSleepNs)) { *abortp = 1; break; }
          unsigned char* st = stage0 + (size_t)r.s * g.stage_bytes;
          tma::mbar_expect_tx(&fullS[r.s], g.stage_bytes);
#pragma unroll
          for (int a = 0; a < kAtoms; ++a)
            tma::load_3d(st + a * g.bbytes, &xmap, kc * kKs + a * kAtom, (int)(g.in_off + c), w.n * kNChunk,
                         &fullS[r.s]);
          ++issued;
        }
      }
      // every issued copy must land before the CTA leaves: the last uses of
      // the stages, and the last strip copy
      const uint32_t first = issued > (uint32_t)g.stages ? issued - g.stages : 0;
      for (uint32_t k = first; k < issued; ++k) tc::wait(&fullS[k % g.stages], (k / g.stages) & 1, nullptr, nullptr);
      if (nload > 0) tc::wait(&sfull, (nload - 1) & 1, nullptr, nullptr);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    Ring r(g.stages);
    uint32_t nch = 0, nunit = 0;
    uint32_t used = 0, uodd = 0;  // per slot: used before; number of uses so far is odd
    int64_t cur_c = -1;
    const uint32_t strips_addr = tma::smem_u32(strips);
    const uint32_t stage_addr = tma::smem_u32(stage0);
    for (Units w(u0, u1, g.NG, g.NCH); w.more(); w.next(), ++nunit) {
      if (w.c != cur_c) {
        if (cur_c >= 0) {
          if (tc::elect_one()) tc::commit(&sfree);
          __syncwarp();
        }
        bool ok = !*abortp && tc::wait(&sfull, nch & 1, timeouts, abortp);
        if (!__all_sync(0xffffffffu, ok)) *abortp = 1;
        ++nch;
        cur_c = w.c;
      }
      const int t0 = w.g * g.G, t1 = min(g.T, t0 + g.G);
      const int sbase = g.nsets == 2 ? (int)(nunit & 1) * g.G : 0;
      int lo, hi;
      unit_range(g, t0, t1, lo, hi);
      for (int kc = lo; kc < hi; ++kc, r.next()) {
        bool ok = !*abortp && tc::wait(&fullS[r.s], r.ph, timeouts, abortp);
        if (!__all_sync(0xffffffffu, ok)) { *abortp = 1; continue; }
        // tiles this K step reaches
        const int tlo = max(t0, kc - g.dmax), thi = min(t1, kc - g.dmin + 1);
        // a tile's first K step: the epilogue must have drained its slot
        for (int t = tlo; t < thi; ++t) {
          int first, end;
          k_range(g.dmin, g.dmax, g.KB, t, first, end);
          const int s = sbase + t - t0;
          if (kc != first) continue;
          if ((used >> s) & 1) {
            bool okf = tc::wait(&accfree[s], ((uodd >> s) & 1) ^ 1, timeouts, abortp);
            if (!__all_sync(0xffffffffu, okf)) *abortp = 1;
          }
          used |= 1u << s;
          uodd ^= 1u << s;
        }
        tc::fence_after();
        const uint32_t st = stage_addr + r.s * g.stage_bytes;
        if (!*abortp && tc::elect_one()) {
          // operand descriptors step by constants: the next tile's A operand
          // starts R strips (128 rows, 1024 descriptor units) further on,
          // atom 1's h strips (64 rows) before atom 0's; a K slice is 32 bytes
          const uint64_t a_lo = tc::desc_sw128(strips_addr + (uint32_t)strip_of(g.jmax, g.R, g.h, g.ph, kc - tlo, 0) *
                                                                 g.strip_bytes);
          const uint64_t b_lo = tc::desc_sw128(st);
          const uint32_t d_lo = tmem + (sbase + tlo - t0) * g.acc_cols;
          // tiles whose sums start at this K step
          uint32_t fresh = 0;
          for (int t = tlo; t < thi; ++t)
            if (kc == max(0, t + g.dmin)) fresh |= 1u << (t - tlo);
          const int nt = thi - tlo;
#pragma unroll
          for (int a = 0; a < kAtoms; ++a) {
#pragma unroll
            for (int ks = 0; ks < kAtom / 16; ++ks) {
              uint64_t ad = a_lo - 512 * a + 2 * ks;
              const uint64_t bd = b_lo + (uint64_t)((a * g.bbytes) >> 4) + 2 * ks;
              uint32_t dt = d_lo;
              for (int i = 0; i < nt; ++i, ad += 1024, dt += g.acc_cols)
                tc::mma_ss(dt, ad, bd, g.idesc, (a == 0 && ks == 0 && ((fresh >> i) & 1)) ? 0u : 1u);
            }
          }
          tc::commit(&freeS[r.s]);
          // tiles whose last K step this was go to the epilogue
          for (int t = tlo; t < thi; ++t) {
            int first, end;
            k_range(g.dmin, g.dmax, g.KB, t, first, end);
            if (kc == end - 1) tc::commit(&accfull[sbase + t - t0]);
          }
        }
        __syncwarp();
      }
    }
    // every MMA must be done before the tensor memory is freed
    if (tc::elect_one()) tc::commit(&done);
    __syncwarp();
    tc::wait(&done, 0, nullptr, nullptr);
    __syncwarp();
  } else {
    // ---- epilogue: warp w reads lanes 32*(w%4).., column chunks 2i + w/4 -----
    const int quarter = warp & 3, half = warp >> 2;
    const int m = quarter * 32 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(quarter * 32) << 16);
    const int64_t plane = (int64_t)g.Ho * g.Wo;
    const int64_t nstride = g.out_ctot * plane;
    uint32_t dodd = 0, nunit = 0;  // per slot: number of drains so far is odd
    for (Units w(u0, u1, g.NG, g.NCH); w.more(); w.next(), ++nunit) {
      const int64_t c = w.c;
      const int t0 = w.g * g.G, t1 = min(g.T, t0 + g.G);
      const int sbase = g.nsets == 2 ? (int)(nunit & 1) * g.G : 0;
      const int nbase = w.n * kNChunk;
      const float bv = bias ? ld(bias + c) : 0.f;
      for (int t = t0; t < t1; ++t) {
        const int s = sbase + t - t0;
        bool ok = !*abortp && tc::wait(&accfull[s], (dodd >> s) & 1, timeouts, abortp, kSleepNs);
        dodd ^= 1u << s;
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          tc::fence_after();
          const int f = t * kM + m;
          const bool mvalid = f < plane;
          T* o0 = y + (g.out_off + c) * plane + f + (int64_t)nbase * nstride;
          for (int n0 = 16 * half; n0 < g.nb; n0 += 32) {
            float v[16];
            tc::ld16(tlane + s * g.acc_cols + n0, v);
            if (mvalid) {
              T* o = o0 + (int64_t)n0 * nstride;
#pragma unroll
              for (int i = 0; i < 16; ++i, o += nstride) {
                if (nbase + n0 + i < g.N) {
                  const float val = v[i] + bv;
                  *o = from_f<T>(accumulate_out ? val + ld_rw(o) : val);
                }
              }
            }
          }
        } else {
          *abortp = 1;
        }
        tc::fence_before();
        tc::arrive(&accfree[s]);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::dealloc(tmem, g.ncols);
}

// Kernel shape for MMA N = nb: as many B stages (2..kMaxStages) as shared
// memory takes beside the strips; tile groups as large as the tensor memory
// holds (two accumulator sets when one set is at most half of it). False
// when the strips do not fit beside two stages of the largest N.
bool plan_kernel(const Geo& q, int nb, KCfg* k, size_t* smem) {
  const size_t strips = (size_t)q.NS * q.Wo * 128;
  const size_t fixed = 1024 + strips;
  if (fixed + 2 * (size_t)(kAtoms * kNChunk * 128) > kSmemLimit) return false;
  const uint32_t bb = (uint32_t)nb * 128;
  const size_t stage = (size_t)kAtoms * bb;
  int S = 0;
  while (S < kMaxStages && fixed + (S + 1) * stage <= kSmemLimit) ++S;
  const int acc_cols = tile::round_up(nb, 32);
  k->stages = S;
  k->bbytes = bb;
  k->stage_bytes = (uint32_t)stage;
  k->strip_bytes = (uint32_t)q.Wo * 128;
  k->strips_bytes = (uint32_t)strips;
  k->acc_cols = acc_cols;
  int gmax = 512 / acc_cols;
  if (gmax > kMaxSlots) gmax = kMaxSlots;
  k->NG = (q.T + gmax - 1) / gmax;
  k->G = (q.T + k->NG - 1) / k->NG;
  k->nsets = 2 * k->G * acc_cols <= 512 && 2 * k->G <= kMaxSlots ? 2 : 1;
  k->ncols = 32;
  while (k->ncols < k->nsets * k->G * acc_cols) k->ncols *= 2;
  *smem = fixed + S * stage;
  return true;
}

// The batch and plane sizes one cached call takes (the cache itself does not
// depend on them).
bool call_supported(const Conv& c, const Geo& q) {
  return c.N >= 1 && (c.N + kNChunk - 1) / kNChunk < (int64_t(1) << 24) && (int64_t)q.Hi * q.Wi < (int64_t(1) << 24) &&
         (int64_t)q.Ho * q.Wo < (int64_t(1) << 24);
}

template <typename T>
cudaError_t run(const Conv& c, const Geo& q, const void* in, const void* cache, const void* bias, void* out, bool acc,
                cudaStream_t s) {
  KCfg g{};
  g.T = q.T; g.KB = q.KB; g.R = q.R; g.h = q.h; g.ph = q.ph; g.dmin = q.dmin; g.dmax = q.dmax;
  g.jmax = q.jmax; g.NS = q.NS; g.W = q.Wo; g.Ho = q.Ho; g.Wo = q.Wo;
  g.nb = tile::round_up(c.N < kNChunk ? c.N : kNChunk, 16);
  g.NCH = (int)((c.N + kNChunk - 1) / kNChunk);
  size_t smem = 0;
  if (!plan_kernel(q, g.nb, &g, &smem)) return cudaErrorInvalidConfiguration;
  g.idesc = tc::idesc_f16(std::is_same<T, __nv_bfloat16>::value, kM, g.nb);
  g.N = c.N;
  g.C = c.C;
  int64_t in_ctot;
  if (q.flip) {  // input: the grad_out slice; output: grad_in
    in_ctot = c.ctot; g.in_off = c.off; g.out_ctot = c.C; g.out_off = 0;
  } else {
    in_ctot = c.C; g.in_off = 0; g.out_ctot = c.ctot; g.out_off = c.off;
  }
  g.units = c.C * g.NG * g.NCH;
  // input as [N][channels][Hi*Wi]: box = 64 positions x 1 channel x nb samples
  alignas(64) CUtensorMap xmap{};
  if (!tma::encode_3d_sw128(&xmap, in, c.dtype, (uint64_t)q.Hi * q.Wi, (uint64_t)in_ctot, (uint64_t)c.N,
                            (uint32_t)kAtom, 1, (uint32_t)g.nb))
    return cudaErrorInvalidValue;
  // cache as [C*NS*W rows][64]: box = one strip
  alignas(64) CUtensorMap amap{};
  if (!tma::encode_3d_sw128(&amap, cache, c.dtype, (uint64_t)kAtom, (uint64_t)c.C * q.NS * q.Wo, 1, (uint32_t)kAtom,
                            (uint32_t)q.Wo, 1))
    return cudaErrorInvalidValue;
  auto kern = cached_kernel<T>;
  cudaError_t e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  int smem_sm = 0;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
    return e;
  cudaFuncAttributes fa{};
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  // CTAs per SM from shared memory, capped so that resident CTAs never need
  // more than the 512 tensor-memory columns
  int occ = smem_sm / (int)(smem + fa.sharedSizeBytes + 1024);
  if (occ > 512 / g.ncols) occ = 512 / g.ncols;
  if (occ > 2) occ = 2;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return e;
  int64_t grid = (int64_t)sms * occ;
  if (grid > g.units) grid = g.units;
  if (grid < 1) return cudaSuccess;
  kern<<<(int)grid, kThreads, smem, s>>>(g, xmap, amap, tma::timeout_counter(), (const T*)bias, (T*)out,
                                         acc ? 1 : 0);
  return cudaGetLastError();
}

template <typename T>
cudaError_t build_t(const Conv& c, const Geo& q, const void* w, void* cache, cudaStream_t s) {
  BCfg b{};
  b.kh = q.kh; b.kw = q.kw; b.pw = q.pw; b.flip = q.flip; b.W = q.Wo; b.jmax = q.jmax; b.NS = q.NS; b.C = c.C;
  const int64_t total = c.C * q.NS * q.Wo * (kAtom / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  build_kernel<T><<<(int)blocks, 256, 0, s>>>(b, (const T*)w, (T*)cache);
  return cudaGetLastError();
}

}  // namespace

size_t cache_bytes(const Conv& c, bool flip) {
  Geo q;
  KCfg k{};
  size_t smem = 0;
  if (!make_geo(c, flip, &q) || !plan_kernel(q, kNChunk, &k, &smem)) return 0;
  return cache_bytes_of(c, q);
}

bool call_supported(const Conv& c, bool flip) {
  Geo q;
  return make_geo(c, flip, &q) && call_supported(c, q);
}

cudaError_t build(const Conv& c, bool flip, const void* w, void* cache, cudaStream_t s) {
  Geo q;
  if (!make_geo(c, flip, &q) || cache_bytes(c, flip) == 0) return cudaErrorInvalidValue;
  if (c.dtype == DWCONV_F16) return build_t<__half>(c, q, w, cache, s);
  return build_t<__nv_bfloat16>(c, q, w, cache, s);
}

cudaError_t run(const Conv& c, bool flip, const void* in, const void* cache, const void* bias, void* out, bool acc,
                cudaStream_t s) {
  Geo q;
  if (!make_geo(c, flip, &q) || !call_supported(c, q) || cache_bytes(c, flip) == 0) return cudaErrorInvalidValue;
  if (c.dtype == DWCONV_F16) return run<__half>(c, q, in, cache, bias, out, acc, s);
  return run<__nv_bfloat16>(c, q, in, cache, bias, out, acc, s);
}

}  // namespace ibc
}  // namespace dwconv
