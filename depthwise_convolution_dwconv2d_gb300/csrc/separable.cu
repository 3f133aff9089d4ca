// Depthwise-separable block, channels-last (x [N, H, W, C], y [N, Ho, Wo,
// out_c_total]):
//   z = act1(scale1 * dwconv(x) + shift1)     C*m depthwise channels, rounded
//                                             to the storage type
//   y = act2(scale2 * (Wp z) + shift2)        cout channels, Wp [cout, C*m]
// The depthwise layer and the 1x1 layer after it, as the MobileNet table of
// "Spatial Depthwise Convolution on the GPU #3057" times them one after the
// other; here z never leaves the chip.
//
// Tensor-core kernel (fp16 / bf16; 3x3 or 5x5, stride 1 or 2, dilation 1,
// one filter per channel, C a multiple of 64). The pointwise step is the GEMM
//   D[p, co] = sum_ci Z[p, ci] * Wp[co, ci]
// over a tile of 128 output pixels p (M) and a tile of nt <= 256 output
// channels (N), K = C in chunks of 64 channels. Both operands are K-major with
// the 128-byte swizzle: Z because a pixel's channels are contiguous, Wp
// because PyTorch stores the 1x1 filter as [cout][cin]. Warp roles, handing
// work on through mbarriers:
//  * producer (warp 12, one lane): per K chunk, one tensor-map copy of the
//    input box the tile's depthwise windows read (64 channels x box columns x
//    box rows x images; zero fill is the padding) and one of the 64-channel
//    slice of Wp for the tile's output channels (128-byte swizzle);
//  * builders (warps 0-7): the depthwise stage for the chunk -- each thread
//    one 16-byte group of 8 channels for a strip of 4 adjacent pixels of a
//    tile row, fp32 accumulation over the box, epilogue 1, rounding -- stored
//    straight into the A stage in the swizzled operand layout;
//  * MMA issuer (warp 13): four K=16 tcgen05.mma per chunk into one of two
//    fp32 accumulators in tensor memory; commits free the stage and hand a
//    finished tile to the epilogue;
//  * epilogue (warps 8-11): tcgen05.ld of the accumulator, epilogue 2,
//    rounding, 32-byte stores per pixel.
// A tile is 128 pixel slots: nimg images x th rows x twp column slots (twp =
// tw rounded up to 4 so a builder's strip never crosses a row); slots past
// the output are computed from the box's zero fill and never stored. Small
// planes pack whole images into one tile.
//
// Every wait is bounded; a wait that gives up raises the CTA's abort flag and
// every role then runs through its loops without waiting, waits (bounded)
// for its own copies and MMAs in flight, frees the tensor memory and returns.
//
// Generic kernel (any dtype and shape): a CTA stages z for a run of pixels in
// shared memory in fp32 (after the same rounding), then computes the
// pointwise sums one output per thread.
#include <type_traits>

#include "nhwc.h"
#include "tc.cuh"
#include "tile.cuh"
#include "tma.cuh"
#include "vec.cuh"

namespace dwconv {
namespace sep {
namespace {

constexpr int kBuilders = 256;
constexpr int kEpiWarp0 = 8;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kThreads = 14 * 32;
constexpr int kM = 128;          // pixel slots per tile (MMA M)
constexpr int kKc = 64;          // channels per K chunk (one 128-byte swizzle row)
constexpr int kMaxStages = 2;
constexpr unsigned kSleepNs = 64;
// Epilogue-2 table: scale2 and shift2 of every output channel (fp32), staged
// once per CTA when cout is at most kEpiTab channels.
constexpr int64_t kEpiTab = 2048;

struct SCfg {
  int nimg, th, tw, twp;   // tile: images x rows x (valid columns, column slots)
  int bh, bw;              // input box rows / columns
  int tiles_h, tiles_w;
  int nt, nq;              // output channels per tile (MMA N) / tiles over cout
  int nkc;                 // K chunks
  int stages;
  int64_t N, Ho, Wo, cout, ctot, off;
  int H, W, ph, pw;
  int64_t units;           // below 2^31
  FastDiv d_nq, d_tpg, d_tw;
  uint32_t box_bytes, b_bytes, stage_bytes, tab_floats;
  int acc_cols, nacc, ncols;
  uint32_t idesc;
  int vec_out;
};

struct Epis {
  const void* s1;
  const void* h1;
  const void* s2;
  const void* h2;
  int a1, a2;
};

// Unit u = (tile t, output-channel tile q), q fastest: consecutive units of a
// CTA reuse the tile's input boxes from L2.
struct UnitPos {
  int n0, oh0, ow0, co0;
};
__device__ __forceinline__ UnitPos unit_pos(const SCfg& g, int64_t u) {
  uint32_t t, grp, thi;
  const uint32_t q = g.d_nq.divmod((uint32_t)u, t);
  const uint32_t tig = g.d_tpg.divmod(t, grp);
  const uint32_t twi = g.d_tw.divmod(tig, thi);
  return UnitPos{(int)grp * g.nimg, (int)thi * g.th, (int)twi * g.tw, (int)q * g.nt};
}

struct Ring {
  int s = 0;
  uint32_t ph = 0;
  bool wrapped = false;
  __device__ __forceinline__ void next(int stages) {
    if (++s == stages) { s = 0; ph ^= 1; wrapped = true; }
  }
};

__device__ __forceinline__ void builders_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kBuilders) : "memory");
}

template <typename T, int K, int S>
__global__ void __launch_bounds__(kThreads, 1)
septc_kernel(SCfg g, const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
             unsigned int* timeouts, const T* __restrict__ wd, Epis ep, T* __restrict__ y) {
  constexpr int WIN = 3 * S + K;  // input columns of a 4-pixel strip's window
  extern __shared__ __align__(1024) unsigned char smdyn[];
  __shared__ __align__(8) uint64_t fullB[kMaxStages], afull[kMaxStages], freeS[kMaxStages], accfull[2],
      accfree[2], done;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  unsigned char* sm = smdyn + ((1024 - (tma::smem_u32(smdyn) & 1023)) & 1023);
  float* const tab0 = reinterpret_cast<float*>(sm + (size_t)g.stages * g.stage_bytes);
  // epilogue-2 scale / shift table after the two filter-table slots (empty
  // when cout is too large: the epilogue then reads global memory)
  float* const etab = tab0 + 2 * g.tab_floats;
  const bool use_etab = g.cout <= kEpiTab;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < g.stages; ++s) {
      tma::mbar_init(&fullB[s], 1);
      tma::mbar_init(&afull[s], kBuilders);
      tma::mbar_init(&freeS[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tma::mbar_init(&accfull[s], 1);
      tma::mbar_init(&accfree[s], 128);
    }
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
  auto A_of = [&](int s) { return sm + (size_t)s * g.stage_bytes; };
  auto B_of = [&](int s) { return sm + (size_t)s * g.stage_bytes + kM * 128; };
  auto box_of = [&](int s) { return sm + (size_t)s * g.stage_bytes + kM * 128 + g.b_bytes; };

  if (warp == kProducerWarp) {
    // ---- producer -----------------------------------------------------------
    if (lane == 0) {
      Ring r;
      uint32_t issued = 0;
      for (int64_t u = u0; u < u1 && !*abortp; ++u) {
        const UnitPos up = unit_pos(g, u);
        for (int kc = 0; kc < g.nkc && !*abortp; ++kc, r.next(g.stages)) {
          if (r.wrapped && !tc::wait(&freeS[r.s], r.ph ^ 1, timeouts, abortp, kSleepNs)) { *abortp = 1; break; }
          tma::mbar_expect_tx(&fullB[r.s], g.box_bytes + g.b_bytes);
          tma::load_4d(box_of(r.s), &xmap, kc * kKc, up.ow0 * S - g.pw, up.oh0 * S - g.ph, up.n0, &fullB[r.s]);
          tma::load_3d(B_of(r.s), &wmap, kc * kKc, up.co0, 0, &fullB[r.s]);
          ++issued;
        }
      }
      // every issued copy lands before the CTA leaves
      const uint32_t first = issued > (uint32_t)g.stages ? issued - g.stages : 0;
      for (uint32_t k = first; k < issued; ++k)
        tc::wait(&fullB[k % g.stages], (k / g.stages) & 1, nullptr, nullptr);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer -------------------------------------------------------------
    Ring r;
    uint32_t tiles = 0;
    for (int64_t u = u0; u < u1; ++u, ++tiles) {
      const int ab = tiles & (g.nacc - 1);
      const uint32_t ause = g.nacc == 2 ? tiles >> 1 : tiles;
      bool okf = ause == 0 || tc::wait(&accfree[ab], (ause - 1) & 1, timeouts, abortp);
      if (!__all_sync(0xffffffffu, okf)) *abortp = 1;
      tc::fence_after();
      const uint32_t dt = tmem + ab * g.acc_cols;
      for (int kc = 0; kc < g.nkc; ++kc, r.next(g.stages)) {
        bool ok = !*abortp && tc::wait(&fullB[r.s], r.ph, timeouts, abortp) &&
                  tc::wait(&afull[r.s], r.ph, timeouts, abortp);
        if (!__all_sync(0xffffffffu, ok)) { *abortp = 1; continue; }
        tc::fence_after();
        const uint64_t ad = tc::desc_sw128(tma::smem_u32(A_of(r.s)));
        const uint64_t bd = tc::desc_sw128(tma::smem_u32(B_of(r.s)));
        if (tc::elect_one()) {
#pragma unroll
          for (int k = 0; k < kKc / 16; ++k)  // 32 bytes = 2 descriptor units per K=16 step
            tc::mma_ss(dt, ad + 2 * k, bd + 2 * k, g.idesc, (kc > 0 || k > 0) ? 1u : 0u);
          tc::commit(&freeS[r.s]);
        }
        __syncwarp();
      }
      if (tc::elect_one()) tc::commit(&accfull[ab]);
      __syncwarp();
    }
    if (tc::elect_one()) tc::commit(&done);
    __syncwarp();
    tc::wait(&done, 0, nullptr, nullptr);
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ---- epilogue: warp 8+q reads lanes 32q..32q+31 = pixel slots ---------------
    const int q = warp - kEpiWarp0;
    const int p = q * 32 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(q * 32) << 16);
    const int per_img = g.th * g.twp;
    const int img = p / per_img, rem = p - img * per_img;
    const int r_ = rem / g.twp, col = rem - r_ * g.twp;
    const T* s2 = reinterpret_cast<const T*>(ep.s2);
    const T* h2 = reinterpret_cast<const T*>(ep.h2);
    if (use_etab) {
      for (int64_t i = p; i < g.cout; i += 128) {
        etab[2 * i] = s2 ? ld(s2 + i) : 1.f;
        etab[2 * i + 1] = h2 ? ld(h2 + i) : 0.f;
      }
      asm volatile("bar.sync 2, 128;\n" ::: "memory");  // the four epilogue warps
    }
    uint32_t tiles = 0;
    for (int64_t u = u0; u < u1; ++u, ++tiles) {
      const UnitPos up = unit_pos(g, u);
      const int ab = tiles & (g.nacc - 1);
      const uint32_t ause = g.nacc == 2 ? tiles >> 1 : tiles;
      bool ok = !*abortp && tc::wait(&accfull[ab], ause & 1, timeouts, abortp, kSleepNs);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc::fence_after();
        const int64_t n = up.n0 + img;
        const int64_t oh = up.oh0 + r_, ow = up.ow0 + col;
        const bool valid = img < g.nimg && n < g.N && r_ < g.th && oh < g.Ho && col < g.tw && ow < g.Wo;
        T* yp = y + ((n * g.Ho + oh) * g.Wo + ow) * g.ctot + g.off + up.co0;
        for (int n0 = 0; n0 < g.nt; n0 += 16) {
          float v[16];
          tc::ld16(tlane + ab * g.acc_cols + n0, v);
          const int co = up.co0 + n0;
          if (!valid || co >= g.cout) continue;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = co + i < g.cout ? co + i : co;
            float sc, sh;
            if (use_etab) {
              const float2 t2 = *reinterpret_cast<const float2*>(etab + 2 * c);
              sc = t2.x;
              sh = t2.y;
            } else {
              sc = s2 ? ld(s2 + c) : 1.f;
              sh = h2 ? ld(h2 + c) : 0.f;
            }
            v[i] = epi_act(fmaf(v[i], sc, sh), ep.a2);
          }
          if (g.vec_out && co + 16 <= g.cout) {
            uint4* d = reinterpret_cast<uint4*>(yp + n0);
            d[0] = pack16<T>(v);
            d[1] = pack16<T>(v + 8);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (co + i < g.cout) yp[n0 + i] = from_f<T>(v[i]);
          }
        }
      } else {
        *abortp = 1;
      }
      tc::fence_before();
      tc::arrive(&accfree[ab]);
    }
  } else {
    // ---- builders: the depthwise stage into the A operand ------------------------
    const int j = tid & 7;          // channel group of 8 (16 bytes)
    const int strip = tid >> 3;     // slots 4*strip .. 4*strip + 3
    const int p0 = 4 * strip;
    const int per_img = g.th * g.twp;
    const int img = p0 / per_img, rem = p0 - img * per_img;
    const int r_ = rem / g.twp, col0 = rem - r_ * g.twp;
    const bool used = p0 < g.nimg * per_img;
    const T* s1 = reinterpret_cast<const T*>(ep.s1);
    const T* h1 = reinterpret_cast<const T*>(ep.h1);
    // A chunk's filters as [tap][channel], then scale1 and shift1, in one of
    // two table slots (chunk t in slot t & 1). Every builder holds its share
    // of the next chunk's table in registers, loaded one chunk ahead so the
    // global loads overlap the current chunk's work, and stores it just
    // before the builders' barrier: the slot it writes was last read two
    // chunks earlier, which every builder finished before the previous
    // barrier.
    constexpr int tabn = K * K * kKc + 2 * kKc;
    constexpr int TPT = (tabn + kBuilders - 1) / kBuilders;  // table values per builder
    float pre[TPT];
    auto fetch_tab = [&](int kc) {
      const int c0 = kc * kKc;
#pragma unroll
      for (int q = 0; q < TPT; ++q) {
        const int i = tid + q * kBuilders;
        float v = 0.f;
        if (i < K * K * kKc) {
          const int cl = i / (K * K), tap = i - cl * (K * K);
          v = ld(wd + (int64_t)(c0 + cl) * (K * K) + tap);
        } else if (i < K * K * kKc + kKc) {
          v = s1 ? ld(s1 + c0 + (i - K * K * kKc)) : 1.f;
        } else if (i < tabn) {
          v = h1 ? ld(h1 + c0 + (i - K * K * kKc - kKc)) : 0.f;
        }
        pre[q] = v;
      }
    };
    auto store_tab = [&](float* tab) {
#pragma unroll
      for (int q = 0; q < TPT; ++q) {
        const int i = tid + q * kBuilders;
        if (i < K * K * kKc) {
          const int cl = i / (K * K), tap = i - cl * (K * K);
          tab[tap * kKc + cl] = pre[q];
        } else if (i < tabn) {
          tab[i] = pre[q];
        }
      }
    };
    if (u0 < u1) fetch_tab(0);
    uint32_t t = 0;
    Ring r;
    for (int64_t u = u0; u < u1; ++u) {
      for (int kc = 0; kc < g.nkc; ++kc, r.next(g.stages), ++t) {
        float* tab = tab0 + (t & 1) * g.tab_floats;
        store_tab(tab);
        builders_sync();
        // the next chunk of this CTA's walk: kc + 1, or chunk 0 of the next unit
        if (kc + 1 < g.nkc) fetch_tab(kc + 1);
        else if (u + 1 < u1) fetch_tab(0);
        if (!*abortp && !tc::wait(&fullB[r.s], r.ph, timeouts, abortp, kSleepNs)) *abortp = 1;
        unsigned char* A = A_of(r.s);
        uint4 out[4];
        if (used && !*abortp) {
          // channels (2i, 2i + 1) of the thread's 8 are one lane pair of the
          // two-lane FMA (taps, inputs and sums pair up without moves)
          f32x2 accp[4][4];
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int i = 0; i < 4; ++i) accp[p][i] = 0ull;
          const unsigned char* box = box_of(r.s);
#pragma unroll
          for (int a = 0; a < K; ++a) {
            f32x2 wr[K][4];
#pragma unroll
            for (int b = 0; b < K; ++b) {
              const ulonglong2 f0 = *reinterpret_cast<const ulonglong2*>(tab + (a * K + b) * kKc + 8 * j);
              const ulonglong2 f1 = *reinterpret_cast<const ulonglong2*>(tab + (a * K + b) * kKc + 8 * j + 4);
              wr[b][0] = f0.x; wr[b][1] = f0.y; wr[b][2] = f1.x; wr[b][3] = f1.y;
            }
            const unsigned char* rowp =
                box + ((size_t)((img * g.bh + r_ * S + a) * g.bw + col0 * S)) * 128 + j * 16;
#pragma unroll
            for (int jj = 0; jj < WIN; ++jj) {
              f32x2 xv[4];
              unpack16_pairs<T>(*reinterpret_cast<const uint4*>(rowp + jj * 128), xv);
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                const int b = jj - p * S;
                if (b >= 0 && b < K) {
#pragma unroll
                  for (int i = 0; i < 4; ++i) fma_f32x2(accp[p][i], wr[b][i], xv[i]);
                }
              }
            }
          }
          float acc[4][8];
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int i = 0; i < 4; ++i) unpack_f32x2(accp[p][i], acc[p][2 * i], acc[p][2 * i + 1]);
          const float* st = tab + K * K * kKc + 8 * j;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[p][e] = epi_act(fmaf(acc[p][e], st[e], st[kKc + e]), ep.a1);
            out[p] = pack16<T>(acc[p]);
          }
        } else {
#pragma unroll
          for (int p = 0; p < 4; ++p) out[p] = make_uint4(0, 0, 0, 0);
        }
        // row p of the 128-byte-swizzled K-major operand: 16-byte group j at
        // position j ^ (p % 8)
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int row = p0 + p;
          *reinterpret_cast<uint4*>(A + (row >> 3) * 1024 + (row & 7) * 128 + ((j ^ (row & 7)) << 4)) = out[p];
        }
        tma::fence_async_smem();
        tc::arrive(&afull[r.s]);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 0) tc::dealloc(tmem, g.ncols);
}

template <typename T>
__global__ void __launch_bounds__(256)
sep_generic_kernel(Conv c, int64_t cout, int64_t ctot, int64_t off, int P, const T* __restrict__ x,
                   const T* __restrict__ wd, const T* __restrict__ wp, Epis ep, T* __restrict__ y) {
  extern __shared__ __align__(16) float zs[];
  const int64_t cin = c.C * c.m;
  const int64_t npix = c.N * c.Ho * c.Wo;
  const T* s1 = reinterpret_cast<const T*>(ep.s1);
  const T* h1 = reinterpret_cast<const T*>(ep.h1);
  const T* s2 = reinterpret_cast<const T*>(ep.s2);
  const T* h2 = reinterpret_cast<const T*>(ep.h2);
  for (int64_t pb = (int64_t)blockIdx.x * P; pb < npix; pb += (int64_t)gridDim.x * P) {
    const int np = (int)((npix - pb) < P ? (npix - pb) : P);
    // depthwise stage for pixels pb .. pb + np - 1, all cin channels
    for (int64_t i = threadIdx.x; i < (int64_t)np * cin; i += blockDim.x) {
      const int64_t pl = i / cin, oc = i - pl * cin;
      const int64_t pix = pb + pl;
      const int64_t ow = pix % c.Wo, t = pix / c.Wo, oh = t % c.Ho, n = t / c.Ho;
      const int64_t ci = oc / c.m;
      float acc = 0.f;
      for (int a = 0; a < c.kh; ++a) {
        const int64_t ih = oh * c.sh - c.ph + (int64_t)a * c.dh;
        if (ih < 0 || ih >= c.H) continue;
        for (int b = 0; b < c.kw; ++b) {
          const int64_t iw = ow * c.sw - c.pw + (int64_t)b * c.dw;
          if (iw < 0 || iw >= c.W) continue;
          acc = fmaf(ld(wd + (oc * c.kh + a) * c.kw + b), ld(x + ((n * c.H + ih) * c.W + iw) * c.C + ci), acc);
        }
      }
      acc = epi_act(fmaf(acc, s1 ? ld(s1 + oc) : 1.f, h1 ? ld(h1 + oc) : 0.f), ep.a1);
      zs[i] = to_f<T>(from_f<T>(acc));  // z rounded to the storage type
    }
    __syncthreads();
    for (int64_t i = threadIdx.x; i < (int64_t)np * cout; i += blockDim.x) {
      const int64_t pl = i / cout, co = i - pl * cout;
      const float* z = zs + pl * cin;
      const T* w = wp + co * cin;
      float acc = 0.f;
      for (int64_t ci = 0; ci < cin; ++ci) acc = fmaf(ld(w + ci), z[ci], acc);
      acc = epi_act(fmaf(acc, s2 ? ld(s2 + co) : 1.f, h2 ? ld(h2 + co) : 0.f), ep.a2);
      y[(pb + pl) * ctot + off + co] = from_f<T>(acc);
    }
    __syncthreads();
  }
}

// ---- host planning ----------------------------------------------------------------

inline size_t epi_tab_bytes(const SCfg& g) { return g.cout <= kEpiTab ? (size_t)g.cout * 8 : 0; }
size_t tc_smem(const SCfg& g) {
  return 1024 + (size_t)g.stages * g.stage_bytes + (size_t)2 * g.tab_floats * 4 + epi_tab_bytes(g);
}

// Tile shape and stages for the tensor-core kernel; false if the shape is
// not one it takes or nothing fits in shared memory.
bool plan_tc(const Conv& c, int64_t cout, SCfg* out) {
  if (c.dtype != DWCONV_F16 && c.dtype != DWCONV_BF16) return false;
  if (c.m != 1 || c.kh != c.kw || (c.kh != 3 && c.kh != 5) || c.sh != c.sw || (c.sh != 1 && c.sh != 2)) return false;
  if (c.dh != 1 || c.dw != 1 || c.C % kKc != 0 || cout < 1 || cout > (1 << 20)) return false;
  if (c.N >= (1 << 30) || c.H >= (1 << 30) || c.W >= (1 << 30) || c.C >= (1 << 30)) return false;
  const int K = c.kh, S = c.sh;
  SCfg g{};
  g.N = c.N; g.Ho = c.Ho; g.Wo = c.Wo; g.cout = cout;
  g.H = (int)c.H; g.W = (int)c.W; g.ph = c.ph; g.pw = c.pw;
  // column slots per tile row: Wo rounded up to 4, at most 128 and small
  // enough that the box stays within 256 columns
  int twp_max = ((256 - K) / S + 1) / 4 * 4;
  if (twp_max > kM) twp_max = kM;
  const int64_t wo4 = (c.Wo + 3) / 4 * 4;
  if (wo4 <= twp_max) {
    g.tw = (int)c.Wo;
    g.twp = (int)wo4;
  } else {
    g.tw = g.twp = twp_max;
  }
  g.th = kM / g.twp;
  if (g.th >= c.Ho) {
    g.th = (int)c.Ho;
    g.nimg = kM / (g.th * g.twp);
  } else {
    g.nimg = 1;
  }
  g.bw = (g.twp - 1) * S + K;
  g.bh = (g.th - 1) * S + K;
  if (g.bw > 256 || g.bh > 256 || g.nimg > 256) return false;
  g.tiles_h = (int)((c.Ho + g.th - 1) / g.th);
  g.tiles_w = (int)((c.Wo + g.tw - 1) / g.tw);
  const int64_t groups = (c.N + g.nimg - 1) / g.nimg;
  g.nkc = (int)(c.C / kKc);
  g.box_bytes = (uint32_t)(128 * g.bw * g.bh * g.nimg);
  g.tab_floats = (uint32_t)((K * K + 2) * kKc);
  // output channels per tile: all of them up to 256, else 256 (the depthwise
  // stage is recomputed per output-channel tile); two pipeline stages if any
  // tile width down to 64 fits them, else one stage at the widest that fits
  const int nt_first = cout <= 256 ? (int)((cout + 15) / 16 * 16) : 256;
  auto set_nt = [&](int nt, int stages) {
    g.nt = nt;
    g.b_bytes = (uint32_t)nt * 128;
    g.stage_bytes = (uint32_t)(kM * 128) + g.b_bytes + (g.box_bytes + 1023) / 1024 * 1024;
    g.stages = stages;
    return tc_smem(g) <= 220 * 1024;
  };
  bool ok = false;
  for (int pass = 0; pass < 2 && !ok; ++pass) {
    for (int nt = nt_first; nt >= 16 && !ok; nt = nt > 64 ? nt / 2 / 16 * 16 : nt - 16) {
      if (pass == 0 && nt < 64 && nt < nt_first) break;
      ok = set_nt(nt, pass == 0 ? 2 : 1);
    }
  }
  if (!ok) return false;
  g.nq = (int)((cout + g.nt - 1) / g.nt);
  g.units = groups * g.tiles_h * g.tiles_w * g.nq;
  if (g.units >= (int64_t(1) << 31) || g.units < 1) return false;
  g.d_nq = FastDiv((uint32_t)g.nq);
  g.d_tpg = FastDiv((uint32_t)(g.tiles_h * g.tiles_w));
  g.d_tw = FastDiv((uint32_t)g.tiles_w);
  g.acc_cols = (g.nt + 31) / 32 * 32;
  g.nacc = 2 * g.acc_cols <= 512 ? 2 : 1;
  g.ncols = 32;
  while (g.ncols < g.nacc * g.acc_cols) g.ncols *= 2;
  g.idesc = tc::idesc_f16(c.dtype == DWCONV_BF16, kM, g.nt);
  *out = g;
  return true;
}

template <typename T, int K, int S>
cudaError_t launch_tc(SCfg g, const Conv& c, const void* x, const void* wd, const void* wp, const Epis& ep,
                      void* y, cudaStream_t s) {
  alignas(64) CUtensorMap xmap{}, wmap{};
  if (!tma::encode_4d(&xmap, x, c.dtype, (uint64_t)c.C, (uint64_t)c.W, (uint64_t)c.H, (uint64_t)c.N,
                      (uint32_t)kKc, (uint32_t)g.bw, (uint32_t)g.bh, (uint32_t)g.nimg))
    return cudaErrorNotSupported;
  if (!tma::encode_3d_sw128(&wmap, wp, c.dtype, (uint64_t)c.C, (uint64_t)g.cout, 1, (uint32_t)kKc,
                            (uint32_t)g.nt, 1))
    return cudaErrorNotSupported;
  unsigned int* to = tma::timeout_counter();
  if (!to) return cudaErrorNotSupported;
  auto kern = septc_kernel<T, K, S>;
  size_t smem = tc_smem(g);
  cudaError_t e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // resident CTAs per SM from registers, threads and shared memory; never
  // more than the 512 tensor-memory columns hold (grow the shared-memory
  // request until few enough fit)
  cudaFuncAttributes fa{};
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  int smem_sm = 0, regs_sm = 0, thr_sm = 0;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev)) != cudaSuccess) return e;
  const int regs_cta = (kThreads / 32) * ((fa.numRegs * 32 + 255) / 256 * 256);
  const int by_regs = regs_sm / regs_cta, by_thr = thr_sm / kThreads;
  const int tmem_cap = 512 / g.ncols;
  int occ = 0;
  for (;;) {
    const int by_smem = smem_sm / (int)(smem + fa.sharedSizeBytes + 1024);
    occ = by_regs < by_thr ? by_regs : by_thr;
    if (by_smem < occ) occ = by_smem;
    if (occ < 1) return cudaErrorNotSupported;
    if (occ <= tmem_cap) break;
    smem += 8 * 1024;
  }
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return e;
  int64_t grid = (int64_t)sms * occ;
  if (grid > g.units) grid = g.units;
  kern<<<(int)grid, kThreads, smem, s>>>(g, xmap, wmap, to, (const T*)wd, ep, (T*)y);
  return cudaGetLastError();
}

template <typename T>
cudaError_t run_tc(const SCfg& g, const Conv& c, const void* x, const void* wd, const void* wp, const Epis& ep,
                   void* y, cudaStream_t s) {
  if (c.kh == 3 && c.sh == 1) return launch_tc<T, 3, 1>(g, c, x, wd, wp, ep, y, s);
  if (c.kh == 3 && c.sh == 2) return launch_tc<T, 3, 2>(g, c, x, wd, wp, ep, y, s);
  if (c.kh == 5 && c.sh == 1) return launch_tc<T, 5, 1>(g, c, x, wd, wp, ep, y, s);
  if (c.kh == 5 && c.sh == 2) return launch_tc<T, 5, 2>(g, c, x, wd, wp, ep, y, s);
  return cudaErrorNotSupported;
}

// Pixels per CTA of the generic kernel: z for them in at most 96 KB.
int generic_pixels(const Conv& c) {
  const int64_t cin = c.C * c.m;
  int64_t P = (96 * 1024) / (cin * 4);
  if (P > 32) P = 32;
  return (int)P;
}

template <typename T>
cudaError_t run_generic(const Conv& c, int64_t cout, int64_t ctot, int64_t off, const void* x, const void* wd,
                        const void* wp, const Epis& ep, void* y, cudaStream_t s) {
  const int P = generic_pixels(c);
  if (P < 1) return cudaErrorNotSupported;
  const size_t smem = (size_t)P * c.C * c.m * 4;
  auto kern = sep_generic_kernel<T>;
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int64_t npix = c.N * c.Ho * c.Wo;
  int64_t blocks = (npix + P - 1) / P;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  kern<<<(unsigned)blocks, 256, smem, s>>>(c, cout, ctot, off, P, (const T*)x, (const T*)wd, (const T*)wp, ep,
                                           (T*)y);
  return cudaGetLastError();
}

}  // namespace

bool supported(const Conv& c) { return generic_pixels(c) >= 1; }

Algo plan(const Conv& c, int64_t cout) {
  SCfg g;
  return plan_tc(c, cout, &g) ? Algo::SepTc : Algo::Generic;
}

cudaError_t run(const Conv& c, int64_t cout, int64_t ctot, int64_t off, const void* x, const void* wd,
                const void* s1, const void* h1, int a1, const void* wp, const void* s2, const void* h2, int a2,
                void* y, cudaStream_t s) {
  const Epis ep{s1, h1, s2, h2, a1, a2};
  SCfg g;
  // tensor maps need 16-byte aligned bases
  if (plan_tc(c, cout, &g) && reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(wp) % 16 == 0) {
    g.ctot = ctot;
    g.off = off;
    const int es = c.dtype == DWCONV_F32 ? 4 : 2;
    g.vec_out = ((off * es) % 16 == 0 && (ctot * es) % 16 == 0 && reinterpret_cast<uintptr_t>(y) % 16 == 0) ? 1 : 0;
    cudaError_t e = cudaErrorNotSupported;
    if (c.dtype == DWCONV_F16) e = run_tc<__half>(g, c, x, wd, wp, ep, y, s);
    if (c.dtype == DWCONV_BF16) e = run_tc<__nv_bfloat16>(g, c, x, wd, wp, ep, y, s);
    if (e != cudaErrorNotSupported) return e;
  }
  cudaError_t e = cudaErrorInvalidValue;
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = run_generic<T>(c, cout, ctot, off, x, wd, wp, ep, y, s));
  return e;
}

}  // namespace sep
}  // namespace dwconv
