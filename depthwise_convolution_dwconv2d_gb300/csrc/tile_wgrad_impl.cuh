// Small-kernel weight and bias gradients, first pass, on shared-memory tiles.
//
// partial[chunk, oc, a*K + b] = sum over (n, oh, ow) in the chunk of
//     gy[n, off + oc, oh, ow] * x[n, oc/m, oh*S - ph + a*D, ow*S - pw + b*D]
// partial[chunk, oc, K*K]   = sum of gy over the chunk (bias gradient)
// ("Spatial Depthwise Convolution on the GPU #3057", the grad-weight kernel
// extended to padding, stride and dilation, and grad_bias.)
//
// A CTA owns one input channel c (all m of its output channels) and a fixed
// chunk of the batch. It stages x and grad_out tiles in shared memory; each
// thread keeps all K*K (+1) sums for its outputs in registers, walking an
// R x V block of output positions at a time with a register window over the
// x tile rows. At the end the CTA reduces the per-thread sums with a warp
// butterfly and an ordered sum over warps and writes one partial per chunk;
// the second pass (generic.cu) adds the chunks in index order. Every sum has
// a fixed order, so the result is bitwise reproducible.
#pragma once
#include "plan.h"
#include "tile_cases.h"
#include "tma.cuh"
#include "tile.cuh"

namespace dwconv {
namespace tile {
namespace {

struct WCfg {
  int spc;         // slices (sample, band) per chunk: chunk q holds slices [q spc, (q + 1) spc)
  int chunks;
  int th, nbands;  // output rows per band, bands per plane
  int tr, pitch;   // x tile rows / pitch (elements)
  int gpitch;      // grad_out tile pitch (th rows)
  int rb, cb;
  int ppc;         // slices (sample, band) staged at once
  int x_elems, g_elems;  // x tile per slice, grad_out tile per plane
  int xstride, gstride;  // slice strides of the x and grad_out regions
  int goff;              // element offset of the grad_out region in a stage
  int stage_elems;
  int xmode, xix0, cshift;  // x tile copy mode / origin / window shift
  int gmode;
  int tma;                  // stage with tensor copies (x and grad_out maps)
  uint32_t tma_bytes;       // bytes per full stage (one band per plane)
  uint32_t tma_slice_bytes; // bytes per slice (banded planes)
  int xseg, gseg;           // dense staging segment sizes (x, grad_out)
  int stg_off, gstg_off;    // element offsets of the dense staging regions in a stage
  FastDiv trdiv, thdiv, d_per, d_cb, d_nbands;
};

template <typename T, int K, int S, int D, int M, int R, int V, int DL>
__global__ void __launch_bounds__(kNT)
wgrad_kernel(Conv c, WCfg g, const __grid_constant__ CUtensorMap xmap,
             const __grid_constant__ CUtensorMap gmap, unsigned int* timeouts,
             const T* __restrict__ x, const T* __restrict__ gy, float* __restrict__ ws) {
  extern __shared__ __align__(16) unsigned char smdyn[];
  __shared__ __align__(8) uint64_t bars[2];
  unsigned char* smraw = smdyn + ((128 - (tma::smem_u32(smdyn) & 127)) & 127);
  if (g.tma && threadIdx.x == 0) {
    tma::mbar_init(&bars[0], 1);
    tma::mbar_init(&bars[1], 1);
    tma::fence_init();
  }
  __syncthreads();
  constexpr int KK = K * K;
  constexpr int NV = M * (KK + 1);
  constexpr int U = (R - 1) * S + (K - 1) * D + 1;
  constexpr int WN = (V - 1) * S + (K - 1) * D + 1;
  constexpr int W4 = (DL + WN + 3) / 4 * 4;
  T* const buf[2] = {reinterpret_cast<T*>(smraw), reinterpret_cast<T*>(smraw) + g.stage_elems};
  float* red = reinterpret_cast<float*>(reinterpret_cast<T*>(smraw) + 2 * g.stage_elems);  // [warps][NV]
  const int64_t units = c.C * g.chunks;
  // slices of a unit: global slice q * spc + sl = (sample, band) =
  // (slice / nbands, slice % nbands) for sl < unit_slices(u)
  // unit u = chunk * C + channel (units < 2^32: the host caps chunks)
  auto unit_split = [&](int64_t uu, int64_t& ch, int& chunk) {
    uint32_t q;
    ch = c.dC.divmod((uint32_t)uu, q);
    chunk = (int)q;
  };
  auto unit_slices = [&](int64_t u) {
    int64_t ch_;
    int chunk;
    unit_split(u, ch_, chunk);
    const int64_t s_first = (int64_t)chunk * g.spc;
    const int64_t left = c.N * g.nbands - s_first;
    return left > 0 ? (int)(left < g.spc ? left : g.spc) : 0;
  };
  auto issue = [&](int64_t u, int s0, T* dst, uint64_t* bar) {
    int64_t ch;
    int chunk;
    unit_split(u, ch, chunk);
    // (one band per plane: slices are samples and n0 the chunk's first one)
    const int64_t n0 = (int64_t)chunk * g.spc;
    const int nsl = unit_slices(u);
    const int ns = (nsl - s0) < g.ppc ? (nsl - s0) : g.ppc;
    T* xs = dst;
    T* gs = dst + g.goff;
    if (!g.tma && (g.xmode == kCopyDense || g.gmode == kCopyDense)) {
      // whole planes (one band): x and grad_out each dense or row-wise
      if (g.xmode == kCopyDense)
        issue_flat<T>(dst + g.stg_off, ns, g.xseg, [&](int q) { return x + c.x_base(n0 + s0 + q, ch); },
                      (int)(c.H * c.W));
      else
        issue_tile<T>(xs, ns, g.xstride, g.pitch, [&](int q) { return x + c.x_base(n0 + s0 + q, ch); },
                      (int)c.H, (int)c.W, -c.ph, g.tr, g.trdiv, g.xix0, g.xmode);
      if (g.gmode == kCopyDense)
        issue_flat<T>(dst + g.gstg_off, ns * M, g.gseg,
                      [&](int qj) { return gy + c.y_base(n0 + s0 + qj / M, ch * M + qj % M); },
                      (int)(c.Ho * c.Wo));
      else
        issue_tile<T>(gs, ns * M, g.g_elems, g.gpitch,
                      [&](int qj) { return gy + c.y_base(n0 + s0 + qj / M, ch * M + qj % M); },
                      (int)c.Ho, (int)c.Wo, 0, g.th, g.thdiv, 0, g.gmode);
      return;
    }
    if (g.tma) {
      if (threadIdx.x == 0) {
        tma::fence_async_smem();
        if (g.nbands == 1) {
          tma::mbar_expect_tx(bar, g.tma_bytes);
          tma::load_4d(xs, &xmap, g.xix0, -c.ph, (int)ch, (int)(n0 + s0), bar);
          tma::load_4d(gs, &gmap, 0, 0, (int)(c.off + ch * M), (int)(n0 + s0), bar);
        } else {
          tma::mbar_expect_tx(bar, g.tma_slice_bytes * ns);
          for (int q = 0; q < ns; ++q) {
            const int64_t sl = (int64_t)chunk * g.spc + s0 + q;  // global slice
            uint32_t sq;
            const int oh0 = (int)g.d_nbands.divmod((uint32_t)sl, sq) * g.th;
            const int n = (int)sq;
            tma::load_4d(xs + q * g.xstride, &xmap, g.xix0, oh0 * S - c.ph, (int)ch, n, bar);
            tma::load_4d(gs + q * g.gstride, &gmap, 0, oh0, (int)(c.off + ch * M), n, bar);
          }
        }
      }
    } else if (g.nbands == 1) {
      issue_tile<T>(xs, ns, g.xstride, g.pitch, [&](int q) { return x + c.x_base(n0 + s0 + q, ch); },
                    (int)c.H, (int)c.W, -c.ph, g.tr, g.trdiv, g.xix0, g.xmode);
      issue_tile<T>(gs, ns * M, g.g_elems, g.gpitch,
                    [&](int qj) { return gy + c.y_base(n0 + s0 + qj / M, ch * M + qj % M); },
                    (int)c.Ho, (int)c.Wo, 0, g.th, g.thdiv, 0, g.gmode);
    } else {
      for (int q = 0; q < ns; ++q) {
        const int64_t sl = (int64_t)chunk * g.spc + s0 + q;  // global slice
        uint32_t sq;
        const int oh0 = (int)g.d_nbands.divmod((uint32_t)sl, sq) * g.th;
        const int64_t n = sq;
        issue_tile<T>(xs + q * g.xstride, 1, g.xstride, g.pitch, [&](int) { return x + c.x_base(n, ch); },
                      (int)c.H, (int)c.W, oh0 * S - c.ph, g.tr, g.trdiv, g.xix0, g.xmode);
        issue_tile<T>(gs + q * g.gstride, M, g.g_elems, g.gpitch,
                      [&](int j) { return gy + c.y_base(n, ch * M + j); }, (int)c.Ho, (int)c.Wo, oh0,
                      g.th, g.thdiv, 0, g.gmode);
      }
    }
  };
  // the CTA's steps: (unit u, first slice s0) for its units u = blockIdx.x + i*gridDim.x
  int64_t u = blockIdx.x;
  int s0 = 0;
  auto advance = [&](int64_t& uu, int& ss) {
    ss += g.ppc;
    if (ss >= unit_slices(uu)) {
      ss = 0;
      uu += gridDim.x;
    }
  };
  // skip empty units (never happens with the host's chunking, kept for safety)
  if (u < units) issue(u, s0, buf[0], &bars[0]);
  cp_async_commit();
  float acc[M][KK + 1];
#pragma unroll
  for (int j = 0; j < M; ++j)
#pragma unroll
    for (int i = 0; i <= KK; ++i) acc[j][i] = 0.f;
  for (int k = 0; u < units; ++k) {
    int64_t un = u;
    int sn = s0;
    advance(un, sn);
    if (un < units) issue(un, sn, (k & 1) ? buf[0] : buf[1], &bars[(k + 1) & 1]);
    cp_async_commit();
    cp_async_wait<1>();
    if (g.tma && !tma::mbar_wait(&bars[k & 1], (uint32_t)(k >> 1) & 1, timeouts)) {
      if (un < units) tma::mbar_wait(&bars[(k + 1) & 1], (uint32_t)((k + 1) >> 1) & 1, nullptr);
      return;
    }
    __syncthreads();
    T* const cbuf = (k & 1) ? buf[1] : buf[0];
    const T* xs = cbuf;
    const T* gs = xs + g.goff;
    const int nsl = unit_slices(u);
    const int ns = (nsl - s0) < g.ppc ? (nsl - s0) : g.ppc;
    int64_t chu;
    int chunku;
    unit_split(u, chu, chunku);
    const int64_t n0u = (int64_t)chunku * g.spc;  // (used by whole-plane staging only)
    const int per = (int)g.d_per.d;
    for (int it = threadIdx.x; it < ns * per; it += kNT) {
      uint32_t q_, rbi_;
      const uint32_t rem = g.d_per.divmod((uint32_t)it, q_);
      const int cbi = (int)g.d_cb.divmod(rem, rbi_);
      const int q = (int)q_, rbi = (int)rbi_;
      float gv[M][R][V];
      if (g.gmode == kCopyDense) {
#pragma unroll
        for (int j = 0; j < M; ++j) {
          const T* gp = dense_plane(cbuf + g.gstg_off, g.gseg, q * M + j,
                                    gy + c.y_base(n0u + s0 + q, chu * M + j));
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int oh = rbi * R + r;
#pragma unroll
            for (int v = 0; v < V; ++v) {
              const int ow = cbi * V + v;
              gv[j][r][v] = (oh < c.Ho && ow < c.Wo) ? ld1<T>(gp + oh * c.Wo + ow) : 0.f;
            }
            acc[j][KK] += (gv[j][r][0] + gv[j][r][1]) + (gv[j][r][2] + gv[j][r][3]);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < M; ++j)
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float f[4];
            ld4<T>(gs + q * g.gstride + j * g.g_elems + (rbi * R + r) * g.gpitch + cbi * V, f);
#pragma unroll
            for (int v = 0; v < V; ++v) gv[j][r][v] = f[v];
            acc[j][KK] += (f[0] + f[1]) + (f[2] + f[3]);
          }
      }
      const bool xd = g.xmode == kCopyDense;
      const T* xp = xd ? dense_plane(cbuf + g.stg_off, g.xseg, q, x + c.x_base(n0u + s0 + q, chu)) : nullptr;
      const int iyb = rbi * R * S - c.ph, ixb = cbi * V * S - c.pw;  // dense: plane coordinates
      bool cin[WN];
#pragma unroll
      for (int i = 0; i < WN; ++i) cin[i] = (unsigned)(ixb + i) < (unsigned)c.W;
      const T* t = xs + q * g.xstride + (rbi * R * S) * g.pitch + cbi * V * S + g.cshift;
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        if (!row_used<K, D, R, S>(uu)) continue;
        float win[W4];
        if (xd) {
          const int iy = iyb + uu;
          if ((unsigned)iy >= (unsigned)c.H) continue;
#pragma unroll
          for (int i = 0; i < WN; ++i) win[DL + i] = cin[i] ? ld1<T>(xp + iy * c.W + ixb + i) : 0.f;
        } else {
#pragma unroll
          for (int i = 0; i < W4 / 4; ++i) ld4<T>(t + uu * g.pitch + 4 * i, win + 4 * i);
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int a = 0; a < K; ++a) {
            if (r * S + a * D != uu) continue;
#pragma unroll
            for (int j = 0; j < M; ++j)
#pragma unroll
              for (int b = 0; b < K; ++b)
#pragma unroll
                for (int v = 0; v < V; ++v)
                  acc[j][a * K + b] = fmaf(gv[j][r][v], win[DL + v * S + b * D], acc[j][a * K + b]);
          }
      }
    }
    const bool last = s0 + g.ppc >= nsl;
    if (last) {
      // CTA reduction: warp butterfly, then warps summed in order.
      const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
      for (int j = 0; j < M; ++j)
#pragma unroll
        for (int i = 0; i <= KK; ++i) {
          float v = acc[j][i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) red[warp * NV + j * (KK + 1) + i] = v;
          acc[j][i] = 0.f;
        }
      __syncthreads();
      int64_t ch;
      int chunk;
      unit_split(u, ch, chunk);
      for (int i = threadIdx.x; i < NV; i += kNT) {
        float sum = 0.f;
        for (int wi = 0; wi < kNT / 32; ++wi) sum += red[wi * NV + i];
        const int j = i / (KK + 1), tap = i - j * (KK + 1);
        ws[((int64_t)chunk * c.OC() + ch * M + j) * (KK + 1) + tap] = sum;
      }
    }
    __syncthreads();
    u = un;
    s0 = sn;
  }
}

template <int K, int S> struct WBlk { static constexpr int R = S == 1 ? 2 : 1, V = 4; };

template <typename T, int K, int S, int D, int M, int DL>
cudaError_t launch_wgrad(const Conv& c, const WCfg& g, const CUtensorMap& xmap, const CUtensorMap& gmap,
                         const void* x, const void* gy, float* ws, cudaStream_t s) {
  constexpr int R = WBlk<K, S>::R, V = WBlk<K, S>::V;
  auto kern = wgrad_kernel<T, K, S, D, M, R, V, DL>;
  const size_t smem = 128 + 2 * (size_t)g.stage_elems * sizeof(T) + (kNT / 32) * M * (K * K + 1) * 4;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = persistent_grid(kern, smem, c.C * g.chunks);
  kern<<<grid, kNT, smem, s>>>(c, g, xmap, gmap, tma::timeout_counter(), (const T*)x, (const T*)gy, ws);
  return cudaGetLastError();
}

template <typename T, int K, int S, int D, int M>
cudaError_t run_wgrad_t(const Conv& c, const void* x, const void* gy, float* ws, int chunks,
                        cudaStream_t s) {
  constexpr int R = WBlk<K, S>::R, V = WBlk<K, S>::V;
  constexpr int ES = sizeof(T);
  constexpr int PA = 16 / ES > 4 ? 16 / ES : 4;  // pitch alignment (elements)
  WCfg g{};
  if (chunks < 1) return cudaErrorInvalidConfiguration;
  g.chunks = chunks;
  g.cb = (int)((c.Wo + V - 1) / V);
  g.gpitch = round_up((int64_t)g.cb * V, PA);
  int ix0 = 0, shift = 0, gshift = 0;
  g.xmode = pick_mode<T>(x, c.W, -c.pw, &ix0, &shift);
  g.xix0 = ix0;
  const int dl = shift % 4;
  g.cshift = shift - dl;
  g.gmode = pick_mode<T>(gy, c.Wo, 0, &ix0, &gshift);  // origin 0 is always a chunk boundary
  const int W4 = (dl + (V - 1) * S + (K - 1) * D + 1 + 3) / 4 * 4;
  g.pitch = round_up((int64_t)(g.cb - 1) * V * S + g.cshift + W4, PA);
  auto tr_of = [&](int64_t th) { return (th - 1) * S + (int64_t)(K - 1) * D + 1; };
  auto bytes_of = [&](int64_t th) { return (tr_of(th) * g.pitch + M * th * g.gpitch) * ES; };
  const int64_t target = 32 * 1024;
  int64_t th = (c.Ho + R - 1) / R * R;
  if (bytes_of(th) > target) {
    th = R;
    while (bytes_of(th + R) <= target) th += R;
    if (bytes_of(th) > 48 * 1024) return cudaErrorInvalidConfiguration;
  }
  g.th = (int)th;
  g.rb = (int)(th / R);
  g.nbands = (int)((c.Ho + th - 1) / th);
  g.d_nbands = FastDiv((uint32_t)g.nbands);
  // the chunks split the N x nbands slices evenly (chunks past the last
  // slice stay empty and write zero partials)
  {
    const int64_t total = c.N * g.nbands;
    int64_t spc = (total + chunks - 1) / chunks;
    if (spc < 1) spc = 1;
    if (total > (int64_t)0x7fffffff) return cudaErrorInvalidConfiguration;
    g.spc = (int)spc;
  }
  g.tr = (int)tr_of(th);
  g.x_elems = g.tr * g.pitch;
  g.g_elems = (int)(th * g.gpitch);
  g.trdiv = FastDiv((uint32_t)g.tr);
  g.thdiv = FastDiv((uint32_t)g.th);
  g.d_per = FastDiv((uint32_t)(g.rb * g.cb));
  g.d_cb = FastDiv((uint32_t)g.cb);
  const int64_t items = (int64_t)g.rb * g.cb;
  int64_t ppc = (2 * kNT + items - 1) / items;
  const int64_t cap = target / bytes_of(th);
  if (ppc > cap) ppc = cap;
  const int64_t slices = g.spc;
  if (ppc > slices) ppc = slices;
  if (ppc < 1) ppc = 1;
  // tensor copies when both tensors allow 16-byte rows and the boxes fit
  alignas(64) CUtensorMap xmap{}, gmap{};
  g.tma = g.xmode == kCopy16 && g.gmode == kCopy16 && g.pitch <= 256 && g.tr <= 256 && g.gpitch <= 256 &&
          g.th <= 256 && ppc <= 256;
  // (a chunk's last box may run past the chunk: the extra samples are
  // copied but not used, and samples past the batch are zero-filled)
  if (g.tma) {
    const uint32_t bp = g.nbands == 1 ? (uint32_t)ppc : 1u;
    g.tma = tma::encode_4d(&xmap, x, c.dtype, c.W, c.H, c.C, c.N, g.pitch, g.tr, 1, bp) &&
            tma::encode_4d(&gmap, gy, c.dtype, c.Wo, c.Ho, c.ctot, c.N, g.gpitch, g.th, M, bp);
  }
  g.ppc = (int)ppc;
  // slices land densely inside one box when a plane is one band; banded
  // slices are separate copies, each starting on a 128-byte boundary
  constexpr int A128 = 128 / ES;
  if (g.nbands == 1) {
    g.xstride = g.x_elems;
    g.gstride = M * g.g_elems;
    g.goff = round_up((int64_t)g.ppc * g.xstride, A128);
  } else {
    g.xstride = round_up(g.x_elems, A128);
    g.gstride = round_up((int64_t)M * g.g_elems, A128);
    g.goff = g.ppc * g.xstride;
  }
  g.stage_elems = stage_round((int64_t)g.goff + (int64_t)g.ppc * g.gstride, ES);
  // dense staging of whole planes whose rows are not 16-byte multiples
  if (!g.tma && g.nbands == 1) {
    if ((g.xmode == kCopy4 || g.xmode == kCopySync) && (reinterpret_cast<uintptr_t>(x) % 16) == 0)
      g.xmode = kCopyDense;
    if ((g.gmode == kCopy4 || g.gmode == kCopySync) && (reinterpret_cast<uintptr_t>(gy) % 16) == 0)
      g.gmode = kCopyDense;
  }
  if (g.xmode == kCopyDense || g.gmode == kCopyDense) {
    // a dense tensor is read in place from its staging segments
    if (g.xmode == kCopyDense) g.xstride = 0;
    if (g.gmode == kCopyDense) g.gstride = 0;
    g.goff = round_up((int64_t)g.ppc * g.xstride, A128);
    g.stage_elems = stage_round((int64_t)g.goff + (int64_t)g.ppc * g.gstride, ES);
    g.xseg = g.xmode == kCopyDense ? dense_seg<T>(c.H * c.W) : 0;
    g.gseg = g.gmode == kCopyDense ? dense_seg<T>(c.Ho * c.Wo) : 0;
    g.stg_off = g.stage_elems;
    g.gstg_off = stage_round((int64_t)g.stg_off + (int64_t)g.ppc * g.xseg, ES);
    g.stage_elems = stage_round((int64_t)g.gstg_off + (int64_t)g.ppc * M * g.gseg, ES);
  }
  g.tma_slice_bytes = (uint32_t)((g.x_elems + (int64_t)M * g.g_elems) * ES);
  g.tma_bytes = g.tma_slice_bytes * g.ppc;
  switch (dl) {
    case 0: return launch_wgrad<T, K, S, D, M, 0>(c, g, xmap, gmap, x, gy, ws, s);
    case 1: return launch_wgrad<T, K, S, D, M, 1>(c, g, xmap, gmap, x, gy, ws, s);
    case 2: return launch_wgrad<T, K, S, D, M, 2>(c, g, xmap, gmap, x, gy, ws, s);
    default: return launch_wgrad<T, K, S, D, M, 3>(c, g, xmap, gmap, x, gy, ws, s);
  }
}

}  // namespace

// Dispatch over the compiled cases with multiplier MSEL only (each
// multiplier's kernels are compiled in their own translation unit).
template <typename T, int MSEL>
cudaError_t wgrad_sel_t(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
#define X(K, S, D, M)                                                                      \
  if constexpr (M == MSEL) {                                                                \
    if (c.kh == K && c.sh == S && c.dh == D && c.m == M) return run_wgrad_t<T, K, S, D, M>(c, x, gy, ws, chunks, s); \
  }
  DW_WGRAD_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace tile
}  // namespace dwconv
