// Channels-last (NHWC) forward: x [N, H, W, C], y [N, Ho, Wo, out_c_total].
//
// In this layout the C values of one pixel are contiguous, so a warp reads
// whole 128-byte lines of channels and the per-channel filters become
// per-lane vectors: the depthwise stencil is the same, only the vector axis
// moves from the image row to the channel. Two kernels:
//
//  - tiled (3x3, 5x5, 7x7; stride 1 or 2; dilation 1; one filter per
//    channel; C * element size a multiple of 16 bytes): a persistent CTA
//    walks (sample, tile row, tile column, channel group) units. Per unit one
//    thread issues a 4-D tensor-memory-accelerator copy of the input box
//    (channel group x box columns x box rows x 1 sample) into shared memory;
//    the copy's zero fill outside the tensor is the zero padding. Two stages:
//    the next unit's box lands while this one is computed. A channel group is
//    128 bytes of channels (32 fp32 or 64 fp16 / bf16); eight lanes cover it
//    with 16-byte vectors, and each of the CTA's 32 lane groups computes a
//    strip of PX consecutive output columns of one output row, accumulating
//    in fp32 and reading each input vector of the strip's window once.
//  - generic: one output per thread, channel fastest; every shape.
//
// Both apply the fused epilogue (scale, shift, activation) before the one
// rounding to the storage type.
#include "nhwc.h"
#include "tile.cuh"
#include "tma.cuh"
#include "vec.cuh"

namespace dwconv {
namespace nhwc {
namespace {

constexpr int kNT = 256;     // threads per CTA: 8 channel lanes x 32 strips

struct NCfg {
  int th, tw;            // output tile rows / columns
  int bh, bw;            // input box rows / columns
  int cg;                // channels per unit (128 bytes)
  int tiles_h, tiles_w, groups;
  int64_t units;         // below 2^31
  FastDiv d_per_n;       // units per sample: tiles_h * tiles_w * groups
  FastDiv d_tpr;         // units per tile row: tiles_w * groups
  FastDiv d_groups;
  int box_bytes;         // bh * bw * 128
  int stage_bytes;       // box, rounded up to 128 bytes
  int tab_floats;        // K*K*cg taps + bias, scale, shift (cg each)
  int vec_out;           // 16-byte output stores are aligned
};

// Resident CTAs the register budget is sized for: three where 80 registers
// hold the block without spilling (fp32, or stride 2), else two.
template <typename T, int S>
constexpr int min_ctas() { return (sizeof(T) == 4 || S == 2) ? 3 : 2; }

template <typename T, int K, int S, int PX>
__global__ void __launch_bounds__(kNT, (min_ctas<T, S>()))
tiled_kernel(Conv c, NCfg g, const __grid_constant__ CUtensorMap tmap, unsigned int* timeouts,
             const T* __restrict__ w, const T* __restrict__ bias, T* __restrict__ y, Epi ep) {
  constexpr int VEC = Vec<T>::n;
  constexpr int WIN = (PX - 1) * S + K;  // input columns of a strip's window
  extern __shared__ __align__(16) unsigned char smdyn[];
  __shared__ __align__(8) uint64_t bars[2];
  unsigned char* sm = smdyn + ((128 - (tma::smem_u32(smdyn) & 127)) & 127);
  if (threadIdx.x == 0) {
    tma::mbar_init(&bars[0], 1);
    tma::mbar_init(&bars[1], 1);
    tma::fence_init();
  }
  __syncthreads();
  unsigned char* const box0 = sm;
  unsigned char* const box1 = sm + g.stage_bytes;
  float* const tab0 = reinterpret_cast<float*>(sm + 2 * g.stage_bytes);
  float* const tab1 = tab0 + g.tab_floats;
  const int lc = threadIdx.x & 7;       // channel lane: channels lc*VEC .. lc*VEC + VEC - 1
  const int strip = threadIdx.x >> 3;   // output strip of the tile
  const int spr = g.tw / PX;            // strips per tile row
  const int sr = strip / spr, sc = strip - sr * spr;
  const bool strip_on = strip < g.th * spr;

  auto coords = [&](int64_t u, int& n, int& oh0, int& ow0, int& c0) {
    uint32_t q, thi, twi;
    uint32_t r = g.d_per_n.divmod((uint32_t)u, q);
    n = (int)q;
    r = g.d_tpr.divmod(r, thi);
    r = g.d_groups.divmod(r, twi);
    c0 = (int)r * g.cg;
    oh0 = (int)thi * g.th;
    ow0 = (int)twi * g.tw;
  };
  auto issue = [&](int64_t u, unsigned char* box, float* tab, uint64_t* bar) {
    int n, oh0, ow0, c0;
    coords(u, n, oh0, ow0, c0);
    if (threadIdx.x == 0) {
      tma::fence_async_smem();
      tma::mbar_expect_tx(bar, g.box_bytes);
      tma::load_4d(box, &tmap, c0, ow0 * S - c.pw, oh0 * S - c.ph, n, bar);
    }
    // filter taps transposed to [tap][channel], then bias, scale and shift
    const int kk = K * K;
    for (int i = threadIdx.x; i < g.cg * kk; i += kNT) {
      const int cl = i / kk, tap = i - cl * kk;
      const int ch = c0 + cl;
      tab[tap * g.cg + cl] = ch < c.C ? ld(w + (int64_t)ch * kk + tap) : 0.f;
    }
    float* bt = tab + kk * g.cg;
    for (int cl = threadIdx.x; cl < g.cg; cl += kNT) {
      const int ch = c0 + cl;
      const bool in = ch < c.C;
      bt[cl] = (bias && in) ? ld(bias + ch) : 0.f;
      bt[g.cg + cl] = (ep.scale && in) ? ld(reinterpret_cast<const T*>(ep.scale) + ch) : 1.f;
      bt[2 * g.cg + cl] = (ep.shift && in) ? ld(reinterpret_cast<const T*>(ep.shift) + ch) : 0.f;
    }
  };

  int64_t u = blockIdx.x;
  if (u < g.units) issue(u, box0, tab0, &bars[0]);
  for (int k = 0; u < g.units; ++k, u += gridDim.x) {
    const int64_t un = u + gridDim.x;
    const bool more = un < g.units;
    if (more) issue(un, (k & 1) ? box0 : box1, (k & 1) ? tab0 : tab1, &bars[(k + 1) & 1]);
    if (!tma::mbar_wait(&bars[k & 1], (uint32_t)(k >> 1) & 1, timeouts)) {
      // the copy never landed: let the one in flight finish (bounded), then stop
      if (more) tma::mbar_wait(&bars[(k + 1) & 1], (uint32_t)((k + 1) >> 1) & 1, nullptr);
      return;
    }
    __syncthreads();
    const unsigned char* box = (k & 1) ? box1 : box0;
    const float* tab = (k & 1) ? tab1 : tab0;
    int n, oh0, ow0, c0;
    coords(u, n, oh0, ow0, c0);
    const int oh = oh0 + sr;
    const int owb = ow0 + sc * PX;
    const int ch = c0 + lc * VEC;
    if (strip_on && oh < c.Ho && owb < c.Wo && ch < c.C) {
      const float* bt = tab + K * K * g.cg + lc * VEC;
      float acc[PX][VEC];
#pragma unroll
      for (int p = 0; p < PX; ++p)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[p][e] = bt[e];
#pragma unroll
      for (int a = 0; a < K; ++a) {
        float wr[K][VEC];
#pragma unroll
        for (int b = 0; b < K; ++b)
#pragma unroll
          for (int e = 0; e < VEC; e += 4) {
            const float4 f = *reinterpret_cast<const float4*>(tab + (a * K + b) * g.cg + lc * VEC + e);
            wr[b][e] = f.x; wr[b][e + 1] = f.y; wr[b][e + 2] = f.z; wr[b][e + 3] = f.w;
          }
        // input row sr*S + a of the box, columns sc*PX*S .. + WIN - 1, this lane's 16 bytes
        const unsigned char* rowp = box + ((int64_t)(sr * S + a) * g.bw + sc * PX * S) * 128 + lc * 16;
#pragma unroll
        for (int j = 0; j < WIN; ++j) {
          float xv[VEC];
          unpack16<T>(*reinterpret_cast<const uint4*>(rowp + j * 128), xv);
#pragma unroll
          for (int p = 0; p < PX; ++p) {
            const int b = j - p * S;
            if (b >= 0 && b < K) {
#pragma unroll
              for (int e = 0; e < VEC; ++e) acc[p][e] = fmaf(wr[b][e], xv[e], acc[p][e]);
            }
          }
        }
      }
      if (ep.active()) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float s_ = bt[g.cg + e], h_ = bt[2 * g.cg + e];
#pragma unroll
          for (int p = 0; p < PX; ++p) acc[p][e] = epi_act(fmaf(acc[p][e], s_, h_), ep.act);
        }
      }
      T* yp = y + (((int64_t)n * c.Ho + oh) * c.Wo + owb) * c.ctot + c.off + ch;
#pragma unroll
      for (int p = 0; p < PX; ++p) {
        if (owb + p >= c.Wo) break;
        T* q = yp + (int64_t)p * c.ctot;
        if (g.vec_out) {
          *reinterpret_cast<uint4*>(q) = pack16<T>(acc[p]);
        } else {
#pragma unroll
          for (int e = 0; e < VEC; ++e) q[e] = from_f<T>(acc[p][e]);
        }
      }
    }
    __syncthreads();
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
generic_kernel(Conv c, int64_t total, const T* __restrict__ x, const T* __restrict__ w,
               const T* __restrict__ bias, T* __restrict__ y, Epi ep) {
  const int64_t OC = c.C * c.m;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t oc = i % OC;
    int64_t r = i / OC;
    const int64_t ow = r % c.Wo;
    r /= c.Wo;
    const int64_t oh = r % c.Ho;
    const int64_t n = r / c.Ho;
    const int64_t ci = oc / c.m;
    float acc = bias ? ld(bias + oc) : 0.f;
    const T* wp = w + oc * c.kh * c.kw;
    for (int a = 0; a < c.kh; ++a) {
      const int64_t ih = oh * c.sh - c.ph + (int64_t)a * c.dh;
      if (ih < 0 || ih >= c.H) continue;
      for (int b = 0; b < c.kw; ++b) {
        const int64_t iw = ow * c.sw - c.pw + (int64_t)b * c.dw;
        if (iw < 0 || iw >= c.W) continue;
        acc = fmaf(ld(wp + a * c.kw + b), ld(x + ((n * c.H + ih) * c.W + iw) * c.C + ci), acc);
      }
    }
    if (ep.active()) {
      const float s_ = ep.scale ? ld(reinterpret_cast<const T*>(ep.scale) + oc) : 1.f;
      const float h_ = ep.shift ? ld(reinterpret_cast<const T*>(ep.shift) + oc) : 0.f;
      acc = epi_act(fmaf(acc, s_, h_), ep.act);
    }
    y[((n * c.Ho + oh) * c.Wo + ow) * c.ctot + c.off + oc] = from_f<T>(acc);
  }
}

template <int S>
constexpr int px_of() { return S == 1 ? 4 : 2; }

constexpr size_t kMaxSmem = 200 * 1024;

// two input boxes, two filter tables, alignment slack
size_t tiled_smem(const NCfg& g) { return 2 * (size_t)g.stage_bytes + 2 * (size_t)g.tab_floats * 4 + 128; }

// Tile shape: among the 32-strip shapes, the one whose units carry the
// fewest box bytes plus output slots for this plane (ragged tiles waste both).
bool plan_tiled(const Conv& c, int px, NCfg* out) {
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  NCfg best{};
  double best_cost = -1;
  const int shapes[4][2] = {{8, 4}, {16, 2}, {4, 8}, {32, 1}};  // rows, strips per row
  for (auto& sh : shapes) {
    NCfg g{};
    g.th = sh[0];
    g.tw = sh[1] * px;
    g.bh = (g.th - 1) * c.sh + c.kh;
    g.bw = (g.tw - 1) * c.sw + c.kw;
    if (g.bh > 256 || g.bw > 256) continue;
    g.cg = 128 / es;
    g.tiles_h = (int)((c.Ho + g.th - 1) / g.th);
    g.tiles_w = (int)((c.Wo + g.tw - 1) / g.tw);
    g.groups = (int)((c.C + g.cg - 1) / g.cg);
    g.units = (int64_t)c.N * g.tiles_h * g.tiles_w * g.groups;
    if (g.units >= (int64_t(1) << 31)) continue;
    g.d_per_n = FastDiv((uint32_t)g.tiles_h * g.tiles_w * g.groups);
    g.d_tpr = FastDiv((uint32_t)g.tiles_w * g.groups);
    g.d_groups = FastDiv((uint32_t)g.groups);
    g.box_bytes = g.bh * g.bw * 128;
    g.stage_bytes = (g.box_bytes + 127) / 128 * 128;
    g.tab_floats = (c.kh * c.kw + 3) * g.cg;
    const double cost = (double)g.units * (g.box_bytes + 2.0 * g.th * g.tw * 128);
    if (tiled_smem(g) > kMaxSmem) continue;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = g;
    }
  }
  if (best_cost < 0) return false;
  *out = best;
  return true;
}

template <typename T, int K, int S>
cudaError_t launch_tiled(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                         const Epi& ep) {
  constexpr int PX = px_of<S>();
  NCfg g;
  if (!plan_tiled(c, PX, &g)) return cudaErrorNotSupported;
  const int es = sizeof(T);
  g.vec_out = ((c.off * es) % 16 == 0 && (c.ctot * es) % 16 == 0 &&
               reinterpret_cast<uintptr_t>(y) % 16 == 0) ? 1 : 0;
  CUtensorMap map;
  if (!tma::encode_4d(&map, x, c.dtype, (uint64_t)c.C, (uint64_t)c.W, (uint64_t)c.H, (uint64_t)c.N,
                      (uint32_t)g.cg, (uint32_t)g.bw, (uint32_t)g.bh, 1))
    return cudaErrorNotSupported;
  unsigned int* to = tma::timeout_counter();
  if (!to) return cudaErrorNotSupported;
  auto kern = tiled_kernel<T, K, S, PX>;
  const size_t smem = tiled_smem(g);
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = tile::persistent_grid(kern, smem, g.units);
  kern<<<grid, kNT, smem, s>>>(c, g, map, to, (const T*)w, (const T*)b, (T*)y, ep);
  return cudaGetLastError();
}

template <typename T>
cudaError_t run_tiled(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                      const Epi& ep) {
#define X(K, S) \
  if (c.kh == K && c.sh == S) return launch_tiled<T, K, S>(c, x, w, b, y, s, ep);
  DW_NHWC_CASES(X)
#undef X
  return cudaErrorNotSupported;
}

template <typename T>
cudaError_t run_generic(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                        const Epi& ep) {
  const int64_t total = c.N * c.Ho * c.Wo * c.C * c.m;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (blocks < 1) blocks = 1;
  generic_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(c, total, (const T*)x, (const T*)w, (const T*)b, (T*)y, ep);
  return cudaGetLastError();
}

}  // namespace

bool tiled_supported(const Conv& c) {
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  bool shape = false;
#define X(K, S) shape = shape || (c.kh == K && c.kw == K && c.sh == S && c.sw == S);
  DW_NHWC_CASES(X)
#undef X
  if (!shape || c.dh != 1 || c.dw != 1 || c.m != 1) return false;
  if ((c.C * es) % 16 != 0) return false;
  // tensor-map limits: dimension sizes below 2^32, box coordinates in int
  if (c.C >= (int64_t(1) << 31) || c.W >= (int64_t(1) << 31) || c.H >= (int64_t(1) << 31) ||
      c.N >= (int64_t(1) << 31))
    return false;
  NCfg g;
  return plan_tiled(c, c.sh == 1 ? 4 : 2, &g);
}

Algo plan(const Conv& c) { return tiled_supported(c) ? Algo::Nhwc : Algo::Generic; }

cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s,
                const Epi& ep) {
  cudaError_t e = cudaErrorNotSupported;
  // a misaligned x rules the tensor-map copy out for this call only
  if (plan(c) == Algo::Nhwc && reinterpret_cast<uintptr_t>(x) % 16 == 0) {
    DWCONV_DISPATCH_DTYPE(c.dtype, T, e = run_tiled<T>(c, x, w, b, y, s, ep));
    if (e != cudaErrorNotSupported) return e;
  }
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = run_generic<T>(c, x, w, b, y, s, ep));
  return e;
}

}  // namespace nhwc
}  // namespace dwconv
