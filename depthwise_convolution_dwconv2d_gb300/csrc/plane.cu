// Small-plane depthwise kernels (3x3 filters, stride 1 or 2, rows of at most
// 32 elements), one warp per group of whole planes.
//
// The "Spatial Depthwise Convolution on the GPU #3057" kernels compute one
// output per thread straight from global memory; the tile kernels stage bands
// of many planes per CTA. For the small MobileNet planes (7², 14², 28²) both
// spend most of their instructions on indexing and staging, so here a warp
// works alone on a few whole planes:
//  * it copies the planes (coalesced, row by row) into its own zero-haloed
//    tile in shared memory -- no CTA barrier, no staging pipeline; latency
//    is hidden by the many warps resident on an SM;
//  * each lane owns one output column of one plane (two or four planes per
//    warp when the planes are narrow) and walks the output rows with the
//    K x K window held in registers (a stride-1 step loads one new row of
//    K values), so an output costs K loads, K*K FMAs and a store, with no
//    bounds checks.
// The same correlation kernel serves the forward and the stride-1
// grad-input (grad_out correlated with the filter rotated by 180 degrees,
// padding K-1-p); the weight-gradient first pass accumulates K*K + 1 sums
// per lane and reduces them in a fixed order into one partial per
// (chunk, channel). Measured against the tile kernels on the MobileNet
// layers, these win for the forward and stride-1 grad-input on rows of
// 9..16 elements and for the weight gradient on output rows of at most 16;
// the planner uses them there only.
#include "plan.h"
#include "tile.cuh"

namespace dwconv {
namespace plane {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxW = 32;  // widest input / output row (one lane per column)

struct PCfg {
  int Hin, Win, Hout, Wout;  // planes read / written
  int pad;                   // padding of the evaluated correlation
  int L, P;                  // lanes per plane (power of two >= output columns), planes per warp (32 / L)
  int Lw;                    // lanes per row when loading (power of two >= Win, <= 32)
  int TR, TP, TS;            // tile rows, pitch and floats per plane
  int64_t nplanes, groups;   // planes, groups of P planes
  int nb;                    // weight gradient: samples per chunk
};

int pow2_at_least(int v) {
  int p = 1;
  while (p < v) p *= 2;
  return p;
}

// Copy plane rows (Hin x Win, from src) into a tile whose element (r, col) is
// source (r - off, col - off), keeping only the tile's TR x TP window.
__device__ __forceinline__ void load_rows_setup(const PCfg& g, int lane, int& lr, int& lc, int& rstep) {
  lr = lane / g.Lw;
  lc = lane - lr * g.Lw;
  rstep = 32 / g.Lw;
}

// fp32 planes are copied with 4-byte asynchronous copies (all in flight at
// once, completed by the caller's cp_async_wait); 16-bit planes are widened
// through registers.
template <typename T>
__device__ __forceinline__ void load_plane(float* __restrict__ dst, const T* __restrict__ src, const PCfg& g,
                                           int off, int lr, int lc, int rstep) {
  if (lc >= g.Win || lc + off >= g.TP) return;
  int rend = g.TR - off;
  if (rend > g.Hin) rend = g.Hin;
  if (sizeof(T) == 4) {
    for (int r = lr; r < rend; r += rstep)
      tile::cp_async4(dst + (r + off) * g.TP + lc + off, src + r * g.Win + lc, 4);
  } else {
#pragma unroll 4
    for (int r = lr; r < rend; r += rstep) dst[(r + off) * g.TP + lc + off] = ld(src + r * g.Win + lc);
  }
}

// One warp's walk over work items first, first + step, ...: item k+1 is
// copied into the other tile buffer while item k is computed.
template <typename Issue, typename Compute>
__device__ __forceinline__ void warp_walk(int64_t first, int64_t step, int64_t end, float* buf0, float* buf1,
                                          Issue issue, Compute compute) {
  if (first < end) issue(first, buf0);
  tile::cp_async_commit();
  int k = 0;
  for (int64_t it = first; it < end; it += step, ++k) {
    const int64_t nx = it + step;
    if (nx < end) issue(nx, (k & 1) ? buf0 : buf1);
    tile::cp_async_commit();
    tile::cp_async_wait<1>();
    __syncwarp();
    compute(it, (k & 1) ? buf1 : buf0);
    __syncwarp();
  }
  tile::cp_async_wait<0>();
}

// out[oy][ox] = bias + sum_{a,b} w'[a][b] in[oy*S - pad + a][ox*S - pad + b]
// MODE 0: forward (in = x, whose planes n*C + c are contiguous; out = y slice)
// MODE 1: stride-1 grad-input (in = grad_out slice, w' = rot180(w), out = gx)
template <typename T, int K, int S, int MODE>
__global__ void __launch_bounds__(kThreads)
conv_kernel(Conv c, PCfg g, const T* __restrict__ in, const T* __restrict__ w, const T* __restrict__ bias,
            T* __restrict__ out, int accumulate) {
  extern __shared__ __align__(16) float psm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* const buf0 = psm + warp * 2 * g.P * g.TS;
  float* const buf1 = buf0 + g.P * g.TS;
  for (int i = lane; i < 2 * g.P * g.TS; i += 32) buf0[i] = 0.f;  // the halo stays zero
  __syncwarp();
  const int pl = lane / g.L, ox = lane - pl * g.L;
  int lr, lc, rstep;
  load_rows_setup(g, lane, lr, lc, rstep);
  const int64_t hw_in = (int64_t)g.Hin * g.Win, hw_out = (int64_t)g.Hout * g.Wout;
  auto issue = [&](int64_t grp, float* tile) {
    const int64_t p0 = grp * g.P;
    for (int q = 0; q < g.P; ++q) {
      const int64_t pin = p0 + q;
      if (pin >= g.nplanes) break;
      const T* src;
      if (MODE == 0) {
        src = in + pin * hw_in;
      } else {
        int64_t n, ch;
        c.split(pin, n, ch);
        src = in + c.y_base(n, ch);
      }
      load_plane<T>(tile + q * g.TS, src, g, g.pad, lr, lc, rstep);
    }
  };
  auto compute = [&](int64_t grp, const float* tile) {
    const int64_t pin = grp * g.P + pl;
    if (ox >= g.Wout || pin >= g.nplanes) return;
    int64_t n, ch;
    c.split(pin, n, ch);
    float wr[K * K];
#pragma unroll
    for (int i = 0; i < K * K; ++i) wr[i] = ld(w + ch * (K * K) + (MODE == 1 ? K * K - 1 - i : i));
    const float bv = (MODE == 0 && bias) ? ld(bias + ch) : 0.f;
    T* dst = MODE == 0 ? out + c.y_base(n, ch) : out + pin * hw_out;
    const float* tp = tile + pl * g.TS + ox * S;
    // window rows oy*S + a; a step of one output row drops the first S rows
    float win[K][K];
#pragma unroll
    for (int a = 0; a < K - S; ++a)
#pragma unroll
      for (int b = 0; b < K; ++b) win[a + S][b] = tp[a * g.TP + b];
    for (int oy = 0; oy < g.Hout; ++oy) {
#pragma unroll
      for (int a = 0; a < K - S; ++a)
#pragma unroll
        for (int b = 0; b < K; ++b) win[a][b] = win[a + S][b];
      const float* rowp = tp + oy * S * g.TP;
#pragma unroll
      for (int a = K - S; a < K; ++a)
#pragma unroll
        for (int b = 0; b < K; ++b) win[a][b] = rowp[a * g.TP + b];
      float acc = bv;
#pragma unroll
      for (int a = 0; a < K; ++a)
#pragma unroll
        for (int b = 0; b < K; ++b) acc = fmaf(wr[a * K + b], win[a][b], acc);
      T* o = dst + oy * g.Wout + ox;
      *o = from_f<T>(accumulate ? acc + ld_rw(o) : acc);
    }
  };
  warp_walk((int64_t)blockIdx.x * kWarps + warp, (int64_t)gridDim.x * kWarps, g.groups, buf0, buf1, issue,
            compute);
}

// Weight-gradient first pass: for unit (chunk, channel c),
// partial[chunk, c, a*K + b] = sum over the chunk's samples of sum_{oy,ox} gy*x̃,
// partial[chunk, c, K*K] = sum of gy. Warp w takes sample groups w, w + 8, ...
// of the chunk (P samples per group, one per lane group); lanes keep K*K + 1
// sums, reduced at the end by a butterfly and then over warps in order.
template <typename T, int K, int S>
__global__ void __launch_bounds__(kThreads)
wgrad_kernel(Conv c, PCfg g, const T* __restrict__ x, const T* __restrict__ gy, float* __restrict__ ws,
             int chunks) {
  extern __shared__ __align__(16) float psm[];
  constexpr int NV = K * K + 1;
  __shared__ float red[kWarps][NV];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* const buf0 = psm + warp * 2 * g.P * g.TS;
  float* const buf1 = buf0 + g.P * g.TS;
  for (int i = lane; i < 2 * g.P * g.TS; i += 32) buf0[i] = 0.f;
  __syncwarp();
  const int pl = lane / g.L, ox = lane - pl * g.L;
  int lr, lc, rstep;
  load_rows_setup(g, lane, lr, lc, rstep);
  const int64_t units = c.C * chunks;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    uint32_t cq;
    const int64_t ch = c.dC.divmod((uint32_t)u, cq);
    const int64_t n0 = (int64_t)cq * g.nb;
    int64_t n1 = n0 + g.nb;
    if (n1 > c.N) n1 = c.N;
    float acc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] = 0.f;
    auto issue = [&](int64_t s0, float* tile) {
      for (int q = 0; q < g.P; ++q) {
        if (s0 + q >= n1) break;
        load_plane<T>(tile + q * g.TS, x + c.x_base(s0 + q, ch), g, g.pad, lr, lc, rstep);
      }
    };
    auto compute = [&](int64_t s0, const float* tile) {
      const int64_t n = s0 + pl;
      if (ox >= g.Wout || n >= n1) return;
      const T* gp = gy + c.y_base(n, ch) + ox;
      const float* tp = tile + pl * g.TS + ox * S;
      float win[K][K];
#pragma unroll
      for (int a = 0; a < K - S; ++a)
#pragma unroll
        for (int b = 0; b < K; ++b) win[a + S][b] = tp[a * g.TP + b];
      for (int oy = 0; oy < g.Hout; ++oy) {
#pragma unroll
        for (int a = 0; a < K - S; ++a)
#pragma unroll
          for (int b = 0; b < K; ++b) win[a][b] = win[a + S][b];
        const float* rowp = tp + oy * S * g.TP;
#pragma unroll
        for (int a = K - S; a < K; ++a)
#pragma unroll
          for (int b = 0; b < K; ++b) win[a][b] = rowp[a * g.TP + b];
        const float gv = ld(gp + oy * g.Wout);
#pragma unroll
        for (int a = 0; a < K; ++a)
#pragma unroll
          for (int b = 0; b < K; ++b) acc[a * K + b] = fmaf(gv, win[a][b], acc[a * K + b]);
        acc[K * K] += gv;
      }
    };
    warp_walk(n0 + (int64_t)warp * g.P, (int64_t)kWarps * g.P, n1, buf0, buf1, issue, compute);
    // butterfly within the warp, then the warps in order
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      float v = acc[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[warp][i] = v;
    }
    __syncthreads();
    if (threadIdx.x < NV) {
      float sum = 0.f;
#pragma unroll
      for (int wi = 0; wi < kWarps; ++wi) sum += red[wi][threadIdx.x];
      ws[((int64_t)cq * c.OC() + ch) * NV + threadIdx.x] = sum;
    }
    __syncthreads();
  }
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

size_t smem_of(const PCfg& g) { return (size_t)kWarps * 2 * g.P * g.TS * sizeof(float); }

int grid_of(const void* kern, size_t smem, int64_t work) {
  int dev = 0, sms = 152, per = 1;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, kThreads, smem) != cudaSuccess || per < 1) per = 1;
  const int64_t cap = (int64_t)sms * per;
  return (int)(work < cap ? (work > 0 ? work : 1) : cap);
}

// Correlation geometry for MODE 0 / 1.
PCfg conv_cfg(const Conv& c, bool grad) {
  PCfg g{};
  g.Hin = grad ? (int)c.Ho : (int)c.H;
  g.Win = grad ? (int)c.Wo : (int)c.W;
  g.Hout = grad ? (int)c.H : (int)c.Ho;
  g.Wout = grad ? (int)c.W : (int)c.Wo;
  g.pad = grad ? c.kh - 1 - c.ph : c.ph;
  const int S = grad ? 1 : c.sh;
  g.L = pow2_at_least(g.Wout);
  g.P = 32 / g.L;
  g.Lw = pow2_at_least(g.Win);
  g.TR = (g.Hout - 1) * S + c.kh;
  g.TP = (g.Wout - 1) * S + c.kw;
  g.TS = g.TR * g.TP;
  g.nplanes = c.N * c.C;
  g.groups = (g.nplanes + g.P - 1) / g.P;
  return g;
}

template <typename T, int S>
cudaError_t fwd_t(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s) {
  const PCfg g = conv_cfg(c, false);
  auto kern = conv_kernel<T, 3, S, 0>;
  const size_t smem = smem_of(g);
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_of((const void*)kern, smem, (g.groups + kWarps - 1) / kWarps);
  kern<<<grid, kThreads, smem, s>>>(c, g, (const T*)x, (const T*)w, (const T*)b, (T*)y, 0);
  return cudaGetLastError();
}

template <typename T>
cudaError_t bwd1_t(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
  const PCfg g = conv_cfg(c, true);
  auto kern = conv_kernel<T, 3, 1, 1>;
  const size_t smem = smem_of(g);
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_of((const void*)kern, smem, (g.groups + kWarps - 1) / kWarps);
  kern<<<grid, kThreads, smem, s>>>(c, g, (const T*)gy, (const T*)w, nullptr, (T*)gx, acc ? 1 : 0);
  return cudaGetLastError();
}

template <typename T, int S>
cudaError_t wgrad_t(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
  PCfg g = conv_cfg(c, false);
  g.nb = (int)wgrad_nb(c);
  if (c.N > 0 && (c.N + g.nb - 1) / g.nb != chunks) return cudaErrorInvalidConfiguration;
  auto kern = wgrad_kernel<T, 3, S>;
  const size_t smem = smem_of(g);
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  const int grid = grid_of((const void*)kern, smem, c.C * chunks);
  kern<<<grid, kThreads, smem, s>>>(c, g, (const T*)x, (const T*)gy, ws, chunks);
  return cudaGetLastError();
}

}  // namespace

bool fwd_supported(const Conv& c) { return shape_ok(c) && c.W > 8 && c.W <= 16; }
bool bwd_data_supported(const Conv& c) { return shape_ok(c) && c.sh == 1 && c.W > 8 && c.W <= 16; }
bool wgrad_supported(const Conv& c) { return shape_ok(c) && c.Wo <= 16; }

int64_t wgrad_nb(const Conv& c) {
  // a chunk is a whole number of sample groups for every warp of a CTA
  // (P samples per warp group), with at least about four units per SM
  const int P = 32 / pow2_at_least((int)c.Wo);
  int64_t nb = (int64_t)P * kWarps;
  const int64_t units_min = 152 * 4;
  while (nb > P && c.C * ((c.N + nb - 1) / nb) < units_min) nb -= P;
  if (nb > c.N) nb = c.N > 0 ? c.N : 1;
  return nb;
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
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = bwd1_t<T>(c, gy, w, gx, acc, s));
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
