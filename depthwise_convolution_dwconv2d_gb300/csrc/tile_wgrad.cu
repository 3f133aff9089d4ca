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
#include "plan.h"
#include "tile.cuh"

namespace dwconv {
namespace tile {
namespace {

struct WCfg {
  int nb;          // batch samples per chunk
  int chunks;
  int th, nbands;  // output rows per band, bands per plane
  int tr, pitch;   // x tile rows / pitch
  int gpitch;      // grad_out tile pitch (th rows)
  int rb, cb;
  int ppc;         // slices (sample, band) staged at once
  int x_floats, g_floats;  // per slice
  int vec_x, vec_g;
};

template <typename T, int K, int S, int D, int M, int R, int V>
__global__ void __launch_bounds__(kNT)
wgrad_kernel(Conv c, WCfg g, const T* __restrict__ x, const T* __restrict__ gy,
             float* __restrict__ ws) {
  extern __shared__ __align__(16) float sm[];
  constexpr int KK = K * K;
  constexpr int NV = M * (KK + 1);
  constexpr int U = (R - 1) * S + (K - 1) * D + 1;
  constexpr int WN = (V - 1) * S + (K - 1) * D + 1;
  constexpr int WN4 = (WN + 3) / 4 * 4;
  const int64_t ch = blockIdx.x % c.C;
  const int chunk = blockIdx.x / c.C;
  const int64_t n0 = (int64_t)chunk * g.nb;
  const int nsl = (int)(((c.N - n0) < g.nb ? (c.N - n0) : g.nb) * g.nbands);  // slices in chunk
  float* xs = sm;
  float* gs = sm + g.ppc * g.x_floats;
  float* red = gs + g.ppc * M * g.g_floats;  // [warps][NV]
  float acc[M][KK + 1];
#pragma unroll
  for (int j = 0; j < M; ++j)
#pragma unroll
    for (int i = 0; i <= KK; ++i) acc[j][i] = 0.f;

  for (int s0 = 0; s0 < nsl; s0 += g.ppc) {
    const int ns = (nsl - s0) < g.ppc ? (nsl - s0) : g.ppc;
    if (s0 > 0) __syncthreads();
    // x tiles: slice q -> sample n0 + (s0+q)/nbands, band (s0+q)%nbands
    for (int q = 0; q < ns; ++q) {
      const int sl = s0 + q;
      const int64_t n = n0 + sl / g.nbands;
      const int band = sl % g.nbands;
      const int oh0 = band * g.th;
      load_planes<T>(xs + q * g.x_floats, 1, g.x_floats, g.pitch,
                     [&](int) { return x + c.x_base(n, ch); }, (int)c.H, (int)c.W,
                     oh0 * S - c.ph, g.tr, -c.pw, g.pitch, g.vec_x);
      load_planes<T>(gs + q * M * g.g_floats, M, g.g_floats, g.gpitch,
                     [&](int j) { return gy + c.y_base(n, ch * M + j); }, (int)c.Ho, (int)c.Wo,
                     oh0, g.th, 0, g.gpitch, g.vec_g);
    }
    __syncthreads();
    const int per = g.rb * g.cb;
    for (int it = threadIdx.x; it < ns * per; it += kNT) {
      const int q = it / per;
      const int rem = it - q * per;
      const int rbi = rem / g.cb;
      const int cbi = rem - rbi * g.cb;
      float gv[M][R][V];
#pragma unroll
      for (int j = 0; j < M; ++j)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 f = *reinterpret_cast<const float4*>(
              gs + (q * M + j) * g.g_floats + (rbi * R + r) * g.gpitch + cbi * V);
          gv[j][r][0] = f.x; gv[j][r][1] = f.y; gv[j][r][2] = f.z; gv[j][r][3] = f.w;
          acc[j][KK] += (f.x + f.y) + (f.z + f.w);
        }
      const float* t = xs + q * g.x_floats + (rbi * R * S) * g.pitch + cbi * V * S;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (!row_used<K, D, R, S>(u)) continue;
        float win[WN4];
#pragma unroll
        for (int i = 0; i < WN4 / 4; ++i) {
          const float4 f = *reinterpret_cast<const float4*>(t + u * g.pitch + 4 * i);
          win[4 * i] = f.x; win[4 * i + 1] = f.y; win[4 * i + 2] = f.z; win[4 * i + 3] = f.w;
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int a = 0; a < K; ++a) {
            if (r * S + a * D != u) continue;
#pragma unroll
            for (int j = 0; j < M; ++j)
#pragma unroll
              for (int b = 0; b < K; ++b)
#pragma unroll
                for (int v = 0; v < V; ++v)
                  acc[j][a * K + b] = fmaf(gv[j][r][v], win[v * S + b * D], acc[j][a * K + b]);
          }
      }
    }
  }
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
    }
  __syncthreads();
  for (int i = threadIdx.x; i < NV; i += kNT) {
    float s = 0.f;
    for (int wi = 0; wi < kNT / 32; ++wi) s += red[wi * NV + i];
    const int j = i / (KK + 1), tap = i - j * (KK + 1);
    const int64_t oc = ch * M + j;
    ws[((int64_t)chunk * c.OC() + oc) * (KK + 1) + tap] = s;
  }
}

template <int K, int S> struct WBlk { static constexpr int R = S == 1 ? 2 : 1, V = 4; };

template <typename T, int K, int S, int D, int M>
cudaError_t run_wgrad_t(const Conv& c, const void* x, const void* gy, float* ws, int chunks,
                        cudaStream_t s) {
  constexpr int R = WBlk<K, S>::R, V = WBlk<K, S>::V;
  const int es = c.dtype == DWCONV_F32 ? 4 : 2;
  WCfg g{};
  g.chunks = chunks;
  g.nb = (int)((c.N + chunks - 1) / chunks);
  g.cb = (int)((c.Wo + V - 1) / V);
  g.gpitch = round4((int64_t)g.cb * V);
  const int WN4 = (((V - 1) * S + (K - 1) * D + 1) + 3) / 4 * 4;
  const int64_t need = (int64_t)(g.cb - 1) * V * S + WN4;
  g.pitch = round4(need > c.W + c.pw ? need : c.W + c.pw);
  auto tr_of = [&](int64_t th) { return (th - 1) * S + (int64_t)(K - 1) * D + 1; };
  auto bytes_of = [&](int64_t th) { return (tr_of(th) * g.pitch + M * th * g.gpitch) * 4; };
  const int64_t target = 40 * 1024;
  int64_t th = (c.Ho + R - 1) / R * R;
  if (bytes_of(th) > target) {
    th = R;
    while (bytes_of(th + R) <= target) th += R;
    if (bytes_of(th) > 96 * 1024) return cudaErrorInvalidConfiguration;
  }
  g.th = (int)th;
  g.rb = (int)(th / R);
  g.nbands = (int)((c.Ho + th - 1) / th);
  g.tr = (int)tr_of(th);
  g.x_floats = g.tr * g.pitch;
  g.g_floats = (int)(th * g.gpitch);
  const int64_t items = (int64_t)g.rb * g.cb;
  int64_t ppc = (2 * kNT + items - 1) / items;
  const int64_t cap = target / bytes_of(th);
  if (ppc > cap) ppc = cap;
  const int64_t slices = (int64_t)g.nb * g.nbands;
  if (ppc > slices) ppc = slices;
  if (ppc < 1) ppc = 1;
  g.ppc = (int)ppc;
  g.vec_x = ((reinterpret_cast<uintptr_t>(x) & 15) == 0) && (c.W * es) % 16 == 0;
  g.vec_g = ((reinterpret_cast<uintptr_t>(gy) & 15) == 0) && (c.Wo * es) % 16 == 0;
  const size_t smem = ((size_t)g.ppc * (g.x_floats + M * g.g_floats) + (kNT / 32) * M * (K * K + 1)) * 4;
  auto kern = wgrad_kernel<T, K, S, D, M, R, V>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)(c.C * chunks), kNT, smem, s>>>(c, g, (const T*)x, (const T*)gy, ws);
  return cudaGetLastError();
}

#define DW_WGRAD_CASES(X) X(3, 1, 1, 1) X(3, 2, 1, 1) X(5, 1, 1, 1) X(5, 2, 1, 1) X(3, 1, 1, 2) \
  X(5, 1, 1, 2) X(3, 2, 1, 2) X(7, 1, 1, 1) X(3, 1, 2, 1) X(3, 1, 3, 1) X(3, 1, 5, 1)

template <typename T>
cudaError_t wgrad_t(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
#define X(K, S, D, M) \
  if (c.kh == K && c.sh == S && c.dh == D && c.m == M) return run_wgrad_t<T, K, S, D, M>(c, x, gy, ws, chunks, s);
  DW_WGRAD_CASES(X)
#undef X
  return cudaErrorInvalidConfiguration;
}

}  // namespace

bool wgrad_supported(const Conv& c) {
  if (c.kh != c.kw || c.sh != c.sw || c.dh != c.dw || c.W > 1024 || c.Wo > 1024) return false;
#define X(K, S, D, M) if (c.kh == K && c.sh == S && c.dh == D && c.m == M) return true;
  DW_WGRAD_CASES(X)
#undef X
  return false;
}

int wgrad_chunks(const Conv& c) {
  // about eight CTAs per SM over channels x chunks, each thread's serial
  // chain (samples x positions / threads) far below 4096 terms
  int64_t chunks = (152 * 8 + c.C - 1) / c.C;
  if (chunks > c.N) chunks = c.N;
  if (chunks < 1) chunks = 1;
  int64_t nb = (c.N + chunks - 1) / chunks;
  const int64_t cap = ((int64_t)1 << 20) / (c.Ho * c.Wo > 0 ? c.Ho * c.Wo : 1);
  if (nb > cap) nb = cap > 0 ? cap : 1;
  chunks = c.N > 0 ? (c.N + nb - 1) / nb : 1;
  if (chunks > 65535) chunks = 65535;
  return (int)chunks;
}

cudaError_t wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidConfiguration;
  DWCONV_DISPATCH_DTYPE(c.dtype, T, e = wgrad_t<T>(c, x, gy, ws, chunks, s));
  return e;
}

}  // namespace tile
}  // namespace dwconv
