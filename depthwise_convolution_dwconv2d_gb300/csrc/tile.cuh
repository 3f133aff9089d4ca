// Shared-memory tile machinery for the small-kernel depthwise kernels.
//
// A CTA stages a band of input rows (with the halo the kernel needs, zero
// outside the plane) of one or more channel planes into shared memory as
// fp32, then every thread computes an R x V block of outputs from it with the
// filter held in registers and a sliding window of the tile row in registers
// (the multi-level blocking of the MegEngine large-kernel depthwise article,
// section "DirectConv": CTA tile -> rows -> a small block of outputs per
// thread).
//
// Output block of a thread: rows oh_b + r*Q, cols ow_b + v*Q (r < R, v < V)
// with Q = D / S when the dilation is a multiple of the stride, else Q = 1.
// With that spacing the taps of neighbouring outputs land on the same input
// samples, so every tile value a thread loads feeds several outputs even for
// dilated filters.
#pragma once

#include "common.cuh"

namespace dwconv {
namespace tile {

constexpr int kNT = 256;  // threads per CTA for every tile kernel

template <int K, int S, int D>
struct Geo {
  static constexpr int Q = (D % S == 0) ? D / S : 1;
  static constexpr int QS = Q * S;
};

// Host/device description of one CTA's tile (computed on the host).
struct TileCfg {
  int ppc;       // channel planes per CTA
  int th;        // output rows per band
  int nbands;    // bands per plane
  int tr, pitch; // tile rows and row pitch (floats); pitch % 4 == 0
  int rb, cb;    // row / col blocks of the item grid
  int ntile;     // staged planes per output plane (1, or m for bwd_data)
  int tile_floats;  // floats per staged plane (tr * pitch)
  int vec_in;    // 16-byte global loads allowed
  int vec_out;   // V-wide vector stores allowed
  int64_t groups;   // plane groups (grid = groups * nbands)
};

// ---- tile loading ------------------------------------------------------------
template <typename T> struct Vec16;
template <> struct Vec16<float> { static constexpr int n = 4; };
template <> struct Vec16<__half> { static constexpr int n = 8; };
template <> struct Vec16<__nv_bfloat16> { static constexpr int n = 8; };

template <typename T>
__device__ __forceinline__ void cvt16(const uint4& u, float* out);
template <>
__device__ __forceinline__ void cvt16<float>(const uint4& u, float* out) {
  out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
  out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void cvt16<__half>(const uint4& u, float* out) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __half22float2(h[i]);
    out[2 * i] = f.x; out[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void cvt16<__nv_bfloat16>(const uint4& u, float* out) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Stage `np` planes into smem. Plane i comes from src_of(i) (H x W elements,
// row-major) and lands at dst + i * tile_floats as rows [iy0, iy0 + tr) x
// cols [ix0, ix0 + cols) with row pitch `pitch`; samples outside the plane
// are zero. vec: every row start is 16-byte aligned in global memory.
template <typename T, typename SrcOf>
__device__ __forceinline__ void load_planes(float* __restrict__ dst, int np, int tile_floats,
                                            int pitch, SrcOf src_of, int H, int W, int iy0,
                                            int tr, int ix0, int cols, bool vec) {
  // rows of the tile that hold plane rows
  const int r_lo = iy0 < 0 ? -iy0 : 0;
  const int r_hi = (H - iy0) < tr ? (H - iy0) : tr;
  const int nrow_in = r_hi > r_lo ? r_hi - r_lo : 0;
  // columns of the tile that hold plane columns: [c_lo, c_hi)
  const int c_lo = ix0 < 0 ? (-ix0 < cols ? -ix0 : cols) : 0;
  const int c_hi0 = (W - ix0) < cols ? (W - ix0) : cols;
  const int c_hi = c_hi0 > c_lo ? c_hi0 : c_lo;
  // 1) zero the halo: whole rows outside the plane, and the side columns
  {
    const int hl = c_lo, hr = cols - c_hi;  // left / right halo widths
    const int side = hl + hr;
    const int nrow_out = tr - nrow_in;
    const int per_plane = nrow_out * cols + nrow_in * side;
    for (int e = threadIdx.x; e < np * per_plane; e += blockDim.x) {
      const int p = e / per_plane;
      int q = e - p * per_plane;
      int row, col;
      if (q < nrow_out * cols) {
        const int rr = q / cols;
        col = q - rr * cols;
        row = rr < r_lo ? rr : rr + nrow_in;
      } else {
        q -= nrow_out * cols;
        const int rr = q / side;
        const int k = q - rr * side;
        row = r_lo + rr;
        col = k < hl ? k : c_hi + (k - hl);
      }
      dst[p * tile_floats + row * pitch + col] = 0.f;
    }
  }
  if (nrow_in == 0 || c_hi <= c_lo) return;
  // 2) copy plane samples in tile columns [c_lo, c_hi), i.e. plane columns
  //    [c_lo + ix0, c_hi + ix0)
  constexpr int VN = Vec16<T>::n;
  if (vec && W % VN == 0 && ix0 <= 0 && W - ix0 <= cols) {
    const int cpr = W / VN;  // chunks per row
    const int total = np * nrow_in * cpr;
    for (int e = threadIdx.x; e < total; e += blockDim.x) {
      const int p = e / (nrow_in * cpr);
      const int q = e - p * (nrow_in * cpr);
      const int rr = q / cpr;
      const int ch = q - rr * cpr;
      const int row = r_lo + rr;
      const T* s = src_of(p) + (int64_t)(iy0 + row) * W + ch * VN;
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(s));
      float f[VN];
      cvt16<T>(u, f);
      float* d = dst + p * tile_floats + row * pitch + (ch * VN - ix0);
#pragma unroll
      for (int i = 0; i < VN; ++i) d[i] = f[i];
    }
  } else {
    const int nc = c_hi - c_lo;
    const int total = np * nrow_in * nc;
    for (int e = threadIdx.x; e < total; e += blockDim.x) {
      const int p = e / (nrow_in * nc);
      const int q = e - p * (nrow_in * nc);
      const int rr = q / nc;
      const int tc = c_lo + (q - rr * nc);
      const int row = r_lo + rr;
      dst[p * tile_floats + row * pitch + tc] = ld(src_of(p) + (int64_t)(iy0 + row) * W + (tc + ix0));
    }
  }
}

// ---- the register-blocked stencil ------------------------------------------
template <int K, int D, int R, int QS>
__device__ constexpr bool row_used(int u) {
  for (int r = 0; r < R; ++r)
    for (int a = 0; a < K; ++a)
      if (r * QS + a * D == u) return true;
  return false;
}

template <int K, int D, int V, int QS>
__device__ constexpr bool col_used(int i) {
  for (int v = 0; v < V; ++v)
    for (int b = 0; b < K; ++b)
      if (v * QS + b * D == i) return true;
  return false;
}

// acc[r][v] += sum_{a,b} wr[a*K+b] * t[(tr0 + r*Q*S + a*D) * pitch + tc0 + v*Q*S + b*D]
// With Q == 1 the window of a tile row is contiguous and is read with float4
// loads, so tc0 must then be a multiple of 4.
template <int K, int S, int D, int R, int V, int Q>
__device__ __forceinline__ void conv_block(const float* __restrict__ t, int pitch, int tr0, int tc0,
                                           const float (&wr)[K * K], float (&acc)[R][V]) {
  constexpr int QS = Q * S;
  constexpr bool VEC = Q == 1;
  constexpr int U = (R - 1) * QS + (K - 1) * D + 1;
  constexpr int WN = (V - 1) * QS + (K - 1) * D + 1;
  constexpr int WN4 = (WN + 3) / 4 * 4;
  constexpr int WA = VEC ? WN4 : WN;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (!row_used<K, D, R, QS>(u)) continue;
    const float* rowp = t + (tr0 + u) * pitch + tc0;
    float win[WA];
    if (VEC) {
#pragma unroll
      for (int i = 0; i < WN4 / 4; ++i) {
        const float4 f = *reinterpret_cast<const float4*>(rowp + 4 * i);
        win[4 * i] = f.x; win[4 * i + 1] = f.y; win[4 * i + 2] = f.z; win[4 * i + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < WA; ++i) win[i] = col_used<K, D, V, QS>(i) ? rowp[i] : 0.f;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int a = 0; a < K; ++a) {
        if (r * QS + a * D != u) continue;
#pragma unroll
        for (int b = 0; b < K; ++b) {
#pragma unroll
          for (int v = 0; v < V; ++v) acc[r][v] = fmaf(wr[a * K + b], win[v * QS + b * D], acc[r][v]);
        }
      }
    }
  }
}

// ---- output stores ---------------------------------------------------------
template <typename T, int V>
__device__ __forceinline__ void store_vec(T* p, const float (&v)[V]);
template <>
__device__ __forceinline__ void store_vec<float, 4>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store_vec<__half, 4>(__half* p, const float (&v)[4]) {
  __half2 a = __floats2half2_rn(v[0], v[1]), b = __floats2half2_rn(v[2], v[3]);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}
template <>
__device__ __forceinline__ void store_vec<__nv_bfloat16, 4>(__nv_bfloat16* p, const float (&v)[4]) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// Store an R x V block at rows oh + r*Q (r-th valid while < rows_left),
// cols ow + v*Q (< Wo). add: read-modify-write (gx += ...).
template <typename T, int R, int V, int Q>
__device__ __forceinline__ void store_block(T* __restrict__ plane, int64_t Wo, int oh, int ow,
                                            int rows_left, int cols, float (&acc)[R][V], bool vec,
                                            bool add) {
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r * Q >= rows_left) break;
    T* rowp = plane + (int64_t)(oh + r * Q) * Wo;
    if (Q == 1 && V == 4 && vec && ow + V <= cols) {
      float o[V];
#pragma unroll
      for (int v = 0; v < V; ++v) o[v] = add ? acc[r][v] + ld_rw(rowp + ow + v) : acc[r][v];
      store_vec<T, 4>(rowp + ow, reinterpret_cast<const float(&)[4]>(o));
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int c = ow + v * Q;
        if (c < cols) rowp[c] = from_f<T>(add ? acc[r][v] + ld_rw(rowp + c) : acc[r][v]);
      }
    }
  }
}

}  // namespace tile
}  // namespace dwconv

namespace dwconv {
namespace tile {

// Geometry of the stencil a tile kernel evaluates, written as a forward
// convolution: out[oy][ox] = sum_{a,b} w'[a][b] * in[oy*S - ph + a*D][ox*S - pw + b*D]
// (for bwd_data at stride 1, `in` is grad_out, w' the flipped filter and
// ph = D*(K-1) - pad).
struct VGeo {
  int K, S, D, Q, R, V;
  int64_t Hin, Win, Hout, Wout;
  int ph, pw;
};

inline int round4(int64_t v) { return (int)((v + 3) / 4 * 4); }

// Widest tile column any thread reads (+1), for a row of cb column blocks.
inline int64_t cols_read(const VGeo& g, int cb) {
  const int QS = g.Q * g.S;
  const int WN = (g.V - 1) * QS + (g.K - 1) * g.D + 1;
  if (g.Q == 1) return (int64_t)(cb - 1) * g.V * g.S + (WN + 3) / 4 * 4;
  const int64_t owb = (int64_t)(cb - 1) * g.Q * g.V + g.Q - 1;
  return owb * g.S + (g.V - 1) * QS + (g.K - 1) * g.D + 1;
}

// Choose band height, planes per CTA and the smem layout. Returns false when
// no band of the minimum height fits the shared-memory limit.
inline bool make_cfg(const VGeo& g, int64_t nplanes, int ntile, int mult, bool vec_in,
                     bool vec_out, TileCfg* out, int64_t ix_extra_left = 0) {
  const int QR = g.Q * g.R;
  TileCfg c{};
  c.cb = (int)((g.Wout + (int64_t)g.Q * g.V - 1) / ((int64_t)g.Q * g.V));
  const int64_t need = cols_read(g, c.cb) > g.Win + g.pw + ix_extra_left
                           ? cols_read(g, c.cb) : g.Win + g.pw + ix_extra_left;
  c.pitch = round4(need);
  auto tr_of = [&](int64_t th) { return (th - 1) * g.S + (int64_t)(g.K - 1) * g.D + 1; };
  const int64_t per_cta = 96 * 1024;  // smem budget per CTA (bytes), two CTAs per SM at least
  const int64_t th_full = (g.Hout + QR - 1) / QR * QR;
  int64_t th = th_full;
  auto bytes_of = [&](int64_t t) { return tr_of(t) * c.pitch * 4 * ntile; };
  const int64_t target = 40 * 1024;
  if (bytes_of(th) > target) {
    th = (target / (c.pitch * 4 * ntile) - (int64_t)(g.K - 1) * g.D - 1) / g.S + 1;
    th = th / QR * QR;
    if (th < QR) th = QR;
    if (bytes_of(th) > per_cta) return false;
  }
  c.th = (int)th;
  c.rb = (int)(th / QR);
  c.nbands = (int)((g.Hout + th - 1) / th);
  c.tr = (int)tr_of(th);
  c.ntile = ntile;
  c.tile_floats = c.tr * c.pitch;
  const int64_t items = (int64_t)mult * c.rb * c.cb * g.Q * g.Q;
  int64_t ppc = 1;
  if (c.nbands == 1) {
    ppc = (2 * kNT + items - 1) / items;
    const int64_t cap = target / bytes_of(th);
    if (ppc > cap) ppc = cap;
    // keep at least ~4 CTAs per SM worth of groups
    const int64_t min_groups = 152 * 4;
    if ((nplanes + ppc - 1) / ppc < min_groups) ppc = (nplanes + min_groups - 1) / min_groups;
    if (ppc < 1) ppc = 1;
  }
  c.ppc = (int)ppc;
  c.groups = (nplanes + ppc - 1) / ppc;
  c.vec_in = vec_in;
  c.vec_out = vec_out;
  *out = c;
  return true;
}

inline size_t smem_bytes(const TileCfg& c) {
  return (size_t)c.ppc * c.ntile * c.tile_floats * sizeof(float);
}

}  // namespace tile
}  // namespace dwconv
