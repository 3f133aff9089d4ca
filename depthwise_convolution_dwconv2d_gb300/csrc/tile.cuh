// Shared-memory tile machinery for the small-kernel depthwise kernels.
//
// A CTA stages a band of input rows (with the halo the filter needs, zero
// outside the plane) of one or more channel planes into shared memory in the
// storage type, then every thread computes an R x V block of outputs from it
// with the filter in registers and a sliding window of each tile row in
// registers (the multi-level blocking of the MegEngine large-kernel depthwise
// article, section "DirectConv": CTA tile -> rows -> a block of outputs per
// thread).
//
// Staging uses cp.async (asynchronous global->shared copies): 16-byte chunks
// when every row start and the tile origin are 16-byte aligned, 4-byte chunks
// otherwise, with zero fill through the copy's source size for chunks outside
// the plane. The tile kernels are persistent and run two stages: the copies
// for a CTA's next tile are in flight while it computes the current one, so
// HBM traffic does not stop at tile boundaries.
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

// Copy mode of a tile: 16-byte chunks, 4-byte chunks, or plain loads and
// stores (2-byte types with odd alignment).
enum CopyMode { kCopySync = 0, kCopy4 = 1, kCopy16 = 2, kCopyTMA = 3, kCopyDense = 4 };

// ---- cp.async ------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem, int src_bytes) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes)
               : "memory");
}
// One entry of a stage's side table (filter taps, bias): fp32 by an
// asynchronous 4-byte copy that completes with the stage's cp.async group
// (so no thread waits on a global load while the previous stage computes),
// 16-bit types widened through a register.
template <typename T>
__device__ __forceinline__ void tab_put(float* dst, const T* src) {
  if (sizeof(T) == 4) cp_async4(dst, src, 4);
  else *dst = ld(src);
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Issue the copies that stage `np` planes into smem (no wait). Plane i comes
// from src_of(i) (H x W elements, row-major) and lands at dst + i*plane_elems
// as rows [iy0, iy0 + tr) x cols [ix0, ix0 + pitch); samples outside the
// plane are zero. Copy modes 16 / 4 need ix0 and W to be multiples of the
// chunk (in elements) and 16- / 4-byte aligned plane bases; pitch is a
// multiple of 16 bytes. Rows are spread over warps, the lanes of a row sweep
// its chunks; narrow rows share a warp.
template <typename T, typename SrcOf>
__device__ __forceinline__ void issue_tile(T* __restrict__ dst, int np, int plane_elems, int pitch,
                                           SrcOf src_of, int H, int W, int iy0, int tr,
                                           const FastDiv& trdiv, int ix0, int mode) {
  constexpr int ES = sizeof(T);
  const int ce = mode == kCopy16 ? 16 / ES : mode == kCopy4 ? 4 / ES : 1;  // elements per chunk
  const int nch = pitch / ce;
  const int lpr = nch > 16 ? 32 : nch > 8 ? 16 : nch > 4 ? 8 : 4;  // lanes per row
  const int rpw = 32 / lpr;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane / lpr, l = lane & (lpr - 1);
  const int nwarps = blockDim.x >> 5;
  const int rows = np * tr;
  for (int q = warp * rpw + sub; q < rows; q += nwarps * rpw) {
    uint32_t p;
    const int r = (int)trdiv.divmod((uint32_t)q, p);
    const int iy = iy0 + r;
    const bool rin = iy >= 0 && iy < H;
    T* drow = dst + (int)p * plane_elems + r * pitch;
    const T* plane = src_of((int)p);
    const T* srow = plane + (int64_t)(rin ? iy : 0) * W;
    if (mode == kCopy16) {
      for (int c = l; c < nch; c += lpr) {
        const int ix = ix0 + c * ce;
        const bool in = rin && ix >= 0 && ix + ce <= W;
        cp_async16(drow + c * ce, in ? srow + ix : plane, in ? 16 : 0);
      }
    } else if (mode == kCopy4) {
      for (int c = l; c < nch; c += lpr) {
        const int ix = ix0 + c * ce;
        const bool in = rin && ix >= 0 && ix + ce <= W;
        cp_async4(drow + c * ce, in ? srow + ix : plane, in ? 4 : 0);
      }
    } else {
      for (int c = l; c < pitch; c += lpr) {
        const int ix = ix0 + c;
        drow[c] = (rin && ix >= 0 && ix < W) ? srow[ix] : from_f<T>(0.f);
      }
    }
  }
}

// Dense staging for planes whose rows are not 16-byte multiples (small
// planes): each plane's H*W contiguous elements are copied with 16-byte
// cp.async chunks into a staging segment of `seg` elements, starting at the
// plane's own offset within its 16-byte chunk (its address mod 16); the last
// chunk is cut at the plane's end by the copy's source size, so nothing
// outside the plane's 16-byte neighbourhood is read.
template <typename T, typename SrcOf>
__device__ __forceinline__ void issue_flat(T* __restrict__ stg, int np, int seg, SrcOf src_of, int HW) {
  constexpr int ES = sizeof(T);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  for (int p = warp; p < np; p += nwarps) {
    const char* a = reinterpret_cast<const char*>(src_of(p));
    const char* a0 = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(a) & ~uintptr_t(15));
    const char* end = a + (int64_t)HW * ES;
    const int nch = (int)((end - a0 + 15) / 16);
    char* d = reinterpret_cast<char*>(stg + p * seg);
    for (int k = lane; k < nch; k += 32) {
      const int64_t left = end - (a0 + 16 * k);
      cp_async16(d + 16 * k, a0 + 16 * k, left >= 16 ? 16 : (int)left);
    }
  }
}

// Dense staging of planes that are one contiguous run in memory (n_elems
// elements from src0): every thread copies 16-byte chunks of the run, so
// small planes do not leave most lanes of a warp idle. Plane data then sits
// at dense_at(stg, src0, offset).
template <typename T>
__device__ __forceinline__ void issue_contig(T* __restrict__ stg, const T* src0, int64_t n_elems) {
  const char* a = reinterpret_cast<const char*>(src0);
  const char* a0 = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(a) & ~uintptr_t(15));
  const char* end = a + n_elems * (int64_t)sizeof(T);
  const int nch = (int)((end - a0 + 15) / 16);
  char* d = reinterpret_cast<char*>(stg);
  for (int k = threadIdx.x; k < nch; k += blockDim.x) {
    const int64_t left = end - (a0 + 16 * k);
    cp_async16(d + 16 * k, a0 + 16 * k, left >= 16 ? 16 : (int)left);
  }
}

template <typename T>
__device__ __forceinline__ const T* dense_at(const T* stg, const T* src0, int off) {
  return stg + (int)((reinterpret_cast<uintptr_t>(src0) & 15) / sizeof(T)) + off;
}


// Segment size (elements) of one densely staged plane: room for the
// in-chunk offset and the rounding of the last chunk.
template <typename T>
inline int dense_seg(int64_t HW) {
  constexpr int CE = 16 / sizeof(T);
  return (int)((HW + 2 * CE + CE - 1) / CE * CE);
}

// Pick the widest copy mode the planes allow and the tile origin column for
// it: want_ix0 (the plane column the kernel wants at tile column 0) rounded
// down to the chunk; *shift = want_ix0 - origin (>= 0) is how far the data
// sits to the right of where the kernel expects it.
template <typename T>
inline int pick_mode(const void* base, int64_t W, int want_ix0, int* ix0, int* shift) {
  constexpr int ES = sizeof(T);
  auto floor_to = [](int v, int m) { return v >= 0 ? v / m * m : -((-v + m - 1) / m) * m; };
  const uintptr_t a = reinterpret_cast<uintptr_t>(base);
  if ((a % 16) == 0 && (W * ES) % 16 == 0) {
    *ix0 = floor_to(want_ix0, 16 / ES);
    *shift = want_ix0 - *ix0;
    return kCopy16;
  }
  if ((a % 4) == 0 && (W * ES) % 4 == 0) {
    *ix0 = floor_to(want_ix0, 4 / ES);
    *shift = want_ix0 - *ix0;
    return kCopy4;
  }
  *ix0 = want_ix0;
  *shift = 0;
  return kCopySync;
}

// ---- reading tile values as fp32 -------------------------------------------
template <typename T>
__device__ __forceinline__ void ld4(const T* p, float* o);
template <>
__device__ __forceinline__ void ld4<float>(const float* p, float* o) {
  const float4 f = *reinterpret_cast<const float4*>(p);
  o[0] = f.x; o[1] = f.y; o[2] = f.z; o[3] = f.w;
}
template <>
__device__ __forceinline__ void ld4<__nv_bfloat16>(const __nv_bfloat16* p, float* o) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  o[0] = __uint_as_float(u.x << 16); o[1] = __uint_as_float(u.x & 0xffff0000u);
  o[2] = __uint_as_float(u.y << 16); o[3] = __uint_as_float(u.y & 0xffff0000u);
}
template <>
__device__ __forceinline__ void ld4<__half>(const __half* p, float* o) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
}
template <typename T>
__device__ __forceinline__ float ld1(const T* p) { return to_f<T>(*p); }

// ---- the register-blocked stencil ------------------------------------------
// Which rows u = r*QS + a*D (r < R, a < K) and window columns i = v*QS + b*D
// (v < V, b < K) a block touches, as bit masks evaluated at compile time (a
// constexpr function called with an unrolled loop index is not folded, so
// the masks are computed once into constants and tested with shifts).
template <int K, int D, int N, int QS>
struct TapMask {
  static constexpr uint64_t value = [] {
    uint64_t m = 0;
    for (int r = 0; r < N; ++r)
      for (int a = 0; a < K; ++a) m |= uint64_t(1) << (r * QS + a * D);
    return m;
  }();
  static_assert((N - 1) * QS + (K - 1) * D < 64, "tap mask wider than 64 bits");
};

template <int K, int D, int R, int QS>
__device__ __forceinline__ constexpr bool row_used(int u) {
  return (TapMask<K, D, R, QS>::value >> u) & 1;
}
template <int K, int D, int V, int QS>
__device__ __forceinline__ constexpr bool col_used(int i) {
  return (TapMask<K, D, V, QS>::value >> i) & 1;
}

// acc[r][v] += sum_{a,b} wr[a*K+b] * t[(tr0 + r*Q*S + a*D) * pitch + tc0 + DL + v*Q*S + b*D]
// With Q == 1 the window of a tile row is contiguous: it is read with 4-wide
// vector loads starting at tc0, which must then be a multiple of 4, and DL
// (0..3) is the compile-time offset of the first used value in it. With
// Q > 1 values are read one by one and DL must be 0 (fold it into tc0).
template <int K, int S, int D, int R, int V, int Q, int DL, typename TS>
__device__ __forceinline__ void conv_block(const TS* __restrict__ t, int pitch, int tr0, int tc0,
                                           const float (&wr)[K * K], float (&acc)[R][V]) {
  constexpr int QS = Q * S;
  constexpr bool VEC = Q == 1;
  constexpr int U = (R - 1) * QS + (K - 1) * D + 1;
  constexpr int WN = (V - 1) * QS + (K - 1) * D + 1;
  constexpr int W4 = (DL + WN + 3) / 4 * 4;
  constexpr int WA = VEC ? W4 : WN;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (!row_used<K, D, R, QS>(u)) continue;
    const TS* rowp = t + (tr0 + u) * pitch + tc0;
    float win[WA];
    if (VEC) {
#pragma unroll
      for (int i = 0; i < W4 / 4; ++i) ld4<TS>(rowp + 4 * i, win + 4 * i);
    } else {
#pragma unroll
      for (int i = 0; i < WA; ++i) win[i] = col_used<K, D, V, QS>(i) ? ld1<TS>(rowp + i) : 0.f;
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int a = 0; a < K; ++a) {
        if (r * QS + a * D != u) continue;
#pragma unroll
        for (int b = 0; b < K; ++b) {
#pragma unroll
          for (int v = 0; v < V; ++v)
            acc[r][v] = fmaf(wr[a * K + b], win[(VEC ? DL : 0) + v * QS + b * D], acc[r][v]);
        }
      }
    }
  }
}

// Same stencil read straight from a densely staged plane (H x W, row-major)
// with zero outside it: iy0 / ix0 are the plane row / column of tap (0, 0) of
// output (0, 0) of the block. Rows outside the plane contribute nothing and
// are skipped; columns outside it read as zero.
template <int K, int S, int D, int R, int V, int Q, typename TS>
__device__ __forceinline__ void conv_block_dense(const TS* __restrict__ plane, int H, int W, int iy0, int ix0,
                                                 const float (&wr)[K * K], float (&acc)[R][V]) {
  constexpr int QS = Q * S;
  constexpr int U = (R - 1) * QS + (K - 1) * D + 1;
  constexpr int WN = (V - 1) * QS + (K - 1) * D + 1;
  bool cin[WN];
#pragma unroll
  for (int i = 0; i < WN; ++i) cin[i] = col_used<K, D, V, QS>(i) && (unsigned)(ix0 + i) < (unsigned)W;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (!row_used<K, D, R, QS>(u)) continue;
    const int iy = iy0 + u;
    if ((unsigned)iy >= (unsigned)H) continue;
    const TS* rowp = plane + iy * W + ix0;
    float win[WN];
#pragma unroll
    for (int i = 0; i < WN; ++i) win[i] = cin[i] ? ld1<TS>(rowp + i) : 0.f;
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

// Start of a densely staged plane: segment p plus the plane's own offset in
// its 16-byte chunk.
template <typename T>
__device__ __forceinline__ const T* dense_plane(const T* stg, int seg, int p, const T* src) {
  return stg + p * seg + (int)((reinterpret_cast<uintptr_t>(src) & 15) / sizeof(T));
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

// Store an R x V block at rows oh + r*Q (r-th valid while r*Q < rows_left),
// cols ow + v*Q (< cols). add: read-modify-write (gx += ...).
template <typename T, int R, int V, int Q>
__device__ __forceinline__ void store_block(T* __restrict__ plane, int64_t Wo, int oh, int ow,
                                            int rows_left, int cols, float (&acc)[R][V], bool vec,
                                            bool add) {
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r * Q >= rows_left) break;
    T* rowp = plane + (int64_t)(oh + r * Q) * Wo;
    if (Q == 1 && V == 4 && vec && ow + V <= cols) {
      float o[4];
#pragma unroll
      for (int v = 0; v < 4; ++v) o[v] = add ? acc[r][v] + ld_rw(rowp + ow + v) : acc[r][v];
      store_vec<T, 4>(rowp + ow, o);
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) {
        const int c = ow + v * Q;
        if (c < cols) rowp[c] = from_f<T>(add ? acc[r][v] + ld_rw(rowp + c) : acc[r][v]);
      }
    }
  }
}

// Work of one persistent CTA, stage by stage. Either units
// u = blockIdx.x + k*gridDim.x of (plane group, band) pairs, or -- when a
// plane is one band and the copies are not tensor copies -- an equal
// contiguous share of the planes, staged ppc planes at a time, so every CTA
// does the same work to within one plane (no tail of idle CTAs).
struct Sched {
  int64_t nplanes, units;
  int ppc;
  int balanced;
  FastDiv d_bands;
  int64_t pb, pe;  // this CTA's share of the planes (balanced)
  __device__ __forceinline__ Sched(int64_t nplanes_, int64_t units_, int ppc_, int balanced_, FastDiv d_bands_)
      : nplanes(nplanes_), units(units_), ppc(ppc_), balanced(balanced_), d_bands(d_bands_) {
    pb = (int64_t)blockIdx.x * nplanes / gridDim.x;
    pe = (int64_t)(blockIdx.x + 1) * nplanes / gridDim.x;
  }
  // stage k of this CTA: first plane, plane count and band; false when done
  __device__ __forceinline__ bool stage(int k, int64_t& p0, int& np, int& band) const {
    if (balanced) {
      p0 = pb + (int64_t)k * ppc;
      if (p0 >= pe) return false;
      np = (int)((pe - p0) < ppc ? (pe - p0) : ppc);
      band = 0;
      return true;
    }
    const int64_t u = blockIdx.x + (int64_t)k * gridDim.x;
    if (u >= units) return false;
    uint32_t grp;
    band = (int)d_bands.divmod((uint32_t)u, grp);
    p0 = (int64_t)grp * ppc;
    np = (int)((nplanes - p0) < ppc ? (nplanes - p0) : ppc);
    return true;
  }
};

// Output staging for units of whole output planes that are contiguous in
// memory but whose rows take no vector stores: the threads write their
// results into a dense copy of the unit's planes in shared memory ...
// ... and the CTA then writes the ne staged elements to dst with 4-element
// vector stores (scalar head and tail up to the alignment), adding the old
// values when add is set. Call after a barrier.
template <typename T>
__device__ __forceinline__ void flush_staged(T* __restrict__ dst, const T* __restrict__ src, int ne, bool add) {
  constexpr int VB = 4 * sizeof(T);  // bytes per vector store
  int head = (int)(((VB - (reinterpret_cast<uintptr_t>(dst) % VB)) % VB) / sizeof(T));
  if (head > ne) head = ne;
  const int nvec = (ne - head) / 4;
  for (int i = threadIdx.x; i < head; i += kNT) dst[i] = add ? from_f<T>(to_f<T>(src[i]) + ld_rw(dst + i)) : src[i];
  for (int i = threadIdx.x; i < nvec; i += kNT) {
    const int e = head + 4 * i;
    float f[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) f[q] = to_f<T>(src[e + q]) + (add ? ld_rw(dst + e + q) : 0.f);
    store_vec<T, 4>(dst + e, f);
  }
  for (int i = head + 4 * nvec + threadIdx.x; i < ne; i += kNT)
    dst[i] = add ? from_f<T>(to_f<T>(src[i]) + ld_rw(dst + i)) : src[i];
}

// ---- host-side planning -------------------------------------------------------
inline int round_up(int64_t v, int m) { return (int)((v + m - 1) / m * m); }

// Stage sizes are kept multiples of 128 bytes (TMA destinations).
inline int stage_round(int64_t elems, int es) { return (int)((elems * es + 127) / 128 * 128 / es); }

// Number of persistent CTAs: every SM's resident capacity, capped by the
// amount of work.
template <typename KernelT>
inline int persistent_grid(KernelT kern, size_t smem, int64_t units) {
  int dev = 0, sms = 152, per_sm = 1;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kNT, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t cap = (int64_t)sms * per_sm;
  return (int)(units < cap ? units : cap);
}

template <typename KernelT>
inline cudaError_t set_smem(KernelT kern, size_t smem) {
  // below the default limit (48 KB, static shared memory included) no opt-in
  // is needed; the tile kernels' static shared memory is a few bytes
  if (smem <= 46 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace tile
}  // namespace dwconv
