// Helpers shared by the large-kernel family (forward / grad-input in
// large_pair.cuh, weight gradient in large_impl.cuh).
#pragma once

#include "plan.h"
#include "tile.cuh"

namespace dwconv {
namespace large {

constexpr int kNT = 256;

// Physical chunk of logical 16-byte chunk q in a row whose even chunks come
// first (half_e = number of even chunks).
__host__ __device__ __forceinline__ int phys_chunk(int q, int half_e) {
  return (q & 1) ? half_e + (q >> 1) : (q >> 1);
}

__device__ __forceinline__ float ld_any(const void* p, int64_t i, int dtype) {
  if (dtype == DWCONV_F32) return __ldg(reinterpret_cast<const float*>(p) + i);
  if (dtype == DWCONV_F16) return __half2float(__ldg(reinterpret_cast<const __half*>(p) + i));
  return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16*>(p) + i));
}

__device__ __forceinline__ float ld_rw_any(const void* p, int64_t i, int dtype) {
  if (dtype == DWCONV_F32) return reinterpret_cast<const float*>(p)[i];
  if (dtype == DWCONV_F16) return __half2float(reinterpret_cast<const __half*>(p)[i]);
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
}

__device__ __forceinline__ void st_any(void* p, int64_t i, float v, int dtype) {
  if (dtype == DWCONV_F32) reinterpret_cast<float*>(p)[i] = v;
  else if (dtype == DWCONV_F16) reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
  else reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

// Stage rows [0, tr) x logical columns [0, 4 nq) of np planes: tile row r,
// column t hold input element (r - pad, t - pad) of plane p (zero outside);
// rows in the de-interleaved chunk layout, planes plane_elems floats apart.
// A warp stages whole rows, its lanes sweeping the columns (coalesced reads).
// Lane l covers columns l + 32 k, which lie in chunks (l >> 2) + 8 k: all of
// one parity, so a lane's destinations are a per-lane base plus 16 k floats.
// fp32 data is copied asynchronously (cp.async with zero fill); 16-bit data
// is widened through registers.
template <typename SrcOf>
__device__ __forceinline__ void stage_planes(float* dst, int np, int plane_elems, int tr, int nq, int half_e,
                                             const FastDiv& d_tr, SrcOf src_of, int Hin, int Win, int pad,
                                             int dtype, bool async4) {
  const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int pitch = 4 * nq;
  const int q0 = lane >> 2;
  const int lane_off = 4 * phys_chunk(q0, half_e) + (lane & 3);
  for (int row = threadIdx.x >> 5; row < np * tr; row += nw) {
    uint32_t p;
    const int r = (int)d_tr.divmod((uint32_t)row, p);
    const int iy = r - pad;
    const bool rin = iy >= 0 && iy < Hin;
    float* d = dst + (int)p * plane_elems + r * pitch + lane_off;
    const char* srow = reinterpret_cast<const char*>(src_of((int)p));
    const int64_t ro = (int64_t)(rin ? iy : 0) * Win;
    for (int col = lane; col < pitch; col += 32, d += 16) {
      const int ix = col - pad;
      const bool in = rin && ix >= 0 && ix < Win;
      if (async4) {
        const float* sp = reinterpret_cast<const float*>(srow) + (in ? ro + ix : 0);
        tile::cp_async4(d, sp, in ? 4 : 0);
      } else {
        *d = in ? ld_any(srow, ro + ix, dtype) : 0.f;
      }
    }
  }
}

}  // namespace large
}  // namespace dwconv
