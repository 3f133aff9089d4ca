// 16-byte vectors of storage-type values: widening to fp32 and rounding
// back (round to nearest even), for kernels whose lanes move 16 bytes of
// channels at a time.
#pragma once

#include "common.cuh"

namespace dwconv {

template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int n = 4; };
template <> struct Vec<__half> { static constexpr int n = 8; };
template <> struct Vec<__nv_bfloat16> { static constexpr int n = 8; };

// 16 bytes of storage-type values -> fp32 (exact)
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& u, float* o);
template <>
__device__ __forceinline__ void unpack16<float>(const uint4& u, float* o) {
  o[0] = __uint_as_float(u.x); o[1] = __uint_as_float(u.y);
  o[2] = __uint_as_float(u.z); o[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4& u, float* o) {
  const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(v[i] << 16);
    o[2 * i + 1] = __uint_as_float(v[i] & 0xffff0000u);
  }
}
template <>
__device__ __forceinline__ void unpack16<__half>(const uint4& u, float* o) {
  const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v[i]));
    o[2 * i] = f.x;
    o[2 * i + 1] = f.y;
  }
}

// 16 bytes of storage-type values -> fp32 lane pairs (channels 2i, 2i + 1 in
// pair i), exact
template <typename T>
__device__ __forceinline__ void unpack16_pairs(const uint4& u, f32x2* o);
template <>
__device__ __forceinline__ void unpack16_pairs<float>(const uint4& u, f32x2* o) {
  o[0] = ((f32x2)u.y << 32) | u.x;
  o[1] = ((f32x2)u.w << 32) | u.z;
}
template <>
__device__ __forceinline__ void unpack16_pairs<__nv_bfloat16>(const uint4& u, f32x2* o) {
  const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = ((f32x2)(v[i] & 0xffff0000u) << 32) | (uint32_t)(v[i] << 16);
}
template <>
__device__ __forceinline__ void unpack16_pairs<__half>(const uint4& u, f32x2* o) {
  const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v[i]));
    o[i] = pack_f32x2(f.x, f.y);
  }
}

// fp32 -> 16 bytes of storage-type values (round to nearest even)
template <typename T>
__device__ __forceinline__ uint4 pack16(const float* a);
template <>
__device__ __forceinline__ uint4 pack16<float>(const float* a) {
  return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]), __float_as_uint(a[3]));
}
template <>
__device__ __forceinline__ uint4 pack16<__half>(const float* a) {
  uint32_t v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __floats2half2_rn(a[2 * i], a[2 * i + 1]);
    v[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float* a) {
  uint32_t v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
    v[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(v[0], v[1], v[2], v[3]);
}

}  // namespace dwconv
