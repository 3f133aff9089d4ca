// Internal types and helpers shared by the libdwconv kernels (not installed).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "dwconv.h"

namespace dwconv {

// Division of 32-bit unsigned numerators by a divisor fixed at launch time,
// as a multiply-high and two shifts (Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, section 4): with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// t = mulhi(m, n), q = (t + ((n - t) >> 1)) >> (l - 1), exact for all n < 2^32.
struct FastDiv {
  uint32_t d, m, s1, s2;
  FastDiv() = default;
  __host__ explicit FastDiv(uint32_t div) : d(div) {
    uint32_t l = 0;
    while ((uint64_t(1) << l) < div) ++l;
    m = (uint32_t)(((uint64_t(1) << 32) * ((uint64_t(1) << l) - div)) / div + 1);
    s1 = l > 0 ? 1u : 0u;
    s2 = l > 0 ? l - 1 : 0u;
  }
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    const uint32_t t = __umulhi(m, n);
    return (t + ((n - t) >> s1)) >> s2;
  }
  // q = n / d, returns n - q * d
  __device__ __forceinline__ uint32_t divmod(uint32_t n, uint32_t& q) const {
    q = div(n);
    return n - q * d;
  }
};

// Validated convolution geometry, passed to kernels by value.
struct Conv {
  int64_t N, C, H, W;
  int m, kh, kw, sh, sw, ph, pw, dh, dw;
  int64_t Ho, Wo;
  int64_t off, ctot;  // channel slice of y / gy
  int dtype;
  FastDiv dC;         // division by C: plane index (n*C + c) -> (n, c)

  // The tiled kernels index planes n*C + c in 32 bits.
  __host__ __device__ bool planes32() const { return N * C * m < (int64_t(1) << 31); }
  // plane index -> (sample, channel); valid when planes32()
  __device__ __forceinline__ void split(int64_t pin, int64_t& n, int64_t& ch) const {
    uint32_t q;
    const uint32_t r = dC.divmod((uint32_t)pin, q);
    n = q;
    ch = r;
  }

  __host__ __device__ int64_t OC() const { return C * m; }
  __host__ __device__ int64_t x_plane() const { return H * W; }
  __host__ __device__ int64_t y_plane() const { return Ho * Wo; }
  // element offset of plane (n, oc) in y / gy
  __host__ __device__ int64_t y_base(int64_t n, int64_t oc) const {
    return (n * ctot + off + oc) * Ho * Wo;
  }
  __host__ __device__ int64_t x_base(int64_t n, int64_t c) const {
    return (n * C + c) * H * W;
  }
};

// ---- storage type <-> fp32 -------------------------------------------------
template <typename T> __device__ __forceinline__ float ld(const T* p);
template <> __device__ __forceinline__ float ld<float>(const float* p) { return __ldg(p); }
template <> __device__ __forceinline__ float ld<__half>(const __half* p) { return __half2float(__ldg(p)); }
template <> __device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Two fp32 values in one 64-bit register (lane 0 in the low word), the operand
// form of the two-lane FP32 instructions of the sm_100 family.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack_f32x2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// d = a * b + d on both lanes (PTX fma.rn.f32x2): each lane is one IEEE fused
// multiply-add with a single rounding, the same as fmaf on that lane.
__device__ __forceinline__ void fma_f32x2(f32x2& d, f32x2 a, f32x2 b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// plain (coherent) load for data this kernel may also write
template <typename T> __device__ __forceinline__ float ld_rw(const T* p) { return to_f<T>(*p); }



// Fused epilogue of the forward: y = act(scale[oc] * (conv + bias[oc]) +
// shift[oc]) -- a folded batch norm (scale = gamma / sqrt(var + eps), shift =
// beta - mean * scale) and an activation, applied to the fp32 result before
// its one rounding to the storage type. scale / shift may be null (1 / 0).
struct Epi {
  const void* scale;
  const void* shift;
  int act;  // DWCONV_ACT_*
  __host__ __device__ bool active() const { return scale != nullptr || shift != nullptr || act != 0; }
};

__device__ __forceinline__ float epi_act(float v, int act) {
  if (act == DWCONV_ACT_RELU) return fmaxf(v, 0.f);
  if (act == DWCONV_ACT_RELU6) return fminf(fmaxf(v, 0.f), 6.f);
  return v;
}

inline int div_up(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// Launch helpers: each family exposes launch functions templated on nothing;
// dtype dispatch happens inside.
#define DWCONV_DISPATCH_DTYPE(dt, T, ...)                        \
  switch (dt) {                                                  \
    case DWCONV_F32: { using T = float; __VA_ARGS__; } break;    \
    case DWCONV_F16: { using T = __half; __VA_ARGS__; } break;   \
    case DWCONV_BF16: { using T = __nv_bfloat16; __VA_ARGS__; } break; \
    default: break;                                              \
  }

// ---- kernel families (each returns cudaGetLastError() after its launches) --
// generic.cu: correct for every valid descriptor, one output per thread.
cudaError_t fwd_generic(const Conv& c, const void* x, const void* w, const void* b, void* y,
                        cudaStream_t s, const Epi& ep = Epi{});
cudaError_t bwd_data_generic(const Conv& c, const void* gy, const void* w, void* gx,
                             bool accumulate, cudaStream_t s);
struct MultiGeneric {
  int nb;
  Conv c[8];
  const void* w[8];
};
cudaError_t bwd_data_multi_generic(const MultiGeneric& m, const void* gy, void* gx, cudaStream_t s);
// pass 1 writes ws[chunk][oc][taps + 1] (last slot = bias) for `chunks` batch chunks.
cudaError_t bwd_weight_generic_pass1(const Conv& c, const void* x, const void* gy, float* ws,
                                     int chunks, bool want_w, bool want_b, cudaStream_t s);
cudaError_t bwd_weight_pass2(const Conv& c, const float* ws, int chunks, void* gw, void* gb,
                             cudaStream_t s);

}  // namespace dwconv
