// Tensor-memory-accelerator (TMA) staging: one thread issues a bulk tensor
// copy of a whole tile (rows x columns x planes) into shared memory; the
// hardware zero-fills every element outside the tensor, which is exactly the
// depthwise zero padding. Completion is tracked by an mbarrier with a
// transaction-byte count.
//
// Every wait on an mbarrier is bounded: after kWaitLimit polls the waiting
// thread gives up, adds one to the library's device timeout counter (its
// address comes from timeout_counter(); the host reads it back with
// dwconv_device_timeouts) and the kernel skips the work of that tile instead
// of hanging.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace dwconv {
namespace tma {

constexpr uint32_t kWaitLimit = 1u << 24;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Order this thread's earlier generic-proxy shared accesses before later
// async-proxy (TMA) writes to the same memory.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// 3-D tiled load: box at coordinates (x, y, z) of the tensor map into dst.
__device__ __forceinline__ void load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                        uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// 4-D tiled load: box at coordinates (x, y, z, w) of the tensor map into dst.
__device__ __forceinline__ void load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                        uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar` (at most `limit` polls); false
// (and *timeouts incremented once per CTA) if it did not complete.
__device__ __forceinline__ bool mbar_wait_n(uint64_t* bar, uint32_t parity, unsigned int* timeouts,
                                            uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  if (threadIdx.x == 0 && timeouts) atomicAdd(timeouts, 1u);
  return false;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* timeouts) {
  return mbar_wait_n(bar, parity, timeouts, kWaitLimit);
}

// Host: encode a 3-D tiled tensor map over a row-major [planes][rows][cols]
// tensor with element size es (cols * es a multiple of 16 bytes, base
// 16-byte aligned). Returns false if the driver refuses it.
bool encode_3d(CUtensorMap* map, const void* base, int dtype, uint64_t cols, uint64_t rows,
               uint64_t planes, uint32_t box_cols, uint32_t box_rows, uint32_t box_planes);

// Host: 4-D tiled tensor map over a row-major [d3][d2][rows][cols] tensor.
bool encode_4d(CUtensorMap* map, const void* base, int dtype, uint64_t cols, uint64_t rows, uint64_t d2,
               uint64_t d3, uint32_t box_cols, uint32_t box_rows, uint32_t box_d2, uint32_t box_d3);

// Host: 3-D tiled tensor map over a row-major [planes][rows][cols] 16-bit
// tensor with the 128-byte swizzle (box_cols * 2 must be 128): the layout the
// tensor-core operand descriptors read as K-major with 128-byte swizzle.
bool encode_3d_sw128(CUtensorMap* map, const void* base, int dtype, uint64_t cols, uint64_t rows,
                     uint64_t planes, uint32_t box_cols, uint32_t box_rows, uint32_t box_planes);

// Host: tiled tensor map of any rank (1..5) with explicit dimensions, byte
// strides of dimensions 1.. (multiples of 16, in any order) and box.
bool encode_strided(CUtensorMap* map, const void* base, int dtype, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box);

// Host: device address of the timeout counter on the current device (looked
// up once per device), or nullptr if the lookup failed.
unsigned int* timeout_counter();

}  // namespace tma
}  // namespace dwconv
