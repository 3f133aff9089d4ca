// Host side of the TMA staging: tensor-map encoding through the driver entry
// point, and the device counter of bounded waits that gave up.
#include <mutex>

#include "tma.cuh"

namespace dwconv {
namespace tma {
namespace {

__device__ unsigned int g_timeouts;

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
unsigned int* g_addr[kMaxDevices];

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeFn>(p);
  }();
  return fn;
}

}  // namespace

bool encode_3d(CUtensorMap* map, const void* base, int dtype, uint64_t cols, uint64_t rows,
               uint64_t planes, uint32_t box_cols, uint32_t box_rows, uint32_t box_planes) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const int es = dtype == DWCONV_F32 ? 4 : 2;
  const CUtensorMapDataType dt = dtype == DWCONV_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == DWCONV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t dims[3] = {cols, rows, planes};
  const cuuint64_t strides[2] = {cols * es, cols * rows * es};
  const cuuint32_t box[3] = {box_cols, box_rows, box_planes};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_4d(CUtensorMap* map, const void* base, int dtype, uint64_t cols, uint64_t rows, uint64_t d2,
               uint64_t d3, uint32_t box_cols, uint32_t box_rows, uint32_t box_d2, uint32_t box_d3) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  const uint64_t es = dtype == DWCONV_F32 ? 4 : 2;
  const CUtensorMapDataType dt = dtype == DWCONV_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == DWCONV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t dims[4] = {cols, rows, d2, d3};
  const cuuint64_t strides[3] = {cols * es, cols * rows * es, cols * rows * d2 * es};
  const cuuint32_t box[4] = {box_cols, box_rows, box_d2, box_d3};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d_sw128(CUtensorMap* map, const void* base, int dtype, uint64_t cols, uint64_t rows,
                     uint64_t planes, uint32_t box_cols, uint32_t box_rows, uint32_t box_planes) {
  EncodeFn fn = encode_fn();
  if (!fn || dtype == DWCONV_F32 || box_cols * 2 != 128) return false;
  const CUtensorMapDataType dt =
      dtype == DWCONV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t dims[3] = {cols, rows, planes};
  const cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  const cuuint32_t box[3] = {box_cols, box_rows, box_planes};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_strided(CUtensorMap* map, const void* base, int dtype, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box) {
  EncodeFn fn = encode_fn();
  if (!fn || rank < 1 || rank > 5) return false;
  const CUtensorMapDataType dt = dtype == DWCONV_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == DWCONV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], estr[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  return fn(map, dt, (cuuint32_t)rank, const_cast<void*>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned int* timeout_counter() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_once[dev], [dev] {
    void* p = nullptr;
    g_addr[dev] = cudaGetSymbolAddress(&p, g_timeouts) == cudaSuccess ? static_cast<unsigned int*>(p) : nullptr;
  });
  return g_addr[dev];
}

}  // namespace tma
}  // namespace dwconv

extern "C" dwconv_status_t dwconv_device_timeouts(unsigned int* count) {
  if (!count) return DWCONV_ERR_INVALID_ARG;
  unsigned int* p = dwconv::tma::timeout_counter();
  if (!p) return DWCONV_ERR_CUDA;
  return cudaMemcpy(count, p, sizeof(unsigned int), cudaMemcpyDeviceToHost) == cudaSuccess ? DWCONV_OK
                                                                                          : DWCONV_ERR_CUDA;
}
