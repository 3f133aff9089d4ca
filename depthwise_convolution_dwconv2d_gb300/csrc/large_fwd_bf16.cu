// Large-kernel forward for __nv_bfloat16 storage.
#include "large_impl.cuh"

namespace dwconv {
namespace large {
template cudaError_t fwd_t<__nv_bfloat16>(const Conv&, const void*, const void*, const void*, void*, cudaStream_t);
}  // namespace large
}  // namespace dwconv
