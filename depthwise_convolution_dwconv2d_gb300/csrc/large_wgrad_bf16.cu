// Large-kernel weight gradient (first pass) for __nv_bfloat16 storage.
#include "large_impl.cuh"

namespace dwconv {
namespace large {
template cudaError_t wgrad_t<__nv_bfloat16>(const Conv&, const void*, const void*, float*, int, cudaStream_t);
}  // namespace large
}  // namespace dwconv
