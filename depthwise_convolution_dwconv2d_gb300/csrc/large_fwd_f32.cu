// Large-kernel forward for float storage.
#include "large_impl.cuh"

namespace dwconv {
namespace large {
template cudaError_t fwd_t<float>(const Conv&, const void*, const void*, const void*, void*, cudaStream_t);
}  // namespace large
}  // namespace dwconv
