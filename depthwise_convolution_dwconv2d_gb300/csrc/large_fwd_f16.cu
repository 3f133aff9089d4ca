// Large-kernel forward for __half storage.
#include "large_impl.cuh"

namespace dwconv {
namespace large {
template cudaError_t fwd_t<__half>(const Conv&, const void*, const void*, const void*, void*, cudaStream_t);
}  // namespace large
}  // namespace dwconv
