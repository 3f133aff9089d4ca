// Large-kernel weight gradient (first pass) for __half storage.
#include "large_impl.cuh"

namespace dwconv {
namespace large {
template cudaError_t wgrad_t<__half>(const Conv&, const void*, const void*, float*, int, cudaStream_t);
}  // namespace large
}  // namespace dwconv
