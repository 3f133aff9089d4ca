// Large-kernel stride-1 grad-input for float storage.
#include "large_impl.cuh"

namespace dwconv {
namespace large {
template cudaError_t bwd_t<float>(const Conv&, const void*, const void*, void*, bool, cudaStream_t);
}  // namespace large
}  // namespace dwconv
