// Stride-1 grad-input tile kernels for __half storage.
#include "tile_fwd_impl.cuh"

namespace dwconv {
namespace tile {
template cudaError_t bwd1_t<__half>(const Conv&, const void*, const void*, void*, bool, cudaStream_t);
}  // namespace tile
}  // namespace dwconv
