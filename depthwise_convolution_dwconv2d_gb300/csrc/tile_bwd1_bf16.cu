// Stride-1 grad-input tile kernels for __nv_bfloat16 storage.
#include "tile_fwd_impl.cuh"

namespace dwconv {
namespace tile {
template cudaError_t bwd1_t<__nv_bfloat16>(const Conv&, const void*, const void*, void*, bool, cudaStream_t);
}  // namespace tile
}  // namespace dwconv
