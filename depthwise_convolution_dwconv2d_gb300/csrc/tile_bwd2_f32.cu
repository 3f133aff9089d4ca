// bwd2 tile kernels for float storage.
#include "tile_bwd2_impl.cuh"

namespace dwconv {
namespace tile {
template cudaError_t bwd2_t<float>(const Conv&, const void*, const void*, void*, bool, cudaStream_t);
}  // namespace tile
}  // namespace dwconv
