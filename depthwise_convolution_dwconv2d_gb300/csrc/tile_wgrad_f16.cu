// wgrad tile kernels for __half storage.
#include "tile_wgrad_impl.cuh"

namespace dwconv {
namespace tile {
template cudaError_t wgrad_t<__half>(const Conv&, const void*, const void*, float*, int, cudaStream_t);
}  // namespace tile
}  // namespace dwconv
