// wgrad tile kernels for __nv_bfloat16 storage.
#include "tile_wgrad_impl.cuh"

namespace dwconv {
namespace tile {
template cudaError_t wgrad_t<__nv_bfloat16>(const Conv&, const void*, const void*, float*, int, cudaStream_t);
}  // namespace tile
}  // namespace dwconv
