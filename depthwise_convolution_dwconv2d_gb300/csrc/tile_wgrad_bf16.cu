// Weight-gradient tile kernels (multiplier 1) for __nv_bfloat16 storage.
#include "tile_wgrad_impl.cuh"

namespace dwconv {
namespace tile {
template cudaError_t wgrad_sel_t<__nv_bfloat16, 1>(const Conv&, const void*, const void*, float*, int, cudaStream_t);
}  // namespace tile
}  // namespace dwconv
