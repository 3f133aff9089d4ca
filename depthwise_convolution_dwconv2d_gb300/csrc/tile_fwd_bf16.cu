// Forward tile kernels for __nv_bfloat16 storage.
#include "tile_fwd_impl.cuh"

namespace dwconv {
namespace tile {
template cudaError_t fwd_t<__nv_bfloat16>(const Conv&, const void*, const void*, const void*, void*, cudaStream_t,
                                 const Epi&);
}  // namespace tile
}  // namespace dwconv
