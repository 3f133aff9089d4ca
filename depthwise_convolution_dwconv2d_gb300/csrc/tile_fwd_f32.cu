// Forward tile kernels for float storage.
#include "tile_fwd_impl.cuh"

namespace dwconv {
namespace tile {
template cudaError_t fwd_t<float>(const Conv&, const void*, const void*, const void*, void*, cudaStream_t,
                                 const Epi&);
}  // namespace tile
}  // namespace dwconv
