// Large-kernel family for 23 x 23 filters: forward, stride-1 grad-input and
// weight gradient (kernels in large_impl.cuh).
#include "large_entries.h"
#include "large_impl.cuh"

namespace dwconv {
namespace large {
DW_LARGE_DEFINE(23)
}  // namespace large
}  // namespace dwconv
