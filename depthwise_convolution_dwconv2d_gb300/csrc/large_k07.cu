// Large-kernel family for 7 x 7 filters: forward, stride-1 grad-input and
// weight gradient (kernels in large_impl.cuh).
#include "large_entries.h"
#include "large_impl.cuh"

namespace dwconv {
namespace large {
DW_LARGE_DEFINE(7)
}  // namespace large
}  // namespace dwconv
