// Large-kernel family for 27 x 27 filters: forward, stride-1 grad-input and
// weight gradient (kernels in large_impl.cuh).
#include "large_entries.h"
#include "large_impl.cuh"

namespace dwconv {
namespace large {
DW_LARGE_DEFINE(27)
}  // namespace large
}  // namespace dwconv
