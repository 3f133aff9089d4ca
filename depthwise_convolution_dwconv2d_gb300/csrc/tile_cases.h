// Shape combinations compiled for the tile kernels.
#pragma once

// (K, S, D) combinations compiled for the forward tile kernel.
#define DW_FWD_CASES(X) X(1, 1, 1) X(3, 1, 1) X(3, 2, 1) X(5, 1, 1) X(5, 2, 1) X(7, 1, 1) \
  X(7, 2, 1) X(3, 1, 2) X(3, 1, 3) X(3, 1, 5) X(5, 1, 2) X(3, 2, 2) X(3, 3, 1) X(5, 1, 3)
// (K, D) combinations compiled for the stride-1 grad-input tile kernel.
#define DW_BWD1_CASES(X) X(1, 1) X(3, 1) X(5, 1) X(7, 1) X(3, 2) X(3, 3) X(3, 5) X(5, 2) X(5, 3)

#define DW_BWD2_CASES(X) X(3, 2, 1, 0) X(3, 2, 1, 1) X(5, 2, 1, 0) X(5, 2, 1, 1) X(7, 2, 1, 1) X(7, 2, 1, 0) \
  X(3, 3, 1, 0) X(3, 3, 1, 1)

#define DW_WGRAD_CASES(X) X(3, 1, 1, 1) X(3, 2, 1, 1) X(5, 1, 1, 1) X(5, 2, 1, 1) X(3, 1, 1, 2) \
  X(5, 1, 1, 2) X(3, 2, 1, 2) X(7, 1, 1, 1) X(3, 1, 2, 1) X(3, 1, 3, 1) X(3, 1, 5, 1) X(3, 3, 1, 1) \
  X(5, 1, 3, 1) X(7, 2, 1, 1)
