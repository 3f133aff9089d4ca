// Host-side bounds on the smallest shared-memory band each tile planner can
// choose. A planner gives up (and its call would fail) when even its
// narrowest band exceeds its limit; the shape-support predicates route a
// shape to a tile kernel only when these bounds fit. Each bound follows its
// planner's own arithmetic with the widest row pitch any pointer alignment
// can produce (the copy origin shifts the row by at most one 16-byte chunk),
// so it never undercounts; near the limit a shape that would just have fit
// goes to the large or generic kernels instead.
#pragma once

#include <cstdint>

namespace dwconv {
namespace tile {

inline int64_t fit_rup(int64_t v, int64_t a) { return (v + a - 1) / a * a; }
inline int64_t fit_pitch_align(int es) { return 16 / es > 4 ? 16 / es : 4; }
inline int64_t fit_max_shift(int es) { return 16 / es - 1; }

// Forward (and the stride-1 grad-input, as a forward on grad_out): ntile
// staged planes per plane group, R x V output blocks per thread, Q output
// phases per direction, output rows Wout wide. The narrowest band has Q*R
// output rows.
inline int64_t band_min_bytes(int K, int S, int D, int R, int V, int64_t Wout, int es, int ntile) {
  const int64_t Q = (D % S == 0) ? D / S : 1;
  const int64_t WN = (V - 1) * Q * S + (int64_t)(K - 1) * D + 1;
  const int64_t cb = (Wout + Q * V - 1) / (Q * V);
  const int64_t need = Q == 1 ? (cb - 1) * V * S + fit_max_shift(es) + WN + 3
                              : ((cb - 1) * Q * V + Q - 1) * S + fit_max_shift(es) + WN;
  const int64_t pitch = fit_rup(need, fit_pitch_align(es));
  const int64_t tr = (Q * R - 1) * S + (int64_t)(K - 1) * D + 1;
  return tr * pitch * es * ntile;
}

// Strided grad-input: R x V blocks of grad_out positions per thread (each an
// S x S block of gx), phase PM of the padding, gx rows W wide, m filters per
// channel. The narrowest band has R grad_out rows plus the phase span.
inline int64_t bwd2_min_bytes(int K, int S, int D, int PM, int64_t W, int es, int m) {
  const int R = 2, V = 4;
  int omin = 1 << 20, omax = -(1 << 20);
  for (int p = 0; p < S; ++p)
    for (int a = 0; a < K; ++a) {
      const int t = p + PM - a * D;
      if (t % S != 0) continue;
      const int o = t / S;
      if (o < omin) omin = o;
      if (o > omax) omax = o;
    }
  const int64_t SP = omax - omin;
  const int64_t cb = (W + (int64_t)S * V - 1) / ((int64_t)S * V);
  const int64_t need = (cb - 1) * V + fit_max_shift(es) + V + SP + 3;
  const int64_t pitch = fit_rup(need, fit_pitch_align(es));
  return (R + SP) * pitch * es * m;
}

// Weight gradient: R output rows x V columns per thread, M filters per
// channel, output rows Wo wide. The narrowest band has R output rows.
inline int64_t wgrad_min_bytes(int K, int S, int D, int M, int64_t Wo, int es) {
  const int64_t R = S == 1 ? 2 : 1, V = 4;
  const int64_t cb = (Wo + V - 1) / V;
  const int64_t need = (cb - 1) * V * S + fit_max_shift(es) + (V - 1) * S + (int64_t)(K - 1) * D + 1 + 3;
  const int64_t pitch = fit_rup(need, fit_pitch_align(es));
  const int64_t gpitch = fit_rup(cb * V, fit_pitch_align(es));
  const int64_t tr = (R - 1) * S + (int64_t)(K - 1) * D + 1;
  return (tr * pitch + M * R * gpitch) * es;
}

// Weight gradient: the most bands of output rows its planner can split a
// plane into (its band search, 32 KB per slice, with the widest pitch; a
// narrower pitch gives taller bands, never more of them).
inline int64_t wgrad_max_bands(int K, int S, int D, int M, int64_t Ho, int64_t Wo, int es) {
  const int64_t R = S == 1 ? 2 : 1, V = 4;
  const int64_t cb = (Wo + V - 1) / V;
  const int64_t need = (cb - 1) * V * S + fit_max_shift(es) + (V - 1) * S + (int64_t)(K - 1) * D + 1 + 3;
  const int64_t pitch = fit_rup(need, fit_pitch_align(es));
  const int64_t gpitch = fit_rup(cb * V, fit_pitch_align(es));
  auto bytes_of = [&](int64_t th) { return (((th - 1) * S + (int64_t)(K - 1) * D + 1) * pitch + M * th * gpitch) * es; };
  const int64_t target = 32 * 1024;
  int64_t th = (Ho + R - 1) / R * R;
  if (bytes_of(th) > target) {
    th = R;
    while (bytes_of(th + R) <= target) th += R;
  }
  return (Ho + th - 1) / th;
}

}  // namespace tile
}  // namespace dwconv
