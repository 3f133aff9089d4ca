// Shape planner: picks a kernel family per pass from the descriptor alone,
// so a descriptor always maps to the same kernels (and the same bwd_weight
// workspace size). DWCONV_FORCE_ALGO=generic pins every pass to the generic
// kernels (used by the tests to cross-check the tiled ones).
#include <cstdlib>
#include <cstring>

#include "plan.h"

namespace dwconv {
namespace {

bool force_generic() {
  const char* e = std::getenv("DWCONV_FORCE_ALGO");
  return e && std::strcmp(e, "generic") == 0;
}

// DWCONV_FORCE_ALGO=direct keeps the large 16-bit shapes on the direct
// kernels (used by the tests to cross-check the tensor-core ones).
bool allow_ibgemm() {
  const char* e = std::getenv("DWCONV_FORCE_ALGO");
  return !(e && (std::strcmp(e, "generic") == 0 || std::strcmp(e, "direct") == 0));
}

}  // namespace

const char* algo_name(Algo a) {
  switch (a) {
    case Algo::Generic: return "generic";
    case Algo::Tile: return "tile";
    case Algo::Large: return "large";
    case Algo::IBGemm: return "ibgemm";
    case Algo::Plane: return "plane";
    case Algo::TcWgrad: return "tcwgrad";
    case Algo::Nhwc: return "nhwc";
    case Algo::SepTc: return "septc";
  }
  return "unknown";
}

Algo plan_fwd(const Conv& c, bool epilogue) {
  if (force_generic()) return Algo::Generic;
  // the small-plane and tensor-core kernels have no fused epilogue
  if (!epilogue && plane::fwd_supported(c)) return Algo::Plane;
  if (tile::fwd_supported(c)) return Algo::Tile;
  if (!epilogue && allow_ibgemm() && ibg::fwd_supported(c)) return Algo::IBGemm;
  if (large::supported(c)) return Algo::Large;
  return Algo::Generic;
}

Algo plan_bwd_data(const Conv& c) {
  if (force_generic()) return Algo::Generic;
  if (plane::bwd_data_supported(c)) return Algo::Plane;
  if (c.sh == 1 ? tile::bwd1_supported(c) : tile::bwd2_supported(c)) return Algo::Tile;
  if (allow_ibgemm() && ibg::bwd_data_supported(c)) return Algo::IBGemm;
  if (large::supported(c)) return Algo::Large;
  return Algo::Generic;
}

WPlan plan_bwd_weight(const Conv& c) {
  if (!force_generic() && plane::wgrad_supported(c)) return WPlan{Algo::Plane, plane::wgrad_chunks(c)};
  if (!force_generic() && tile::wgrad_supported(c)) return WPlan{Algo::Tile, tile::wgrad_chunks(c)};
  if (!force_generic() && allow_ibgemm() && wtc::supported(c)) return WPlan{Algo::TcWgrad, large::sample_chunks(c)};
  if (!force_generic() && large::wgrad_supported(c)) return WPlan{Algo::Large, large::wgrad_chunks(c)};
  // generic first pass: a chunk of whole samples per block, at most 2^20
  // positions per chunk so each thread's serial chain stays <= 4096 terms.
  const int64_t hw = c.Ho * c.Wo;
  int64_t nb = (int64_t(1) << 20) / hw;
  if (nb < 1) nb = 1;
  if (nb > c.N) nb = c.N > 0 ? c.N : 1;
  int64_t chunks = c.N > 0 ? (c.N + nb - 1) / nb : 1;
  if (chunks > 65535) chunks = 65535;
  return WPlan{Algo::Generic, (int)chunks};
}

cudaError_t run_fwd(Algo a, const Conv& c, const void* x, const void* w, const void* b, void* y,
                    cudaStream_t s, const Epi& ep) {
  switch (a) {
    case Algo::Plane: return plane::fwd(c, x, w, b, y, s);
    case Algo::Tile: return tile::fwd(c, x, w, b, y, s, ep);
    case Algo::Large: return large::fwd(c, x, w, b, y, s, ep);
    case Algo::IBGemm: {
      // a misaligned pointer rules the tensor-core kernel out for this call
      // only; it has no fused epilogue
      const cudaError_t e = ep.active() ? cudaErrorNotSupported : ibg::fwd(c, x, w, b, y, s);
      if (e != cudaErrorNotSupported) return e;
      return large::supported(c) ? large::fwd(c, x, w, b, y, s, ep) : fwd_generic(c, x, w, b, y, s, ep);
    }
    default: return fwd_generic(c, x, w, b, y, s, ep);
  }
}

cudaError_t run_bwd_data(Algo a, const Conv& c, const void* gy, const void* w, void* gx,
                         bool accumulate, cudaStream_t s) {
  switch (a) {
    case Algo::Plane: return plane::bwd_data(c, gy, w, gx, accumulate, s);
    case Algo::Tile:
      return c.sh == 1 ? tile::bwd1(c, gy, w, gx, accumulate, s) : tile::bwd2(c, gy, w, gx, accumulate, s);
    case Algo::Large: return large::bwd_data(c, gy, w, gx, accumulate, s);
    case Algo::IBGemm: {
      const cudaError_t e = ibg::bwd_data(c, gy, w, gx, accumulate, s);
      if (e != cudaErrorNotSupported) return e;
      return large::supported(c) ? large::bwd_data(c, gy, w, gx, accumulate, s)
                                 : bwd_data_generic(c, gy, w, gx, accumulate, s);
    }
    default: return bwd_data_generic(c, gy, w, gx, accumulate, s);
  }
}

cudaError_t run_bwd_weight(const WPlan& p, const Conv& c, const void* x, const void* gy, void* gw,
                           void* gb, float* ws, cudaStream_t s) {
  cudaError_t e;
  switch (p.algo) {
    case Algo::Plane:
      e = plane::wgrad(c, x, gy, ws, p.chunks, s);
      break;
    case Algo::Tile:
      e = tile::wgrad(c, x, gy, ws, p.chunks, s);
      break;
    case Algo::Large:
      e = large::wgrad(c, x, gy, ws, p.chunks, s);
      break;
    case Algo::TcWgrad:
      // a misaligned pointer rules the tensor-core kernel out for this call
      // only; the direct kernels take the same chunks (same workspace)
      e = wtc::wgrad(c, x, gy, ws, p.chunks, s);
      if (e == cudaErrorNotSupported)
        e = large::wgrad_scalar_supported(c) ? large::wgrad_scalar(c, x, gy, ws, p.chunks, s)
                                      : bwd_weight_generic_pass1(c, x, gy, ws, p.chunks, gw != nullptr, gb != nullptr, s);
      break;
    default:
      e = bwd_weight_generic_pass1(c, x, gy, ws, p.chunks, gw != nullptr, gb != nullptr, s);
      break;
  }
  if (e != cudaSuccess) return e;
  return bwd_weight_pass2(c, ws, p.chunks, gw, gb, s);
}

Algo plan_multi(int nb, const Conv* cs) {
  if (!force_generic() && tile::multi_supported(nb, cs)) return Algo::Tile;
  return Algo::Generic;
}

cudaError_t run_fwd_multi(int nb, const Conv* cs, const void* x, const void* const* w,
                          const void* const* bias, void* y, cudaStream_t s) {
  if (plan_multi(nb, cs) == Algo::Tile) return tile::fwd_multi(nb, cs, x, w, bias, y, s);
  // branches write disjoint slices: one launch per branch
  for (int i = 0; i < nb; ++i) {
    cudaError_t e = run_fwd(plan_fwd(cs[i]), cs[i], x, w[i], bias ? bias[i] : nullptr, y, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t run_bwd_data_multi(int nb, const Conv* cs, const void* gy, const void* const* w,
                               void* gx, cudaStream_t s) {
  if (plan_multi(nb, cs) == Algo::Tile) return tile::bwd_multi(nb, cs, gy, w, gx, s);
  MultiGeneric m{};
  m.nb = nb;
  for (int i = 0; i < nb; ++i) {
    m.c[i] = cs[i];
    m.w[i] = w[i];
  }
  return bwd_data_multi_generic(m, gy, gx, s);
}

}  // namespace dwconv
