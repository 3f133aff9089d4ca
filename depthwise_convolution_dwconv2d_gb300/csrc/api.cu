// libdwconv C ABI: argument validation, the shape planner and dispatch.
//
// Everything here runs on the host. A call validates its descriptor and
// pointers, asks the planner which kernel family to use (a deterministic
// function of the descriptor: the role MegEngine's automatic algorithm
// selection plays in the large-kernel depthwise article, section
// "DirectConv", reduced to fixed shape rules), and enqueues the launches on
// the caller's stream. No allocation, no synchronisation, no global mutable
// state.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "nhwc.h"
#include "plan.h"

namespace dwconv {
namespace {

constexpr int64_t kMaxParam = 1 << 16;
constexpr int64_t kMaxElems = int64_t(1) << 40;

int64_t out_extent(int64_t in, int64_t k, int64_t s, int64_t p, int64_t d) {
  const int64_t span = in + 2 * p - d * (k - 1) - 1;
  return span < 0 ? 0 : span / s + 1;
}

int esize(int dtype) { return dtype == DWCONV_F32 ? 4 : 2; }

dwconv_status_t make_conv(const dwconv2d_desc_t* d, Conv* c) {
  if (!d) return DWCONV_ERR_INVALID_ARG;
  if (d->dtype != DWCONV_F32 && d->dtype != DWCONV_F16 && d->dtype != DWCONV_BF16)
    return DWCONV_ERR_UNSUPPORTED;
  if (d->N < 0 || d->C < 1 || d->H < 1 || d->W < 1 || d->multiplier < 1) return DWCONV_ERR_INVALID_ARG;
  if (d->kh < 1 || d->kw < 1 || d->stride_h < 1 || d->stride_w < 1 || d->dil_h < 1 ||
      d->dil_w < 1 || d->pad_h < 0 || d->pad_w < 0)
    return DWCONV_ERR_INVALID_ARG;
  if (d->kh > 255 || d->kw > 255) return DWCONV_ERR_UNSUPPORTED;
  if (d->stride_h > kMaxParam || d->stride_w > kMaxParam || d->dil_h > kMaxParam ||
      d->dil_w > kMaxParam || d->pad_h > kMaxParam || d->pad_w > kMaxParam ||
      d->multiplier > kMaxParam || d->H > kMaxElems || d->W > kMaxElems || d->C > kMaxElems)
    return DWCONV_ERR_UNSUPPORTED;
  Conv v{};
  v.N = d->N; v.C = d->C; v.H = d->H; v.W = d->W;
  v.m = d->multiplier; v.kh = d->kh; v.kw = d->kw;
  v.sh = d->stride_h; v.sw = d->stride_w; v.ph = d->pad_h; v.pw = d->pad_w;
  v.dh = d->dil_h; v.dw = d->dil_w; v.dtype = d->dtype;
  v.dC = FastDiv((uint32_t)v.C);
  v.Ho = out_extent(v.H, v.kh, v.sh, v.ph, v.dh);
  v.Wo = out_extent(v.W, v.kw, v.sw, v.pw, v.dw);
  if (v.Ho < 1 || v.Wo < 1) return DWCONV_ERR_INVALID_ARG;
  if (v.C * v.m > (int64_t(1) << 31) - 1) return DWCONV_ERR_UNSUPPORTED;
  v.off = d->out_c_offset;
  v.ctot = d->out_c_total == 0 ? v.C * v.m : d->out_c_total;
  if (v.off < 0 || v.ctot < 1 || v.off + v.C * v.m > v.ctot) return DWCONV_ERR_INVALID_ARG;
  // every tensor must stay well inside 64-bit element arithmetic
  if (v.H * v.W > kMaxElems || v.Ho * v.Wo > kMaxElems) return DWCONV_ERR_UNSUPPORTED;
  if (v.N > 0 && (v.N > kMaxElems / (v.C * v.H * v.W) || v.N > kMaxElems / (v.ctot * v.Ho * v.Wo)))
    return DWCONV_ERR_UNSUPPORTED;
  *c = v;
  return DWCONV_OK;
}

bool aligned(const void* p, int es) { return (reinterpret_cast<uintptr_t>(p) % es) == 0; }

dwconv_status_t check_ptr(const void* p, int es, bool required) {
  if (!p) return required ? DWCONV_ERR_INVALID_ARG : DWCONV_OK;
  return aligned(p, es) ? DWCONV_OK : DWCONV_ERR_MISALIGNED;
}

bool act_ok(int a) { return a == DWCONV_ACT_NONE || a == DWCONV_ACT_RELU || a == DWCONV_ACT_RELU6; }

#define DW_TRY(expr)                          \
  do {                                        \
    dwconv_status_t st__ = (expr);            \
    if (st__ != DWCONV_OK) return st__;       \
  } while (0)

dwconv_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DWCONV_OK;
  return DWCONV_ERR_CUDA;
}

size_t ws_bytes(const Conv& c, int chunks) {
  const size_t b = (size_t)chunks * (size_t)c.OC() * (size_t)(c.kh * c.kw + 1) * sizeof(float);
  return (b + 255) & ~size_t(255);
}

// Multi-branch descriptors must agree on everything but the per-branch
// kernel geometry and slice, give one output size, and not overlap.
dwconv_status_t make_multi(int nb, const dwconv2d_desc_t* descs, Conv* cs) {
  if (nb < 1 || nb > kMaxBranches || !descs) return DWCONV_ERR_INVALID_ARG;
  for (int i = 0; i < nb; ++i) {
    DW_TRY(make_conv(&descs[i], &cs[i]));
    const Conv& a = cs[0];
    const Conv& b = cs[i];
    if (b.N != a.N || b.C != a.C || b.H != a.H || b.W != a.W || b.m != a.m ||
        b.dtype != a.dtype || b.ctot != a.ctot || b.Ho != a.Ho || b.Wo != a.Wo)
      return DWCONV_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j) {
      const int64_t lo = cs[j].off, hi = cs[j].off + cs[j].OC();
      if (b.off < hi && lo < b.off + b.OC()) return DWCONV_ERR_INVALID_ARG;
    }
  }
  return DWCONV_OK;
}

}  // namespace
}  // namespace dwconv

using namespace dwconv;

extern "C" {

const char* dwconv_status_string(dwconv_status_t s) {
  switch (s) {
    case DWCONV_OK: return "ok";
    case DWCONV_ERR_INVALID_ARG: return "invalid argument";
    case DWCONV_ERR_UNSUPPORTED: return "unsupported configuration";
    case DWCONV_ERR_MISALIGNED: return "pointer not aligned to its element size";
    case DWCONV_ERR_WORKSPACE: return "workspace missing or too small";
    case DWCONV_ERR_CUDA: return "CUDA launch failed";
  }
  return "unknown status";
}

dwconv_status_t dwconv2d_output_shape(const dwconv2d_desc_t* desc, int64_t* Ho, int64_t* Wo) {
  Conv c;
  DW_TRY(make_conv(desc, &c));
  if (Ho) *Ho = c.Ho;
  if (Wo) *Wo = c.Wo;
  return DWCONV_OK;
}

const char* dwconv2d_plan_name(const dwconv2d_desc_t* desc, int pass) {
  Conv c;
  if (make_conv(desc, &c) != DWCONV_OK || pass < 0 || pass > 4) return "invalid";
  if (pass == 3) return algo_name(plan_fwd(c, true));
  if (pass == 4) return algo_name(nhwc::plan(c));
  return algo_name(pass == 0 ? plan_fwd(c) : pass == 1 ? plan_bwd_data(c) : plan_bwd_weight(c).algo);
}

const char* dwconv2d_multi_plan_name(int nbranch, const dwconv2d_desc_t* descs) {
  Conv cs[kMaxBranches];
  if (make_multi(nbranch, descs, cs) != DWCONV_OK) return "invalid";
  return algo_name(plan_multi(nbranch, cs));
}

dwconv_status_t dwconv2d_fwd(const dwconv2d_desc_t* desc, const void* x, const void* w,
                             const void* bias, void* y, cudaStream_t stream) {
  Conv c;
  DW_TRY(make_conv(desc, &c));
  const int es = esize(c.dtype);
  DW_TRY(check_ptr(w, es, true));
  DW_TRY(check_ptr(bias, es, false));
  if (c.N == 0) return DWCONV_OK;
  DW_TRY(check_ptr(x, es, true));
  DW_TRY(check_ptr(y, es, true));
  return cuda_status(run_fwd(plan_fwd(c), c, x, w, bias, y, stream));
}

dwconv_status_t dwconv2d_fwd_epilogue(const dwconv2d_desc_t* desc, const void* x, const void* w,
                                      const void* bias, const void* scale, const void* shift,
                                      int act, void* y, cudaStream_t stream) {
  Conv c;
  DW_TRY(make_conv(desc, &c));
  if (!act_ok(act)) return DWCONV_ERR_INVALID_ARG;
  const int es = esize(c.dtype);
  DW_TRY(check_ptr(w, es, true));
  DW_TRY(check_ptr(bias, es, false));
  DW_TRY(check_ptr(scale, es, false));
  DW_TRY(check_ptr(shift, es, false));
  if (c.N == 0) return DWCONV_OK;
  DW_TRY(check_ptr(x, es, true));
  DW_TRY(check_ptr(y, es, true));
  const Epi ep{scale, shift, act};
  return cuda_status(run_fwd(plan_fwd(c, ep.active()), c, x, w, bias, y, stream, ep));
}

dwconv_status_t dwconv2d_fwd_nhwc(const dwconv2d_desc_t* desc, const void* x, const void* w,
                                  const void* bias, const void* scale, const void* shift, int act,
                                  void* y, cudaStream_t stream) {
  Conv c;
  DW_TRY(make_conv(desc, &c));
  if (!act_ok(act)) return DWCONV_ERR_INVALID_ARG;
  const int es = esize(c.dtype);
  DW_TRY(check_ptr(w, es, true));
  DW_TRY(check_ptr(bias, es, false));
  DW_TRY(check_ptr(scale, es, false));
  DW_TRY(check_ptr(shift, es, false));
  if (c.N == 0) return DWCONV_OK;
  DW_TRY(check_ptr(x, es, true));
  DW_TRY(check_ptr(y, es, true));
  return cuda_status(nhwc::fwd(c, x, w, bias, y, stream, Epi{scale, shift, act}));
}

namespace {

// The separable block's descriptor: its slice fields describe y's channels
// (cout of them), not the depthwise layer's C*m.
dwconv_status_t make_sep(const dwconv2d_desc_t* desc, int64_t cout, Conv* c, int64_t* ctot, int64_t* off) {
  if (!desc) return DWCONV_ERR_INVALID_ARG;
  dwconv2d_desc_t d = *desc;
  d.out_c_offset = 0;
  d.out_c_total = 0;
  DW_TRY(make_conv(&d, c));
  if (cout < 1) return DWCONV_ERR_INVALID_ARG;
  if (cout > (int64_t(1) << 20)) return DWCONV_ERR_UNSUPPORTED;
  *off = desc->out_c_offset;
  *ctot = desc->out_c_total == 0 ? cout : desc->out_c_total;
  if (*off < 0 || *ctot < 1 || *off + cout > *ctot) return DWCONV_ERR_INVALID_ARG;
  if (c->N > 0 && c->N > kMaxElems / (*ctot * c->Ho * c->Wo)) return DWCONV_ERR_UNSUPPORTED;
  if (!sep::supported(*c)) return DWCONV_ERR_UNSUPPORTED;
  return DWCONV_OK;
}

}  // namespace

dwconv_status_t dwconv2d_separable_nhwc(const dwconv2d_desc_t* desc, const void* x, const void* w_dw,
                                        const void* dw_scale, const void* dw_shift, int dw_act, int64_t cout,
                                        const void* w_pw, const void* pw_scale, const void* pw_shift,
                                        int pw_act, void* y, cudaStream_t stream) {
  Conv c;
  int64_t ctot = 0, off = 0;
  DW_TRY(make_sep(desc, cout, &c, &ctot, &off));
  if (!act_ok(dw_act) || !act_ok(pw_act)) return DWCONV_ERR_INVALID_ARG;
  const int es = esize(c.dtype);
  DW_TRY(check_ptr(w_dw, es, true));
  DW_TRY(check_ptr(w_pw, es, true));
  DW_TRY(check_ptr(dw_scale, es, false));
  DW_TRY(check_ptr(dw_shift, es, false));
  DW_TRY(check_ptr(pw_scale, es, false));
  DW_TRY(check_ptr(pw_shift, es, false));
  if (c.N == 0) return DWCONV_OK;
  DW_TRY(check_ptr(x, es, true));
  DW_TRY(check_ptr(y, es, true));
  return cuda_status(sep::run(c, cout, ctot, off, x, w_dw, dw_scale, dw_shift, dw_act, w_pw, pw_scale, pw_shift,
                              pw_act, y, stream));
}

const char* dwconv2d_separable_plan_name(const dwconv2d_desc_t* desc, int64_t cout) {
  Conv c;
  int64_t ctot = 0, off = 0;
  if (make_sep(desc, cout, &c, &ctot, &off) != DWCONV_OK) return "invalid";
  return algo_name(sep::plan(c, cout));
}

dwconv_status_t dwconv2d_bwd_data(const dwconv2d_desc_t* desc, const void* gy, const void* w,
                                  void* gx, int accumulate, cudaStream_t stream) {
  Conv c;
  DW_TRY(make_conv(desc, &c));
  const int es = esize(c.dtype);
  DW_TRY(check_ptr(w, es, true));
  if (accumulate != 0 && accumulate != 1) return DWCONV_ERR_INVALID_ARG;
  if (c.N == 0) return DWCONV_OK;
  DW_TRY(check_ptr(gy, es, true));
  DW_TRY(check_ptr(gx, es, true));
  return cuda_status(run_bwd_data(plan_bwd_data(c), c, gy, w, gx, accumulate != 0, stream));
}

size_t dwconv2d_bwd_weight_workspace_size(const dwconv2d_desc_t* desc) {
  Conv c;
  if (make_conv(desc, &c) != DWCONV_OK) return 0;
  return ws_bytes(c, plan_bwd_weight(c).chunks);
}

dwconv_status_t dwconv2d_bwd_weight(const dwconv2d_desc_t* desc, const void* x, const void* gy,
                                    void* gw, void* gbias, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
  Conv c;
  DW_TRY(make_conv(desc, &c));
  const int es = esize(c.dtype);
  DW_TRY(check_ptr(gw, es, false));
  DW_TRY(check_ptr(gbias, es, false));
  if (!gw && !gbias) return DWCONV_OK;
  const WPlan p = plan_bwd_weight(c);
  if (!workspace || workspace_bytes < ws_bytes(c, p.chunks)) return DWCONV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return DWCONV_ERR_MISALIGNED;
  if (c.N > 0) {
    DW_TRY(check_ptr(x, es, true));
    DW_TRY(check_ptr(gy, es, true));
  }
  return cuda_status(run_bwd_weight(p, c, x, gy, gw, gbias, (float*)workspace, stream));
}

size_t dwconv2d_filter_cache_size(const dwconv2d_desc_t* desc, int pass) {
  Conv c;
  if (make_conv(desc, &c) != DWCONV_OK || (pass != 0 && pass != 1)) return 0;
  return ibc::cache_bytes(c, pass == 1);
}

namespace {

// Checks shared by the cache build and the cached calls: a cached form for
// this pass, a cache pointer that is 16-byte aligned and large enough.
dwconv_status_t check_cache(const Conv& c, bool flip, const void* cache, size_t cache_bytes) {
  const size_t need = ibc::cache_bytes(c, flip);
  if (need == 0) return DWCONV_ERR_UNSUPPORTED;
  if (!cache || cache_bytes < need) return DWCONV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(cache) % 16 != 0) return DWCONV_ERR_MISALIGNED;
  return DWCONV_OK;
}

}  // namespace

dwconv_status_t dwconv2d_filter_cache_build(const dwconv2d_desc_t* desc, int pass, const void* w, void* cache,
                                            size_t cache_bytes, cudaStream_t stream) {
  Conv c;
  DW_TRY(make_conv(desc, &c));
  if (pass != 0 && pass != 1) return DWCONV_ERR_INVALID_ARG;
  DW_TRY(check_cache(c, pass == 1, cache, cache_bytes));
  DW_TRY(check_ptr(w, esize(c.dtype), true));
  return cuda_status(ibc::build(c, pass == 1, w, cache, stream));
}

dwconv_status_t dwconv2d_fwd_cached(const dwconv2d_desc_t* desc, const void* x, const void* cache,
                                    size_t cache_bytes, const void* bias, void* y, cudaStream_t stream) {
  Conv c;
  DW_TRY(make_conv(desc, &c));
  DW_TRY(check_cache(c, false, cache, cache_bytes));
  const int es = esize(c.dtype);
  DW_TRY(check_ptr(bias, es, false));
  if (c.N == 0) return DWCONV_OK;
  if (!ibc::call_supported(c, false)) return DWCONV_ERR_UNSUPPORTED;
  DW_TRY(check_ptr(x, 16, true));
  DW_TRY(check_ptr(y, es, true));
  return cuda_status(ibc::run(c, false, x, cache, bias, y, false, stream));
}

dwconv_status_t dwconv2d_bwd_data_cached(const dwconv2d_desc_t* desc, const void* gy, const void* cache,
                                         size_t cache_bytes, void* gx, int accumulate, cudaStream_t stream) {
  Conv c;
  DW_TRY(make_conv(desc, &c));
  DW_TRY(check_cache(c, true, cache, cache_bytes));
  if (accumulate != 0 && accumulate != 1) return DWCONV_ERR_INVALID_ARG;
  if (c.N == 0) return DWCONV_OK;
  if (!ibc::call_supported(c, true)) return DWCONV_ERR_UNSUPPORTED;
  DW_TRY(check_ptr(gy, 16, true));
  DW_TRY(check_ptr(gx, esize(c.dtype), true));
  return cuda_status(ibc::run(c, true, gy, cache, nullptr, gx, accumulate != 0, stream));
}

dwconv_status_t dwconv2d_fwd_multi(int nbranch, const dwconv2d_desc_t* descs, const void* x,
                                   const void* const* w, const void* const* bias, void* y,
                                   cudaStream_t stream) {
  Conv cs[kMaxBranches];
  DW_TRY(make_multi(nbranch, descs, cs));
  if (!w) return DWCONV_ERR_INVALID_ARG;
  const int es = esize(cs[0].dtype);
  for (int i = 0; i < nbranch; ++i) {
    DW_TRY(check_ptr(w[i], es, true));
    DW_TRY(check_ptr(bias ? bias[i] : nullptr, es, false));
  }
  if (cs[0].N == 0) return DWCONV_OK;
  DW_TRY(check_ptr(x, es, true));
  DW_TRY(check_ptr(y, es, true));
  return cuda_status(run_fwd_multi(nbranch, cs, x, w, bias, y, stream));
}

dwconv_status_t dwconv2d_bwd_data_multi(int nbranch, const dwconv2d_desc_t* descs, const void* gy,
                                        const void* const* w, void* gx, cudaStream_t stream) {
  Conv cs[kMaxBranches];
  DW_TRY(make_multi(nbranch, descs, cs));
  if (!w) return DWCONV_ERR_INVALID_ARG;
  const int es = esize(cs[0].dtype);
  for (int i = 0; i < nbranch; ++i) DW_TRY(check_ptr(w[i], es, true));
  if (cs[0].N == 0) return DWCONV_OK;
  DW_TRY(check_ptr(gy, es, true));
  DW_TRY(check_ptr(gx, es, true));
  return cuda_status(run_bwd_data_multi(nbranch, cs, gy, w, gx, stream));
}

}  // extern "C"
