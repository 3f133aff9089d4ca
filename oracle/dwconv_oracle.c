/*
 * Depthwise 2-D convolution oracle: plain nested loops, fp64 accumulation.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker that the CUDA path is
 * compared against. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it. It shares no code, header, table or helper
 * with the CUDA library, and it never calls it.
 *
 * What it computes (all three are exact linear maps, so each function below
 * is the plain definition written out, with no blocking, fusion or reordering):
 *
 *   forward     y[n, off + c*m + j, oh, ow] =
 *                   bias[c*m + j]
 *                 + sum_{a, b} w[c*m + j, a, b] * x[n, c, oh*sh - ph + a*dh,
 *                                                       ow*sw - pw + b*dw]
 *               with taps that land outside the input skipped (zero padding).
 *               Sources: "Spatial Depthwise Convolution on the GPU #3057"
 *               (the forward binding conv_depthwise2d_forward_out with
 *               kernel_size, bias, stride, padding, dilation, and the commits
 *               that add padding, strides, dilation, the depth multiplier and
 *               bias); the MegEngine large-kernel depthwise article, section
 *               "From convolution to matrix multiplication" (the sliding
 *               window over the input, one channel at a time); the
 *               DynamicConvolutionOperator README, section "Solution" (each
 *               branch stored into its own channel slice of one concatenated
 *               output, hence off / c_total).
 *   bwd_data    gx = adjoint of forward in x (the grad-input kernel of #3057).
 *               Written as a gather over the forward index relation: input
 *               pixel (ih, iw) receives w * gy from every output (oh, ow) and
 *               tap (a, b) with oh*sh - ph + a*dh == ih, ow*sw - pw + b*dw == iw.
 *   bwd_weight  gw[oc, a, b] = sum_{n, oh, ow} gy[n, off+oc, oh, ow] *
 *                                x[n, oc/m, oh*sh - ph + a*dh, ow*sw - pw + b*dw]
 *               gb[oc] = sum_{n, oh, ow} gy[n, off+oc, oh, ow]
 *               (the grad-weight kernel and grad_bias of #3057).
 *   epilogue    y = act(scale * y + shift) per output channel after the
 *               forward (oracle_epilogue below).
 *   pointwise   the 1x1 convolution that follows the depthwise layer in a
 *               depthwise-separable block (oracle_pointwise below).
 *
 * Readings where the pages are silent: cross-correlation (no kernel flip, as
 * PyTorch's conv2d); Ho = floor((H + 2ph - dh(kh-1) - 1)/sh) + 1; symmetric
 * zero padding; output channel oc = c*m + j reads input channel c.
 *
 * Parallelism: OpenMP over outputs that are independent (n, oc for forward;
 * n, c for bwd_data; oc for bwd_weight). Inside each, the sum runs serially in
 * a fixed order, so results do not depend on the thread count.
 */
#include <stdint.h>
#include <stddef.h>

typedef struct {
  int64_t N, C, H, W;
  int64_t m;                 /* depth multiplier */
  int64_t kh, kw, sh, sw, ph, pw, dh, dw;
  int64_t off;               /* first channel of this op in y / gy */
  int64_t c_total;           /* channel count of the y / gy buffer */
} oracle_desc;

static int64_t out_extent(int64_t in, int64_t k, int64_t s, int64_t p, int64_t d) {
  int64_t span = in + 2 * p - d * (k - 1) - 1;
  if (span < 0) return 0;
  return span / s + 1;
}

int64_t oracle_out_h(const oracle_desc* d) { return out_extent(d->H, d->kh, d->sh, d->ph, d->dh); }
int64_t oracle_out_w(const oracle_desc* d) { return out_extent(d->W, d->kw, d->sw, d->pw, d->dw); }

void oracle_dwconv2d_fwd(const oracle_desc* d, const double* x, const double* w,
                         const double* bias, double* y) {
  const int64_t Ho = oracle_out_h(d), Wo = oracle_out_w(d);
  const int64_t OC = d->C * d->m;
  const int64_t total = d->N * OC;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < total; ++t) {
    const int64_t n = t / OC, oc = t % OC, c = oc / d->m;
    const double* xp = x + (n * d->C + c) * d->H * d->W;
    const double* wp = w + oc * d->kh * d->kw;
    double* yp = y + (n * d->c_total + d->off + oc) * Ho * Wo;
    for (int64_t oh = 0; oh < Ho; ++oh) {
      for (int64_t ow = 0; ow < Wo; ++ow) {
        double acc = 0.0;
        for (int64_t a = 0; a < d->kh; ++a) {
          const int64_t ih = oh * d->sh - d->ph + a * d->dh;
          if (ih < 0 || ih >= d->H) continue;
          for (int64_t b = 0; b < d->kw; ++b) {
            const int64_t iw = ow * d->sw - d->pw + b * d->dw;
            if (iw < 0 || iw >= d->W) continue;
            acc += wp[a * d->kw + b] * xp[ih * d->W + iw];
          }
        }
        if (bias) acc += bias[oc];
        yp[oh * Wo + ow] = acc;
      }
    }
  }
}

/* gx is overwritten. */
void oracle_dwconv2d_bwd_data(const oracle_desc* d, const double* gy, const double* w,
                              double* gx) {
  const int64_t Ho = oracle_out_h(d), Wo = oracle_out_w(d);
  const int64_t total = d->N * d->C;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < total; ++t) {
    const int64_t n = t / d->C, c = t % d->C;
    double* gxp = gx + (n * d->C + c) * d->H * d->W;
    for (int64_t ih = 0; ih < d->H; ++ih) {
      for (int64_t iw = 0; iw < d->W; ++iw) {
        double acc = 0.0;
        for (int64_t j = 0; j < d->m; ++j) {
          const int64_t oc = c * d->m + j;
          const double* gyp = gy + (n * d->c_total + d->off + oc) * Ho * Wo;
          const double* wp = w + oc * d->kh * d->kw;
          for (int64_t a = 0; a < d->kh; ++a) {
            const int64_t num_h = ih + d->ph - a * d->dh;   /* = oh * sh */
            if (num_h < 0 || num_h % d->sh != 0) continue;
            const int64_t oh = num_h / d->sh;
            if (oh >= Ho) continue;
            for (int64_t b = 0; b < d->kw; ++b) {
              const int64_t num_w = iw + d->pw - b * d->dw;  /* = ow * sw */
              if (num_w < 0 || num_w % d->sw != 0) continue;
              const int64_t ow = num_w / d->sw;
              if (ow >= Wo) continue;
              acc += wp[a * d->kw + b] * gyp[oh * Wo + ow];
            }
          }
        }
        gxp[ih * d->W + iw] = acc;
      }
    }
  }
}

/* gw [C*m, kh, kw] and gb [C*m] are overwritten; either may be NULL. */
void oracle_dwconv2d_bwd_weight(const oracle_desc* d, const double* x, const double* gy,
                                double* gw, double* gb) {
  const int64_t Ho = oracle_out_h(d), Wo = oracle_out_w(d);
  const int64_t OC = d->C * d->m;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t oc = 0; oc < OC; ++oc) {
    const int64_t c = oc / d->m;
    if (gw) {
      for (int64_t a = 0; a < d->kh; ++a) {
        for (int64_t b = 0; b < d->kw; ++b) {
          double acc = 0.0;
          for (int64_t n = 0; n < d->N; ++n) {
            const double* xp = x + (n * d->C + c) * d->H * d->W;
            const double* gyp = gy + (n * d->c_total + d->off + oc) * Ho * Wo;
            for (int64_t oh = 0; oh < Ho; ++oh) {
              const int64_t ih = oh * d->sh - d->ph + a * d->dh;
              if (ih < 0 || ih >= d->H) continue;
              for (int64_t ow = 0; ow < Wo; ++ow) {
                const int64_t iw = ow * d->sw - d->pw + b * d->dw;
                if (iw < 0 || iw >= d->W) continue;
                acc += gyp[oh * Wo + ow] * xp[ih * d->W + iw];
              }
            }
          }
          gw[(oc * d->kh + a) * d->kw + b] = acc;
        }
      }
    }
    if (gb) {
      double acc = 0.0;
      for (int64_t n = 0; n < d->N; ++n) {
        const double* gyp = gy + (n * d->c_total + d->off + oc) * Ho * Wo;
        for (int64_t i = 0; i < Ho * Wo; ++i) acc += gyp[i];
      }
      gb[oc] = acc;
    }
  }
}

/* Fused forward epilogue, applied in place to this op's channels
 * [off, off + C*m) of y once oracle_dwconv2d_fwd has written them:
 *   v = scale[oc] * v + shift[oc]        (scale NULL: 1, shift NULL: 0)
 *   act 1: v = max(v, 0);  act 2: v = min(max(v, 0), 6);  act 0: unchanged.
 * Source: the Megvii article on custom convolution operators with cutlass
 * (its opening list: a user of a basic operator library cannot add a new
 * activation to the convolution). Reading: scale / shift are a batch norm in
 * inference form folded per output channel; the activation comes last. */
void oracle_epilogue(const oracle_desc* d, const double* scale, const double* shift, int act,
                     double* y) {
  const int64_t Ho = oracle_out_h(d), Wo = oracle_out_w(d);
  const int64_t OC = d->C * d->m;
  for (int64_t n = 0; n < d->N; ++n) {
    for (int64_t oc = 0; oc < OC; ++oc) {
      double* yp = y + (n * d->c_total + d->off + oc) * Ho * Wo;
      const double sc = scale ? scale[oc] : 1.0;
      const double sh = shift ? shift[oc] : 0.0;
      for (int64_t i = 0; i < Ho * Wo; ++i) {
        double v = sc * yp[i] + sh;
        if (act == 1 || act == 2) v = v > 0.0 ? v : 0.0;
        if (act == 2) v = v < 6.0 ? v : 6.0;
        yp[i] = v;
      }
    }
  }
}

/* Pointwise (1x1) convolution of a depthwise-separable block:
 *   y[n, co, i] = sum_{ci < cin} wp[co, ci] * z[n, ci, i]     (i over hw pixels)
 * z [n][cin][hw], wp [cout][cin] (PyTorch's [cout, cin, 1, 1]), y
 * [n][cout][hw], overwritten. Source: "Spatial Depthwise Convolution on the
 * GPU #3057", the MobileNet benchmark table that times the 1x1 layer after
 * each depthwise layer. */
void oracle_pointwise(int64_t n, int64_t cin, int64_t cout, int64_t hw, const double* z,
                      const double* wp, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n * cout; ++t) {
    const int64_t b = t / cout, co = t % cout;
    double* yp = y + (b * cout + co) * hw;
    for (int64_t i = 0; i < hw; ++i) yp[i] = 0.0;
    for (int64_t ci = 0; ci < cin; ++ci) {
      const double wv = wp[co * cin + ci];
      const double* zp = z + (b * cin + ci) * hw;
      for (int64_t i = 0; i < hw; ++i) yp[i] += wv * zp[i];
    }
  }
}

/* Thread count OpenMP will use (1 when built without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int oracle_num_threads(void) { return 1; }
#endif
