/*
 * libdwconv -- depthwise 2-D convolution on NVIDIA GB300 (sm_103a).
 *
 * C ABI. Every entry point takes a descriptor, plain pointers and sizes, and
 * a CUDA stream. No framework types cross this boundary.
 *
 * The operation (sources: "Spatial Depthwise Convolution on the GPU #3057",
 * the forward binding conv_depthwise2d_forward_out(output, input, weight,
 * kernel_size, bias, stride, padding, dilation) and the commits that add
 * padding, strides, dilation, the depth multiplier, bias and grad_bias; the
 * MegEngine large-kernel depthwise article, "From convolution to matrix
 * multiplication", for the per-channel sliding window; the
 * DynamicConvolutionOperator README, "Solution", for branches stored straight
 * into strided slices of one concatenated output):
 *
 *   x  : [N, C, H, W]                 input, NCHW, contiguous
 *   w  : [C*m, kh, kw]                filters (PyTorch's [C*m, 1, kh, kw])
 *   b  : [C*m]                        bias, optional
 *   y  : [N, out_c_total, Ho, Wo]     output; this call owns channels
 *                                     [out_c_offset, out_c_offset + C*m)
 *   Ho = floor((H + 2*pad_h - dil_h*(kh-1) - 1) / stride_h) + 1   (same for Wo)
 *
 *   y[n, off + c*m + j, oh, ow] = b[c*m + j]
 *       + sum_{a<kh, b<kw} w[c*m + j, a, b] * x[n, c, oh*sh - ph + a*dh, ow*sw - pw + b*dw]
 *
 * Taps outside the input read zero (zero padding). This is cross-correlation
 * (no kernel flip), the convention of PyTorch's conv2d. Output channel
 * oc = c*m + j reads input channel c (PyTorch groups = C).
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns all memory, including the bwd_weight
 *    workspace. The library never allocates, frees or synchronises, and
 *    never changes the current device. Data pointers are device pointers on
 *    the current device (or managed memory).
 *  - Precision: x, w, b, y, gy, gx, gw, gb all share desc->dtype. Arithmetic
 *    is fp32 (fp16 / bf16 operands are widened exactly, products and sums are
 *    fp32); results are rounded to the storage type once, round to nearest even.
 *  - Work is enqueued on `stream` (0 = legacy default stream) and nothing
 *    waits for it. A launch failure returns DWCONV_ERR_CUDA; faults during
 *    execution surface at the caller's next synchronisation.
 *  - Graph capture: a compute call (every entry point that takes a stream;
 *    dwconv_device_timeouts is a synchronous read) enqueues only kernel
 *    launches on `stream` (no allocation, copy, memset or synchronisation,
 *    no other stream), so calls on a capturing stream are recorded into the
 *    caller's CUDA graph and give bitwise the same results on replay. Make
 *    the first call of a shape and entry point on a device outside any
 *    capture: it sets the kernels' shared-memory limits and looks up device
 *    addresses (for dwconv2d_bwd_weight_noalloc this is required, see
 *    below).
 *  - Errors: arguments are checked on the host before any launch; on any
 *    error nothing is enqueued and nothing is written. Nothing prints or aborts.
 *  - Alignment: each pointer must be aligned to its element size
 *    (DWCONV_ERR_MISALIGNED otherwise); wider alignment is used when present.
 *  - Determinism: every entry point gives bitwise identical results on
 *    repeated calls with the same inputs on the same GPU.
 *  - Thread safety: calls may come from any thread. The library keeps
 *    three pieces of global state: the device counter of bounded waits that
 *    gave up (dwconv_device_timeouts), the per-device address cache of
 *    dwconv2d_bwd_weight_noalloc (guarded by a mutex), and that entry
 *    point's fixed scratch array, which all its calls share: calls of
 *    dwconv2d_bwd_weight_noalloc that can overlap on the GPU must be
 *    serialised by the caller. Every other entry point touches only the
 *    memory its arguments name.
 *  - Empty batch (N == 0) is valid and enqueues nothing.
 */
#ifndef DWCONV_H_
#define DWCONV_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DWCONV_F32 = 0,
  DWCONV_F16 = 1,
  DWCONV_BF16 = 2
} dwconv_dtype_t;

/* Activation of the fused forward epilogue (dwconv2d_fwd_epilogue). */
typedef enum {
  DWCONV_ACT_NONE = 0,
  DWCONV_ACT_RELU = 1,   /* max(v, 0) */
  DWCONV_ACT_RELU6 = 2   /* min(max(v, 0), 6) */
} dwconv_act_t;

typedef enum {
  DWCONV_OK = 0,
  DWCONV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, Ho or Wo < 1, slice out of range */
  DWCONV_ERR_UNSUPPORTED = 2,   /* unknown dtype, kernel larger than 255, ... */
  DWCONV_ERR_MISALIGNED = 3,    /* pointer not aligned to its element size */
  DWCONV_ERR_WORKSPACE = 4,     /* bwd_weight workspace missing or too small */
  DWCONV_ERR_CUDA = 5           /* a CUDA runtime call or launch failed */
} dwconv_status_t;

/* One depthwise convolution. 88 bytes, no padding holes. */
typedef struct {
  int64_t N, C, H, W;          /* input NCHW; N >= 0, C, H, W >= 1 */
  int32_t multiplier;          /* m >= 1: output channel c*m + j reads input channel c */
  int32_t kh, kw;              /* 1 .. 255 */
  int32_t stride_h, stride_w;  /* >= 1 */
  int32_t pad_h, pad_w;        /* >= 0, zero padding on both sides */
  int32_t dil_h, dil_w;        /* >= 1 */
  int32_t dtype;               /* dwconv_dtype_t */
  int64_t out_c_offset;        /* first channel of this op's slice in y / gy (>= 0) */
  int64_t out_c_total;         /* channel count of the y / gy buffer; 0 means C*m */
} dwconv2d_desc_t;

/* Output spatial size. Returns DWCONV_ERR_INVALID_ARG if the descriptor is
 * invalid (Ho or Wo would be < 1, slice out of range, ...). */
dwconv_status_t dwconv2d_output_shape(const dwconv2d_desc_t* desc, int64_t* Ho, int64_t* Wo);

/* Forward (#3057 forward kernel; the bias of its "add bias for forward"
 * commit). Writes only channels [off, off + C*m) of y; the other channels of
 * y are left bit-identical. bias may be NULL. */
dwconv_status_t dwconv2d_fwd(const dwconv2d_desc_t* desc, const void* x, const void* w,
                             const void* bias, void* y, cudaStream_t stream);

/* Gradient with respect to the input (#3057 grad-input kernel): the adjoint
 * of dwconv2d_fwd in x,
 *   gx[n, c, ih, iw] = sum_j sum_{a, b} w[c*m+j, a, b] * gy[n, off+c*m+j, oh, ow]
 * over the (oh, ow, a, b) with oh*sh - ph + a*dh == ih and
 * ow*sw - pw + b*dw == iw. gy is read from the same channel slice that the
 * forward wrote. accumulate = 0 overwrites gx, 1 adds to it (gx += ...). */
dwconv_status_t dwconv2d_bwd_data(const dwconv2d_desc_t* desc, const void* gy, const void* w,
                                  void* gx, int accumulate, cudaStream_t stream);

/* Bytes of device workspace dwconv2d_bwd_weight needs for this descriptor
 * (0 if the descriptor is invalid). Depends only on the descriptor. */
size_t dwconv2d_bwd_weight_workspace_size(const dwconv2d_desc_t* desc);

/* Gradients with respect to the filters and bias (#3057 grad-weight kernel,
 * extended there to padding, stride and dilation; grad_bias from its
 * output_mask):
 *   gw[oc, a, b] = sum_{n, oh, ow} gy[n, off+oc, oh, ow] * x[n, oc/m, oh*sh-ph+a*dh, ow*sw-pw+b*dw]
 *   gb[oc]       = sum_{n, oh, ow} gy[n, off+oc, oh, ow]
 * gw and gbias are overwritten; either may be NULL (then it is not computed).
 * Two launches: per-chunk fp32 partial sums into `workspace`, then a sum of
 * the chunks in index order, so the result is bitwise reproducible.
 * workspace_bytes must be >= dwconv2d_bwd_weight_workspace_size(desc); the
 * workspace must be 16-byte aligned and must not be used concurrently. */
dwconv_status_t dwconv2d_bwd_weight(const dwconv2d_desc_t* desc, const void* x, const void* gy,
                                    void* gw, void* gbias, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream);

/* Weight and bias gradients without a caller-provided workspace.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory when they need the gradient -- for
 * example code inside a host application that owns every device allocation
 * through its own pool, or a latency-critical loop where a cudaMalloc (which
 * may synchronise the device) is not acceptable.
 * Same arguments, results and errors as dwconv2d_bwd_weight minus the
 * workspace: the partial sums go to a fixed 8 MiB (8388608-byte) array that
 * is part of the library's device code, so every GPU that loads the library
 * holds those 8 MiB until the process exits. Descriptors whose
 * dwconv2d_bwd_weight_workspace_size exceeds 8 MiB are rejected with
 * DWCONV_ERR_WORKSPACE and nothing is enqueued. The call allocates and frees
 * nothing. The first call on each device (with that device current) looks up
 * the array's device address and keeps it for later calls (a failed lookup
 * returns DWCONV_ERR_CUDA and is retried by the next call); make that first
 * call before any stream capture. All calls share the one array and each
 * call's first pass overwrites every slot its second pass reads, so stale
 * contents from an earlier call do no harm -- but calls that may run at the
 * same time on the GPU (different streams, or different host threads) race
 * on the array and must be serialised by the caller. */
dwconv_status_t dwconv2d_bwd_weight_noalloc(const dwconv2d_desc_t* desc, const void* x,
                                            const void* gy, void* gw, void* gbias,
                                            cudaStream_t stream);

/* Forward with a fused epilogue: y = act(scale[oc] * (conv + bias[oc]) +
 * shift[oc]) for every output channel oc of the descriptor, computed in fp32
 * and rounded once to the storage type. With scale = gamma / sqrt(var + eps)
 * and shift = beta - mean * scale it is a convolution followed by an
 * inference batch norm and an activation in one pass over y. (Source: the
 * Megvii article "黑科技：用cutlass进行低成本、高性能卷积算子定制开发"
 * (custom convolution operators with cutlass), its opening list of what the
 * basic operator libraries lack: a user cannot add a new activation to
 * their convolution.)
 * scale and shift are C*m values of desc->dtype (either may be NULL: 1 / 0);
 * act is a dwconv_act_t (DWCONV_ERR_INVALID_ARG otherwise). Same arguments,
 * layouts, slices and errors as dwconv2d_fwd otherwise; with NULL scale and
 * shift and DWCONV_ACT_NONE it is dwconv2d_fwd. The small-plane and
 * tensor-core forward kernels have no epilogue, so shapes they would serve
 * run on the tile, direct or generic kernels here. */
dwconv_status_t dwconv2d_fwd_epilogue(const dwconv2d_desc_t* desc, const void* x, const void* w,
                                      const void* bias, const void* scale, const void* shift,
                                      int act, void* y, cudaStream_t stream);

/* Channels-last forward: the same operation and descriptor as dwconv2d_fwd
 * with the channel axis innermost,
 *   x : [N, H, W, C]               input, contiguous
 *   w : [C*m, kh, kw]              filters, as dwconv2d_fwd
 *   y : [N, Ho, Wo, out_c_total]   output; this call writes channels
 *                                  [out_c_offset, out_c_offset + C*m) of
 *                                  every pixel and nothing else
 * with the fused epilogue of dwconv2d_fwd_epilogue (scale / shift / act;
 * NULL, NULL, DWCONV_ACT_NONE for none). The layout is PyTorch's
 * channels_last memory format. (The pages' kernels are NCHW; this variant
 * is this library's, for callers whose tensors are channels-last, so that
 * they need no transpose.) Same errors as dwconv2d_fwd_epilogue. 3x3, 5x5
 * and 7x7 filters with equal strides of 1 or 2, dilation 1, one filter per
 * channel and C * element size a multiple of 16 bytes run on a tiled
 * kernel that stages input boxes with the tensor memory accelerator (x must
 * then be 16-byte aligned, else the generic kernel runs); every other shape
 * runs on a one-output-per-thread kernel. */
dwconv_status_t dwconv2d_fwd_nhwc(const dwconv2d_desc_t* desc, const void* x, const void* w,
                                  const void* bias, const void* scale, const void* shift, int act,
                                  void* y, cudaStream_t stream);

/* Depthwise-separable block, channels-last: the depthwise layer of desc,
 * its epilogue, then a 1x1 (pointwise) convolution to cout channels and its
 * epilogue, in one call:
 *   z[n, h, w, k]  = dw_act(dw_scale[k] * dwconv(x)[n, h, w, k] + dw_shift[k])
 *                    for the k < C*m depthwise channels (no bias: fold it
 *                    into dw_shift), rounded to desc->dtype
 *   y[n, h, w, off + o] = pw_act(pw_scale[o] * sum_k w_pw[o, k] z[n, h, w, k]
 *                                + pw_shift[o])       for o < cout
 * with fp32 accumulation in both stages. x [N, H, W, C] and y [N, Ho, Wo,
 * out_c_total] are channels-last; w_dw [C*m, kh, kw]; w_pw [cout, C*m]
 * (PyTorch's [cout, C*m, 1, 1]); dw_scale / dw_shift have C*m values,
 * pw_scale / pw_shift cout values, each NULL for 1 / 0; the acts are
 * dwconv_act_t values. desc->out_c_offset / out_c_total describe y's channel
 * axis (0 / 0: y has exactly cout channels); z never reaches memory.
 * (Source: the MobileNet table of "Spatial Depthwise Convolution on the GPU
 * #3057", which times each depthwise layer with the 1x1 layer after it.)
 * fp16 / bf16 blocks with a 3x3 or 5x5 filter, equal strides of 1 or 2,
 * dilation 1, one filter per channel and C a multiple of 64 (x and w_pw
 * 16-byte aligned) run the pointwise step on the tensor cores; every other
 * block runs on a generic kernel (DWCONV_ERR_UNSUPPORTED when C*m fp32
 * values of one pixel exceed 96 KB). Errors as dwconv2d_fwd_epilogue;
 * cout < 1 or a y slice past out_c_total is DWCONV_ERR_INVALID_ARG. */
dwconv_status_t dwconv2d_separable_nhwc(const dwconv2d_desc_t* desc, const void* x, const void* w_dw,
                                        const void* dw_scale, const void* dw_shift, int dw_act, int64_t cout,
                                        const void* w_pw, const void* pw_scale, const void* pw_shift,
                                        int pw_act, void* y, cudaStream_t stream);

/* Filter cache for repeated large-kernel calls with a fixed filter
 * (inference; or the forward and grad-input of one training step). Source:
 * the MegEngine large-kernel depthwise article, section on the
 * implicit-batched-GEMM algorithm: each channel's convolution is a GEMM
 * whose A operand is the im2col of the filter,
 *   T_c[oh*W + ow, ih*W + iw] = w_c[ih - oh + ph][iw - ow + pw]  (0 off the filter)
 * and, when shapes stay fixed between calls, that filter-side im2col can be
 * prepared ahead of the calls instead of inside each one.
 *
 * A cached form exists for fp16 / bf16 descriptors with stride 1, dilation
 * 1, one filter per channel, pad_h <= kh - 1, pad_w <= kw - 1 and, for the
 * pass's correlation, equal input and output row widths W that divide 64
 * (8, 16, 32 or 64; for both passes: Wo == W, i.e. 2 * pad_w == kw - 1),
 * when one channel's expanded filter fits in shared memory beside the
 * kernel's input stages: C x NS x W x 128 bytes in all, NS = the number of
 * filter-row offsets a 128-position tile meets (38 for 31x31 at W = 32; at
 * W = 64 filters up to 21 rows have a cached form, 27 and 31 do not).
 * Pass 0 caches the forward's filter, pass 1 the grad-input's (the filter
 * rotated by 180 degrees); each pass needs its own cache.
 *
 * dwconv2d_filter_cache_size: bytes of the cache (0 when the descriptor is
 * invalid, pass is not 0 or 1, or the shape has no cached form). It depends
 * on C, W, the kernel size, the padding and the dtype -- not on N or H, so
 * one cache serves every batch and height of that layer.
 *
 * dwconv2d_filter_cache_build: expands w ([C, kh, kw], desc->dtype) into
 * `cache` (caller-owned device memory, 16-byte aligned, cache_bytes >= the
 * size above); one launch on `stream`, nothing else written. Build again
 * whenever w changes.
 *
 * dwconv2d_fwd_cached / dwconv2d_bwd_data_cached: the results of
 * dwconv2d_fwd / dwconv2d_bwd_data (same arguments, slices, accumulate
 * flag and rounding), with the filter taken from a cache that
 * dwconv2d_filter_cache_build made for the same pass from a descriptor that
 * agrees in C, W, kh, kw, pad_h, pad_w and dtype (the library cannot check
 * the cache's contents; another cache gives wrong results, not an error).
 * x (resp. gy) must be 16-byte aligned.
 *
 * Errors: DWCONV_ERR_UNSUPPORTED when the shape has no cached form;
 * DWCONV_ERR_WORKSPACE when cache is NULL or cache_bytes is too small;
 * DWCONV_ERR_MISALIGNED for a cache or x / gy not 16-byte aligned (other
 * pointers: their element size); DWCONV_ERR_INVALID_ARG for pass not 0 or 1
 * and as dwconv2d_fwd / dwconv2d_bwd_data otherwise. An empty batch
 * (N == 0) enqueues nothing. */
size_t dwconv2d_filter_cache_size(const dwconv2d_desc_t* desc, int pass);
dwconv_status_t dwconv2d_filter_cache_build(const dwconv2d_desc_t* desc, int pass, const void* w,
                                            void* cache, size_t cache_bytes, cudaStream_t stream);
dwconv_status_t dwconv2d_fwd_cached(const dwconv2d_desc_t* desc, const void* x, const void* cache,
                                    size_t cache_bytes, const void* bias, void* y, cudaStream_t stream);
dwconv_status_t dwconv2d_bwd_data_cached(const dwconv2d_desc_t* desc, const void* gy, const void* cache,
                                         size_t cache_bytes, void* gx, int accumulate,
                                         cudaStream_t stream);

/* Fused multi-branch forward (the DynamicConvolutionOperator's single launch
 * for dilation 1, 3, 5 whose results are stored straight into slices of one
 * concatenated tensor): nbranch (1..8) descriptors over the same x. All
 * branches must share N, C, H, W, multiplier, dtype and out_c_total, and give
 * equal Ho, Wo; each has its own kernel size, stride, padding, dilation and
 * out_c_offset. Slices must not overlap. w[i] and bias[i] (bias or bias[i]
 * may be NULL) belong to branch i. For 2 or 3 branches of 3x3 filters at
 * stride 1, m = 1 and dilation sets {1,3,5}, {1,2,3}, {1,2}, {1,3} one launch
 * reads each x tile once and writes every branch; other sets run one launch
 * per branch (see dwconv2d_multi_plan_name). */
dwconv_status_t dwconv2d_fwd_multi(int nbranch, const dwconv2d_desc_t* descs, const void* x,
                                   const void* const* w, const void* const* bias, void* y,
                                   cudaStream_t stream);

/* Input gradient of dwconv2d_fwd_multi: gx = sum over branches of each
 * branch's dwconv2d_bwd_data (the chain rule through the concatenation),
 * accumulated in fp32 in one launch and rounded once (gx is overwritten). */
dwconv_status_t dwconv2d_bwd_data_multi(int nbranch, const dwconv2d_desc_t* descs, const void* gy,
                                        const void* const* w, void* gx, cudaStream_t stream);

/* Static text for a status code. */
const char* dwconv_status_string(dwconv_status_t status);

/* Name of the kernel family the planner picks for a pass (0 = fwd,
 * 1 = bwd_data, 2 = bwd_weight, 3 = dwconv2d_fwd_epilogue with a scale, a
 * shift or an activation, 4 = dwconv2d_fwd_nhwc) of this descriptor: "nhwc"
 * (the tiled channels-last forward), "plane" (3x3 on small
 * planes, one warp per group of whole planes), "tile" (small filters),
 * "large" (large-filter direct convolution), "ibgemm" (large-filter fp16 /
 * bf16 forward and grad-input as an implicit batched GEMM on the tensor
 * cores), "tcwgrad" (large-filter fp16 / bf16 weight gradient on the tensor
 * cores), "generic" (any shape) or "invalid". Host only; for logs and tests.
 * An "ibgemm" pass whose input pointer (a "tcwgrad" pass whose x or grad_out
 * pointer) is not 16-byte aligned runs on the direct kernels instead. */
const char* dwconv2d_plan_name(const dwconv2d_desc_t* desc, int pass);

/* Kernel family of dwconv2d_separable_nhwc for this block: "septc" (the
 * fused tensor-core kernel), "generic" or "invalid". Host only. */
const char* dwconv2d_separable_plan_name(const dwconv2d_desc_t* desc, int64_t cout);

/* Kernel family used by dwconv2d_fwd_multi / dwconv2d_bwd_data_multi for
 * these branches ("tile" = the fused single-launch kernels, "generic" = the
 * any-shape fallback: one launch per branch for the forward, one launch for
 * the grad-input), or "invalid". Host only. */
const char* dwconv2d_multi_plan_name(int nbranch, const dwconv2d_desc_t* descs);

/* Health check: the number of bounded waits in the library's kernels that
 * gave up since the library was loaded on the current device (0 in a healthy
 * run). Tile copies that use the tensor memory accelerator are waited for
 * with an iteration limit; a wait that runs out increments this counter and
 * the kernel stops early instead of hanging, leaving its outputs incomplete.
 * Synchronous: copies the counter to *count. */
dwconv_status_t dwconv_device_timeouts(unsigned int* count);

/* Health-check helper, not part of the convolution: exercises the give-up
 * path of the library's bounded waits. One CTA waits, at most `polls`
 * (1..65536) polls, on a shared-memory barrier that nothing will ever
 * complete -- no copy or tensor-core operation targets it, so nothing is in
 * flight -- gives up, adds one to the counter that dwconv_device_timeouts
 * reads, and returns. After the kernel has run, that counter is larger by
 * exactly one. Asynchronous like the other entry points;
 * DWCONV_ERR_INVALID_ARG for `polls` out of range. */
dwconv_status_t dwconv_wait_selftest(unsigned int polls, cudaStream_t stream);

/* Measurement helper, not part of the convolution: runs a register-only
 * fp32 FMA loop on every SM (`blocks` x 256 threads, `iters` iterations of 16
 * independent FMA chains) and writes one float per thread to `sink`
 * (blocks * 256 floats) so the work cannot be elided. Time it with events to
 * get the device's fp32 FMA rate: 2 * 16 * iters * blocks * 256 FLOP. */
dwconv_status_t dwconv_fma_probe(int blocks, int iters, float* sink, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DWCONV_H_ */
