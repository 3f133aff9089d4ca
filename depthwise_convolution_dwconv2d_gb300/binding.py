"""Thin ctypes binding over libdwconv's C ABI (argument marshalling only).

Each function has the C entry point's name and argument order. Tensor
arguments may be torch tensors (their device pointer is passed; they must be
contiguous) or raw integer addresses. ``stream`` defaults to PyTorch's current
CUDA stream. Every computation happens in libdwconv's CUDA kernels: there is
no fallback, and a missing library raises at the first call.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
ESIZE = {"f32": 4, "f16": 2, "bf16": 2}

STATUS = {0: "DWCONV_OK", 1: "DWCONV_ERR_INVALID_ARG", 2: "DWCONV_ERR_UNSUPPORTED",
          3: "DWCONV_ERR_MISALIGNED", 4: "DWCONV_ERR_WORKSPACE", 5: "DWCONV_ERR_CUDA"}

# every symbol include/dwconv.h declares
SYMBOLS = ("dwconv2d_output_shape", "dwconv2d_fwd", "dwconv2d_bwd_data",
           "dwconv2d_bwd_weight_workspace_size", "dwconv2d_bwd_weight", "dwconv2d_fwd_multi",
           "dwconv2d_bwd_data_multi", "dwconv_status_string", "dwconv2d_plan_name",
           "dwconv2d_multi_plan_name", "dwconv_fma_probe", "dwconv2d_bwd_weight_noalloc",
           "dwconv_device_timeouts", "dwconv_wait_selftest", "dwconv2d_fwd_epilogue",
           "dwconv2d_fwd_nhwc", "dwconv2d_separable_nhwc", "dwconv2d_separable_plan_name",
           "dwconv2d_filter_cache_size", "dwconv2d_filter_cache_build", "dwconv2d_fwd_cached",
           "dwconv2d_bwd_data_cached")

# dwconv_act_t
ACTS = {"none": 0, "relu": 1, "relu6": 2}


class DwconvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = load().dwconv_status_string(status).decode()
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg})")


class Desc(ctypes.Structure):
    """dwconv2d_desc_t (88 bytes)."""
    _fields_ = [("N", ctypes.c_int64), ("C", ctypes.c_int64), ("H", ctypes.c_int64),
                ("W", ctypes.c_int64), ("multiplier", ctypes.c_int32), ("kh", ctypes.c_int32),
                ("kw", ctypes.c_int32), ("stride_h", ctypes.c_int32), ("stride_w", ctypes.c_int32),
                ("pad_h", ctypes.c_int32), ("pad_w", ctypes.c_int32), ("dil_h", ctypes.c_int32),
                ("dil_w", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("out_c_offset", ctypes.c_int64), ("out_c_total", ctypes.c_int64)]


assert ctypes.sizeof(Desc) == 88


def _pair(v):
    return (v, v) if isinstance(v, int) else (int(v[0]), int(v[1]))


def make_desc(N, C, H, W, kernel=3, stride=1, pad=0, dilation=1, multiplier=1, dtype="f32",
              out_c_offset=0, out_c_total=0) -> Desc:
    kh, kw = _pair(kernel)
    sh, sw = _pair(stride)
    ph, pw = _pair(pad)
    dh, dw = _pair(dilation)
    return Desc(N, C, H, W, multiplier, kh, kw, sh, sw, ph, pw, dh, dw,
                DTYPES[dtype] if isinstance(dtype, str) else int(dtype), out_c_offset, out_c_total)


_lib = None


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libdwconv.so (built by ``build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libdwconv is not built ({path} missing); run "
                           "depthwise_convolution_dwconv2d_gb300.build.build() first")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(Desc)
    vp, st = ctypes.c_void_p, ctypes.c_int
    lib.dwconv2d_output_shape.argtypes = [P, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
    lib.dwconv2d_fwd.argtypes = [P, vp, vp, vp, vp, vp]
    lib.dwconv2d_fwd_epilogue.argtypes = [P, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp]
    lib.dwconv2d_fwd_nhwc.argtypes = [P, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp]
    lib.dwconv2d_separable_nhwc.argtypes = [P, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int64, vp, vp, vp,
                                            ctypes.c_int, vp, vp]
    lib.dwconv2d_separable_plan_name.argtypes = [P, ctypes.c_int64]
    lib.dwconv2d_separable_plan_name.restype = ctypes.c_char_p
    lib.dwconv2d_bwd_data.argtypes = [P, vp, vp, vp, ctypes.c_int, vp]
    lib.dwconv2d_bwd_weight_workspace_size.argtypes = [P]
    lib.dwconv2d_bwd_weight_workspace_size.restype = ctypes.c_size_t
    lib.dwconv2d_bwd_weight.argtypes = [P, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.dwconv2d_bwd_weight_noalloc.argtypes = [P, vp, vp, vp, vp, vp]
    lib.dwconv2d_fwd_multi.argtypes = [ctypes.c_int, P, vp, ctypes.POINTER(vp), ctypes.POINTER(vp), vp, vp]
    lib.dwconv2d_bwd_data_multi.argtypes = [ctypes.c_int, P, vp, ctypes.POINTER(vp), vp, vp]
    lib.dwconv_status_string.argtypes = [st]
    lib.dwconv_status_string.restype = ctypes.c_char_p
    lib.dwconv2d_plan_name.argtypes = [P, ctypes.c_int]
    lib.dwconv2d_plan_name.restype = ctypes.c_char_p
    lib.dwconv2d_multi_plan_name.argtypes = [ctypes.c_int, P]
    lib.dwconv2d_multi_plan_name.restype = ctypes.c_char_p
    lib.dwconv_device_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.dwconv_fma_probe.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp]
    lib.dwconv_wait_selftest.argtypes = [ctypes.c_uint, vp]
    lib.dwconv2d_filter_cache_size.argtypes = [P, ctypes.c_int]
    lib.dwconv2d_filter_cache_size.restype = ctypes.c_size_t
    lib.dwconv2d_filter_cache_build.argtypes = [P, ctypes.c_int, vp, vp, ctypes.c_size_t, vp]
    lib.dwconv2d_fwd_cached.argtypes = [P, vp, vp, ctypes.c_size_t, vp, vp, vp]
    lib.dwconv2d_bwd_data_cached.argtypes = [P, vp, vp, ctypes.c_size_t, vp, ctypes.c_int, vp]
    for name in SYMBOLS:
        if name not in ("dwconv2d_bwd_weight_workspace_size", "dwconv_status_string", "dwconv2d_plan_name",
                        "dwconv2d_multi_plan_name", "dwconv2d_separable_plan_name", "dwconv2d_filter_cache_size"):
            getattr(lib, name).restype = st
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if hasattr(t, "data_ptr"):
        if hasattr(t, "is_contiguous") and not t.is_contiguous():
            raise ValueError("libdwconv needs contiguous tensors")
        return ctypes.c_void_p(t.data_ptr())
    raise TypeError(f"cannot pass {type(t).__name__} as a device pointer")


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream) if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise DwconvError(status, where)


def dwconv2d_output_shape(desc: Desc):
    ho, wo = ctypes.c_int64(), ctypes.c_int64()
    _check(load().dwconv2d_output_shape(ctypes.byref(desc), ctypes.byref(ho), ctypes.byref(wo)),
           "dwconv2d_output_shape")
    return ho.value, wo.value


def dwconv2d_fwd(desc: Desc, x, w, bias, y, stream=None):
    _check(load().dwconv2d_fwd(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias), _ptr(y),
                               _stream(stream)), "dwconv2d_fwd")


def dwconv2d_fwd_epilogue(desc: Desc, x, w, bias, scale, shift, act, y, stream=None):
    """``act`` is a dwconv_act_t value or one of ``ACTS``' names."""
    a = ACTS[act] if isinstance(act, str) else int(act)
    _check(load().dwconv2d_fwd_epilogue(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias), _ptr(scale),
                                         _ptr(shift), a, _ptr(y), _stream(stream)),
           "dwconv2d_fwd_epilogue")


def dwconv2d_fwd_nhwc(desc: Desc, x, w, bias, y, scale=None, shift=None, act=0, stream=None):
    """x [N, H, W, C], y [N, Ho, Wo, out_c_total]; optional fused epilogue."""
    a = ACTS[act] if isinstance(act, str) else int(act)
    _check(load().dwconv2d_fwd_nhwc(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(bias), _ptr(scale),
                                     _ptr(shift), a, _ptr(y), _stream(stream)),
           "dwconv2d_fwd_nhwc")


def dwconv2d_separable_nhwc(desc: Desc, x, w_dw, cout: int, w_pw, y, dw_scale=None, dw_shift=None,
                            dw_act=0, pw_scale=None, pw_shift=None, pw_act=0, stream=None):
    """Depthwise-separable block; x [N, H, W, C], y [N, Ho, Wo, out_c_total]."""
    a1 = ACTS[dw_act] if isinstance(dw_act, str) else int(dw_act)
    a2 = ACTS[pw_act] if isinstance(pw_act, str) else int(pw_act)
    _check(load().dwconv2d_separable_nhwc(ctypes.byref(desc), _ptr(x), _ptr(w_dw), _ptr(dw_scale),
                                           _ptr(dw_shift), a1, int(cout), _ptr(w_pw), _ptr(pw_scale),
                                           _ptr(pw_shift), a2, _ptr(y), _stream(stream)),
           "dwconv2d_separable_nhwc")


def dwconv2d_separable_plan_name(desc: Desc, cout: int) -> str:
    return load().dwconv2d_separable_plan_name(ctypes.byref(desc), int(cout)).decode()


def dwconv2d_bwd_data(desc: Desc, gy, w, gx, accumulate=0, stream=None):
    _check(load().dwconv2d_bwd_data(ctypes.byref(desc), _ptr(gy), _ptr(w), _ptr(gx), int(accumulate),
                                    _stream(stream)), "dwconv2d_bwd_data")


def dwconv2d_bwd_weight_workspace_size(desc: Desc) -> int:
    return int(load().dwconv2d_bwd_weight_workspace_size(ctypes.byref(desc)))


def dwconv2d_bwd_weight(desc: Desc, x, gy, gw, gbias, workspace, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().dwconv2d_bwd_weight(ctypes.byref(desc), _ptr(x), _ptr(gy), _ptr(gw), _ptr(gbias),
                                      _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "dwconv2d_bwd_weight")


def dwconv2d_bwd_weight_noalloc(desc: Desc, x, gy, gw, gbias, stream=None):
    """dwconv2d_bwd_weight for callers that cannot allocate device memory:
    the partial sums use the library's fixed 8 MiB device array instead of a
    workspace argument (see include/dwconv.h)."""
    _check(load().dwconv2d_bwd_weight_noalloc(ctypes.byref(desc), _ptr(x), _ptr(gy), _ptr(gw),
                                              _ptr(gbias), _stream(stream)),
           "dwconv2d_bwd_weight_noalloc")


def dwconv2d_filter_cache_size(desc: Desc, pass_: int) -> int:
    """Bytes of the filter cache of pass 0 (forward) or 1 (grad-input); 0 if none."""
    return int(load().dwconv2d_filter_cache_size(ctypes.byref(desc), int(pass_)))


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def dwconv2d_filter_cache_build(desc: Desc, pass_: int, w, cache, cache_bytes=None, stream=None):
    if cache_bytes is None:
        cache_bytes = _nbytes(cache)
    _check(load().dwconv2d_filter_cache_build(ctypes.byref(desc), int(pass_), _ptr(w), _ptr(cache),
                                              int(cache_bytes), _stream(stream)),
           "dwconv2d_filter_cache_build")


def dwconv2d_fwd_cached(desc: Desc, x, cache, bias, y, cache_bytes=None, stream=None):
    if cache_bytes is None:
        cache_bytes = _nbytes(cache)
    _check(load().dwconv2d_fwd_cached(ctypes.byref(desc), _ptr(x), _ptr(cache), int(cache_bytes), _ptr(bias),
                                      _ptr(y), _stream(stream)), "dwconv2d_fwd_cached")


def dwconv2d_bwd_data_cached(desc: Desc, gy, cache, gx, accumulate=0, cache_bytes=None, stream=None):
    if cache_bytes is None:
        cache_bytes = _nbytes(cache)
    _check(load().dwconv2d_bwd_data_cached(ctypes.byref(desc), _ptr(gy), _ptr(cache), int(cache_bytes), _ptr(gx),
                                           int(accumulate), _stream(stream)), "dwconv2d_bwd_data_cached")


def _desc_array(descs):
    arr = (Desc * len(descs))(*descs)
    return arr


def _ptr_array(ts):
    if ts is None:
        return None
    return (ctypes.c_void_p * len(ts))(*[None if p is None else _ptr(p).value for p in ts])


def dwconv2d_fwd_multi(descs, x, ws, biases, y, stream=None):
    _check(load().dwconv2d_fwd_multi(len(descs), _desc_array(descs), _ptr(x), _ptr_array(ws),
                                     _ptr_array(biases), _ptr(y), _stream(stream)), "dwconv2d_fwd_multi")


def dwconv2d_bwd_data_multi(descs, gy, ws, gx, stream=None):
    _check(load().dwconv2d_bwd_data_multi(len(descs), _desc_array(descs), _ptr(gy), _ptr_array(ws),
                                          _ptr(gx), _stream(stream)), "dwconv2d_bwd_data_multi")


def dwconv_status_string(status: int) -> str:
    return load().dwconv_status_string(int(status)).decode()


def dwconv2d_plan_name(desc: Desc, pass_: int) -> str:
    return load().dwconv2d_plan_name(ctypes.byref(desc), int(pass_)).decode()


def dwconv2d_multi_plan_name(descs) -> str:
    return load().dwconv2d_multi_plan_name(len(descs), _desc_array(descs)).decode()


def dwconv_device_timeouts() -> int:
    n = ctypes.c_uint(0)
    _check(load().dwconv_device_timeouts(ctypes.byref(n)), "dwconv_device_timeouts")
    return int(n.value)


def dwconv_fma_probe(blocks: int, iters: int, sink, stream=None):
    _check(load().dwconv_fma_probe(int(blocks), int(iters), _ptr(sink), _stream(stream)), "dwconv_fma_probe")


def dwconv_wait_selftest(polls: int, stream=None):
    _check(load().dwconv_wait_selftest(int(polls), _stream(stream)), "dwconv_wait_selftest")
