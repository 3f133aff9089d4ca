"""Depthwise 2-D convolution oracle (fp64, plain CPU nested loops).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers. The product path never imports this
package, and this package never imports the product. It shares no code with
the CUDA library.

The arithmetic lives in ``dwconv_oracle.c`` (direct nested loops over the
definition of forward, bwd_data and bwd_weight, the per-channel epilogue of
the fused forward, and the pointwise 1x1 step of a depthwise-separable
block). This module only compiles it
with gcc, marshals numpy float64 arrays to it, and expresses the fused
multi-branch calls the way the DynamicConvolutionOperator README describes
them ("Solution": one output per dilation branch, each stored into its own
slice of one concatenated tensor): one single-branch call per branch, and, for
the input gradient, the sum of the per-branch gradients (the chain rule through
the concatenation).

Parity status: every function here is pinned by tests/test_oracle_pins.py
(brute force by impulse scattering, shifted-input delta kernels, box sums,
separable kernels, adjoint identities, finite differences, a float64 library
cross-check). No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dwconv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "N", "C", "H", "W", "m", "kh", "kw", "sh", "sw", "ph", "pw", "dh", "dw",
        "off", "c_total")]


@dataclass
class Conv:
    """Shape and hyper-parameters of one depthwise convolution.

    x: [N, C, H, W]; w: [C*m, kh, kw]; bias: [C*m];
    y / gy: [N, c_total, Ho, Wo] with this op's channels at [off, off + C*m).
    """
    N: int
    C: int
    H: int
    W: int
    kh: int = 3
    kw: int = 3
    sh: int = 1
    sw: int = 1
    ph: int = 0
    pw: int = 0
    dh: int = 1
    dw: int = 1
    m: int = 1
    off: int = 0
    c_total: int | None = None

    @property
    def OC(self) -> int:
        return self.C * self.m

    @property
    def Ctot(self) -> int:
        return self.OC if self.c_total is None else self.c_total

    @property
    def Ho(self) -> int:
        span = self.H + 2 * self.ph - self.dh * (self.kh - 1) - 1
        return span // self.sh + 1 if span >= 0 else 0

    @property
    def Wo(self) -> int:
        span = self.W + 2 * self.pw - self.dw * (self.kw - 1) - 1
        return span // self.sw + 1 if span >= 0 else 0

    def _c(self) -> _Desc:
        return _Desc(self.N, self.C, self.H, self.W, self.m, self.kh, self.kw,
                     self.sh, self.sw, self.ph, self.pw, self.dh, self.dw,
                     self.off, self.Ctot)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC]
        try:
            subprocess.run(base[:2] + ["-fopenmp"] + base[2:], check=True,
                           capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base, check=True, capture_output=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        # DWCONV_ORACLE_LIB points at a deliberately broken copy of the oracle
        # (tests/test_oracle_mutants.py) to show that the pins catch it.
        path = os.environ.get("DWCONV_ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(_Desc)
        dp = ctypes.c_void_p
        lib.oracle_dwconv2d_fwd.argtypes = [P, dp, dp, dp, dp]
        lib.oracle_dwconv2d_bwd_data.argtypes = [P, dp, dp, dp]
        lib.oracle_dwconv2d_bwd_weight.argtypes = [P, dp, dp, dp, dp]
        lib.oracle_epilogue.argtypes = [P, dp, dp, ctypes.c_int, dp]
        i64 = ctypes.c_int64
        lib.oracle_pointwise.argtypes = [i64, i64, i64, i64, dp, dp, dp]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a, shape):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if tuple(a.shape) != tuple(shape):
        a = a.reshape(shape)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def fwd(cv: Conv, x, w, bias=None, y=None):
    """Forward. Writes channels [off, off+C*m) of y (allocated as zeros if None)."""
    lib = _load()
    x = _f64(x, (cv.N, cv.C, cv.H, cv.W))
    w = _f64(w, (cv.OC, cv.kh, cv.kw))
    b = None if bias is None else _f64(bias, (cv.OC,))
    if y is None:
        y = np.zeros((cv.N, cv.Ctot, cv.Ho, cv.Wo), dtype=np.float64)
    assert y.dtype == np.float64 and y.flags.c_contiguous
    assert y.shape == (cv.N, cv.Ctot, cv.Ho, cv.Wo)
    d = cv._c()
    lib.oracle_dwconv2d_fwd(ctypes.byref(d), _ptr(x), _ptr(w), _ptr(b), _ptr(y))
    return y


ACTS = {"none": 0, "relu": 1, "relu6": 2}


def fwd_epilogue(cv: Conv, x, w, bias=None, scale=None, shift=None, act="none", y=None):
    """Forward, then y = act(scale[oc] * y + shift[oc]) on this op's channels.

    ``act`` is "none", "relu" (max(v, 0)) or "relu6" (min(max(v, 0), 6));
    scale / shift of None mean 1 / 0.
    """
    y = fwd(cv, x, w, bias, y)
    sc = None if scale is None else _f64(scale, (cv.OC,))
    sh = None if shift is None else _f64(shift, (cv.OC,))
    d = cv._c()
    _load().oracle_epilogue(ctypes.byref(d), _ptr(sc), _ptr(sh), ACTS[act], _ptr(y))
    return y


def separable(cv: Conv, x, w_dw, dw_scale=None, dw_shift=None, dw_act="none", w_pw=None,
              pw_scale=None, pw_shift=None, pw_act="none"):
    """Depthwise-separable block: z = act1(scale1 * dwconv(x) + shift1) over
    all C*m depthwise channels, then y = act2(scale2 * (w_pw @ z) + shift2)
    with w_pw [cout, C*m]. Returns y [N, cout, Ho, Wo] (cv's slice fields
    are ignored: z is the full C*m channels)."""
    lib = _load()
    dcv = Conv(N=cv.N, C=cv.C, H=cv.H, W=cv.W, kh=cv.kh, kw=cv.kw, sh=cv.sh, sw=cv.sw, ph=cv.ph, pw=cv.pw,
               dh=cv.dh, dw=cv.dw, m=cv.m)
    z = fwd_epilogue(dcv, x, w_dw, None, dw_scale, dw_shift, dw_act)
    cin = dcv.OC
    wp = np.ascontiguousarray(np.asarray(w_pw, dtype=np.float64))
    cout = wp.shape[0]
    assert wp.shape == (cout, cin)
    hw = dcv.Ho * dcv.Wo
    y = np.empty((cv.N, cout, dcv.Ho, dcv.Wo), dtype=np.float64)
    lib.oracle_pointwise(cv.N, cin, cout, hw, _ptr(z), _ptr(wp), _ptr(y))
    pcv = Conv(N=cv.N, C=cout, H=dcv.Ho, W=dcv.Wo, kh=1, kw=1)
    sc = None if pw_scale is None else _f64(pw_scale, (cout,))
    sh = None if pw_shift is None else _f64(pw_shift, (cout,))
    pd = pcv._c()
    lib.oracle_epilogue(ctypes.byref(pd), _ptr(sc), _ptr(sh), ACTS[pw_act], _ptr(y))
    return y


def bwd_data(cv: Conv, gy, w):
    """Gradient with respect to x, read from channels [off, off+C*m) of gy."""
    lib = _load()
    gy = _f64(gy, (cv.N, cv.Ctot, cv.Ho, cv.Wo))
    w = _f64(w, (cv.OC, cv.kh, cv.kw))
    gx = np.empty((cv.N, cv.C, cv.H, cv.W), dtype=np.float64)
    d = cv._c()
    lib.oracle_dwconv2d_bwd_data(ctypes.byref(d), _ptr(gy), _ptr(w), _ptr(gx))
    return gx


def bwd_weight(cv: Conv, x, gy, want_w: bool = True, want_b: bool = False):
    """Gradients with respect to w ([C*m, kh, kw]) and bias ([C*m])."""
    lib = _load()
    x = _f64(x, (cv.N, cv.C, cv.H, cv.W))
    gy = _f64(gy, (cv.N, cv.Ctot, cv.Ho, cv.Wo))
    gw = np.empty((cv.OC, cv.kh, cv.kw), dtype=np.float64) if want_w else None
    gb = np.empty((cv.OC,), dtype=np.float64) if want_b else None
    d = cv._c()
    lib.oracle_dwconv2d_bwd_weight(ctypes.byref(d), _ptr(x), _ptr(gy), _ptr(gw), _ptr(gb))
    return gw, gb


def fwd_multi(branches, x, ws, biases=None):
    """Several branches over one x, each writing its own channel slice of one y.

    All branches must share N, C, H, W and c_total and give equal Ho, Wo.
    """
    cv0 = branches[0]
    y = np.zeros((cv0.N, cv0.Ctot, cv0.Ho, cv0.Wo), dtype=np.float64)
    for i, cv in enumerate(branches):
        assert (cv.N, cv.C, cv.H, cv.W, cv.Ctot, cv.Ho, cv.Wo) == (
            cv0.N, cv0.C, cv0.H, cv0.W, cv0.Ctot, cv0.Ho, cv0.Wo)
        fwd(cv, x, ws[i], None if biases is None else biases[i], y=y)
    return y


def bwd_data_multi(branches, gy, ws):
    """Input gradient of fwd_multi: the sum of each branch's input gradient."""
    gx = None
    for i, cv in enumerate(branches):
        g = bwd_data(cv, gy, ws[i])
        gx = g if gx is None else gx + g
    return gx
