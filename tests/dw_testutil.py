"""Helpers for the GPU parity tests: move synthetic tensors to the device,
call libdwconv through its C ABI binding, bring results back as float64, and
compare them with the oracle under the stated tolerances."""
from __future__ import annotations

import math

import numpy as np

import oracle
from depthwise_convolution_dwconv2d_gb300 import binding as B
from depthwise_convolution_dwconv2d_gb300 import synth
from oracle import Conv


def torch():
    import torch as _t
    return _t


TORCH_DT = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}


def to_dev(t: synth.Tensor):
    th = torch()
    if t.dtype == "bf16":
        return th.from_numpy(t.store.view(np.int16).copy()).view(th.bfloat16).cuda()
    return th.from_numpy(np.ascontiguousarray(t.store)).cuda()


def empty_dev(shape, dtype, fill=None):
    th = torch()
    out = th.empty(tuple(shape), dtype=getattr(th, TORCH_DT[dtype]), device="cuda")
    if fill is not None:
        out.fill_(fill)
    return out


def to_f64(tt) -> np.ndarray:
    th = torch()
    tt = tt.detach().cpu()
    if tt.dtype == th.bfloat16:
        return synth.bf16_bits_to_f64(tt.view(th.int16).numpy().view(np.uint16))
    return tt.to(th.float64).numpy()


def oconv(L, off=0, c_total=None, N=None, C=None) -> Conv:
    return Conv(N=L.N if N is None else N, C=L.C if C is None else C, H=L.H, W=L.W, kh=L.k, kw=L.k,
                sh=L.s, sw=L.s, ph=L.p, pw=L.p, dh=L.d, dw=L.d, m=L.m, off=off, c_total=c_total)


def tol_ok(got: np.ndarray, ref: np.ndarray, dtype: str, taps: int):
    """fp32: normwise max|g - r| / max|r| <= 1e-5 sqrt(taps);
    fp16/bf16: elementwise |g - r| <= 1e-2 + 2e-2 |r|. Returns (ok, measure)."""
    if got.shape != ref.shape:
        return False, f"shape {got.shape} != {ref.shape}"
    if got.size == 0:
        return True, 0.0
    if not np.all(np.isfinite(got)):
        return False, "non-finite output"
    if dtype == "f32":
        scale = max(np.max(np.abs(ref)), 1e-30)
        err = float(np.max(np.abs(got - ref)) / scale)
        return err <= 1e-5 * math.sqrt(taps), err
    excess = np.abs(got - ref) - (1e-2 + 2e-2 * np.abs(ref))
    worst = float(np.max(excess))
    return worst <= 0.0, worst


def assert_close(got, ref, dtype, taps, what=""):
    ok, m = tol_ok(got, ref, dtype, taps)
    assert ok, f"{what}: tolerance exceeded ({m})"


def ws_for(desc):
    th = torch()
    nbytes = B.dwconv2d_bwd_weight_workspace_size(desc)
    return th.empty(max(nbytes, 16) // 4 + 4, dtype=th.float32, device="cuda"), nbytes
