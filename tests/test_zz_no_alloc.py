"""The scratch-free weight-gradient entry point (dwconv2d_bwd_weight_noalloc).

It serves callers that cannot allocate device memory when they need the
gradient (a host application that owns all device allocations, or a loop
that cannot afford a cudaMalloc). It runs the same kernels as
dwconv2d_bwd_weight with a caller-provided workspace, so on consecutive
calls that share its fixed device array its gradients must equal that entry
point's bit for bit, and match the fp64 oracle within the parity tolerance.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

import oracle
from depthwise_convolution_dwconv2d_gb300 import binding as B
from depthwise_convolution_dwconv2d_gb300 import workloads as WL
from dw_testutil import assert_close, empty_dev, oconv, to_dev, to_f64, torch, ws_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    th = pytest.importorskip("torch")
    if not th.cuda.is_available():
        pytest.skip("no CUDA device")
    from depthwise_convolution_dwconv2d_gb300 import build
    build.build()
    B.load()


def grads(L, use_noalloc):
    th = torch()
    inp = WL.make_inputs(L)
    d = B.make_desc(**L.desc_kwargs())
    x, gy = to_dev(inp.x), to_dev(inp.gy)
    gw = empty_dev((L.OC, L.k, L.k), L.dtype, fill=9.0)
    gb = empty_dev((L.OC,), L.dtype, fill=9.0) if L.bias else None
    if use_noalloc:
        B.dwconv2d_bwd_weight_noalloc(d, x, gy, gw, gb)
    else:
        ws, nbytes = ws_for(d)
        B.dwconv2d_bwd_weight(d, x, gy, gw, gb, ws, nbytes)
    th.cuda.synchronize()
    return to_f64(gw), (to_f64(gb) if gb is not None else None)


# two different calls in a row: the second must not see the first's leftovers
CALLS = [WL.Layer(N=8, C=64, H=56, W=56, k=3, s=1, p=1, name="mb56"),
         WL.Layer(N=4, C=32, H=28, W=28, k=5, s=1, p=2, m=2, bias=True, dtype="bf16",
                  x_dist="normal", w_std=0.2, name="mult_bf16")]


def check_against_workspace_call_and_oracle(L, label):
    ref_w, ref_b = grads(L, use_noalloc=False)
    got_w, got_b = grads(L, use_noalloc=True)
    # the same kernels and the same summation order: bitwise equal
    assert np.array_equal(got_w, ref_w), f"{label} gw differs from the workspace entry point"
    if L.bias:
        assert np.array_equal(got_b, ref_b), f"{label} gb differs from the workspace entry point"
    inp = WL.make_inputs(L)
    rgw, rgb = oracle.bwd_weight(oconv(L), inp.x.f64, inp.gy.f64, want_w=True, want_b=L.bias)
    assert_close(got_w, rgw, L.dtype, L.k * L.k, f"{label} gw vs oracle")
    if L.bias:
        assert_close(got_b, rgb, L.dtype, 1, f"{label} gb vs oracle")


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    for L in CALLS:
        check_against_workspace_call_and_oracle(L, L.name)
    # and once more on the first shape, after the second call reused the array
    check_against_workspace_call_and_oracle(CALLS[0], "repeat")


def test_noalloc_rejects_descriptors_beyond_the_array():
    # 64 channels x (255*255 + 1) taps x 4 B per chunk is far above 8 MiB
    d = B.make_desc(1, 64, 300, 300, 255, 1, 127)
    assert B.dwconv2d_bwd_weight_workspace_size(d) > (8 << 20)
    P = 0x10000
    with pytest.raises(B.DwconvError) as e:
        B.dwconv2d_bwd_weight_noalloc(d, P, P, P, None, 0)
    assert e.value.status == 4  # DWCONV_ERR_WORKSPACE
