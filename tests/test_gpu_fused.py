"""GPU parity of the fused forward variants against the fp64 oracle.

dwconv2d_fwd_epilogue: y = act(scale * (conv + bias) + shift) per output
channel, for every kernel family the planner can route it to (tile, large,
generic), with channel slices, ragged planes and each activation. Scale and
shift are a folded inference batch norm drawn from fixed seeds.
Tolerances as in the other parity tests: fp32 normwise max|g-r|/max|r| <=
1e-5 sqrt(taps); fp16/bf16 elementwise |g-r| <= 1e-2 + 2e-2 |r|.
"""
import numpy as np
import pytest

import oracle
from depthwise_convolution_dwconv2d_gb300 import binding as B
from depthwise_convolution_dwconv2d_gb300 import synth, workloads as WL
from dw_testutil import assert_close, empty_dev, oconv, to_dev, to_f64, torch

pytestmark = pytest.mark.gpu

# seeded streams of the batch-norm statistics (distinct from x, w, b, gy)
STREAM_GAMMA, STREAM_BETA, STREAM_MEAN, STREAM_VAR = 40, 41, 42, 43


@pytest.fixture(scope="module", autouse=True)
def _lib():
    th = pytest.importorskip("torch")
    if not th.cuda.is_available():
        pytest.skip("no CUDA device")
    from depthwise_convolution_dwconv2d_gb300 import build
    build.build()
    B.load()


def folded_bn(OC, dtype, seed=0):
    """Per-channel scale / shift of an inference batch norm, rounded to the
    storage type (the kernels and the oracle both see the rounded values)."""
    gamma = synth.normal_tensor((OC,), "f32", seed, STREAM_GAMMA, std=0.3).f64 + 1.0
    beta = synth.normal_tensor((OC,), "f32", seed, STREAM_BETA, std=0.5).f64
    mean = synth.normal_tensor((OC,), "f32", seed, STREAM_MEAN, std=0.2).f64
    var = synth.uniform_tensor((OC,), "f32", seed, STREAM_VAR, lo=0.25, hi=1.0).f64
    scale = gamma / np.sqrt(var + 1e-5)
    shift = beta - mean * scale
    return synth.Tensor(scale, (OC,), dtype), synth.Tensor(shift, (OC,), dtype)


EPI_CASES = [
    (WL.Layer(N=4, C=64, H=28, W=28, k=3, s=1, p=1, bias=True), "relu6", "tile"),
    (WL.Layer(N=2, C=32, H=57, W=57, k=3, s=2, p=1, dtype="bf16"), "relu", "tile"),
    (WL.Layer(N=3, C=24, H=20, W=19, k=5, s=1, p=2, m=2, bias=True, dtype="f16"), "none", "tile"),
    (WL.Layer(N=8, C=32, H=14, W=14, k=3, s=1, p=1), "relu", "tile"),      # small planes
    (WL.Layer(N=3, C=8, H=40, W=40, k=13, p=6, bias=True), "relu", "large"),
    (WL.Layer(N=2, C=4, H=32, W=32, k=31, p=15, dtype="f16"), "relu6", "large"),
    (WL.Layer(N=2, C=5, H=23, W=17, k=4, s=1, p=1, bias=True), "relu", "generic"),
    (WL.Layer(N=2, C=6, H=21, W=21, k=3, s=1, p=7, d=7, dtype="bf16"), "relu6", "generic"),
]
EPI_IDS = ["mb3x3_f32_relu6", "s2_bf16_relu", "m2_f16_slice", "plane_shape_f32", "k13_f32",
           "k31_f16", "k4_generic", "d7_bf16_generic"]


@pytest.mark.parametrize("L,act,family", EPI_CASES, ids=EPI_IDS)
def test_epilogue_vs_oracle(L, act, family):
    th = torch()
    off, ctot = (3, L.OC + 5) if L.m == 2 else (0, 0)
    d = B.make_desc(**L.desc_kwargs(), out_c_offset=off, out_c_total=ctot)
    assert B.dwconv2d_plan_name(d, 3) == family
    inp = WL.make_inputs(L)
    scale, shift = folded_bn(L.OC, L.dtype)
    x, w = to_dev(inp.x), to_dev(inp.w)
    b = to_dev(inp.b) if inp.b is not None else None
    y = empty_dev((L.N, ctot or L.OC, L.Ho, L.Wo), L.dtype, fill=-7.0)
    B.dwconv2d_fwd_epilogue(d, x, w, b, to_dev(scale), to_dev(shift), act, y)
    th.cuda.synchronize()
    got = to_f64(y)
    cv = oconv(L, off=off, c_total=ctot or None)
    ref = np.full(got.shape, -7.0)
    oracle.fwd_epilogue(cv, inp.x.f64, inp.w.f64, None if inp.b is None else inp.b.f64,
                        scale.f64, shift.f64, act, y=ref)
    assert_close(got, ref, L.dtype, L.k * L.k, f"{L.label()} {act}")
    if act != "none":
        s = got[:, off:off + L.OC]
        assert s.min() >= 0.0 and (act != "relu6" or s.max() <= 6.0)
    if ctot:
        assert np.all(got[:, :off] == -7.0) and np.all(got[:, off + L.OC:] == -7.0)


@pytest.mark.parametrize("L", [EPI_CASES[0][0], EPI_CASES[3][0], EPI_CASES[5][0], EPI_CASES[6][0]],
                         ids=["tile", "plane_shape", "ibgemm_shape", "generic"])
def test_epilogue_without_scale_shift_or_activation_is_plain_forward(L):
    """NULL scale and shift with no activation is dwconv2d_fwd, bit for bit,
    on whichever kernel the plain forward picks."""
    th = torch()
    d = B.make_desc(**L.desc_kwargs())
    inp = WL.make_inputs(L)
    x, w = to_dev(inp.x), to_dev(inp.w)
    b = to_dev(inp.b) if inp.b is not None else None
    y0 = empty_dev((L.N, L.OC, L.Ho, L.Wo), L.dtype)
    y1 = empty_dev((L.N, L.OC, L.Ho, L.Wo), L.dtype)
    B.dwconv2d_fwd(d, x, w, b, y0)
    B.dwconv2d_fwd_epilogue(d, x, w, b, None, None, "none", y1)
    th.cuda.synchronize()
    assert th.equal(y0, y1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_epilogue_matches_unfused_sequence(dtype):
    """The fused result equals conv -> (scale, shift) -> ReLU6 done as three
    fp32 steps in torch on the kernel's own unfused fp32 output, up to the one
    rounding the fused path saves (the check is of the index mapping of scale
    and shift, not of the arithmetic)."""
    th = torch()
    L = WL.Layer(N=2, C=48, H=33, W=30, k=3, s=1, p=1, bias=True, dtype=dtype)
    d = B.make_desc(**L.desc_kwargs())
    inp = WL.make_inputs(L)
    scale, shift = folded_bn(L.OC, dtype, seed=3)
    x, w, b = to_dev(inp.x), to_dev(inp.w), to_dev(inp.b)
    y = empty_dev((L.N, L.OC, L.Ho, L.Wo), dtype)
    B.dwconv2d_fwd_epilogue(d, x, w, b, to_dev(scale), to_dev(shift), "relu6", y)
    y0 = empty_dev((L.N, L.OC, L.Ho, L.Wo), dtype)
    B.dwconv2d_fwd(d, x, w, b, y0)
    th.cuda.synchronize()
    sc = th.tensor(scale.f64, dtype=th.float32, device="cuda").view(1, -1, 1, 1)
    sh = th.tensor(shift.f64, dtype=th.float32, device="cuda").view(1, -1, 1, 1)
    want = th.clamp(y0.float() * sc + sh, 0.0, 6.0)
    tol = 1e-5 if dtype == "f32" else 3e-2
    assert th.allclose(y.float(), want, rtol=tol, atol=tol)


# ------------------------------------------------------- channels-last forward
# (layer, out_c_offset, out_c_total, activation, expected kernel)
NHWC_CASES = [
    (WL.Layer(N=2, C=64, H=29, W=29, k=3, s=1, p=1, bias=True), 0, 0, "relu6", "nhwc"),
    (WL.Layer(N=3, C=72, H=33, W=33, k=3, s=2, p=1, dtype="bf16"), 0, 0, "relu", "nhwc"),
    (WL.Layer(N=2, C=40, H=21, W=26, k=5, s=1, p=2, bias=True, dtype="f16"), 0, 0, "none", "nhwc"),
    (WL.Layer(N=2, C=36, H=30, W=31, k=7, s=2, p=3), 0, 0, "relu", "nhwc"),
    (WL.Layer(N=1, C=32, H=56, W=56, k=7, s=1, p=3, dtype="bf16"), 0, 0, "relu6", "nhwc"),
    (WL.Layer(N=2, C=16, H=14, W=14, k=5, s=2, p=2, dtype="f16"), 0, 0, "none", "nhwc"),
    (WL.Layer(N=2, C=32, H=17, W=17, k=3, s=1, p=0), 4, 40, "relu", "nhwc"),      # 16-byte-aligned slice
    (WL.Layer(N=2, C=32, H=17, W=17, k=3, s=1, p=1, dtype="bf16"), 1, 35, "none", "nhwc"),  # unaligned slice
    (WL.Layer(N=2, C=6, H=15, W=15, k=3, s=1, p=1), 0, 0, "relu", "generic"),     # C*4 not a multiple of 16
    (WL.Layer(N=2, C=8, H=12, W=12, k=3, s=1, p=1, m=2, bias=True, dtype="f16"), 2, 20, "relu6", "generic"),
    (WL.Layer(N=2, C=16, H=19, W=19, k=3, s=1, p=2, d=2), 0, 0, "none", "generic"),
    (WL.Layer(N=2, C=16, H=16, W=16, k=9, s=1, p=4), 0, 0, "none", "generic"),
]
NHWC_IDS = ["k3s1_f32", "k3s2_bf16_chtail", "k5s1_f16", "k7s2_f32", "k7s1_bf16_56", "k5s2_f16_small",
            "slice_aligned", "slice_unaligned", "C6_generic", "m2_generic", "d2_generic", "k9_generic"]


def nhwc_inputs(L, seed=0):
    inp = WL.make_inputs(L, seed)
    x = to_dev(inp.x).permute(0, 2, 3, 1).contiguous()
    return inp, x


def nhwc_run(L, off, ctot, act, x, inp, scale=None, shift=None):
    th = torch()
    d = B.make_desc(**L.desc_kwargs(), out_c_offset=off, out_c_total=ctot)
    y = empty_dev((L.N, L.Ho, L.Wo, ctot or L.OC), L.dtype, fill=-9.0)
    B.dwconv2d_fwd_nhwc(d, x, to_dev(inp.w), to_dev(inp.b) if inp.b is not None else None, y,
                        scale=None if scale is None else to_dev(scale),
                        shift=None if shift is None else to_dev(shift), act=act)
    th.cuda.synchronize()
    return d, np.ascontiguousarray(to_f64(y).transpose(0, 3, 1, 2))


@pytest.mark.parametrize("L,off,ctot,act,family", NHWC_CASES, ids=NHWC_IDS)
def test_nhwc_vs_oracle(L, off, ctot, act, family):
    inp, x = nhwc_inputs(L)
    scale, shift = folded_bn(L.OC, L.dtype, seed=1) if act != "none" else (None, None)
    d, got = nhwc_run(L, off, ctot, act, x, inp, scale, shift)
    assert B.dwconv2d_plan_name(d, 4) == family
    cv = oconv(L, off=off, c_total=ctot or None)
    ref = np.full(got.shape, -9.0)
    oracle.fwd_epilogue(cv, inp.x.f64, inp.w.f64, None if inp.b is None else inp.b.f64,
                        None if scale is None else scale.f64, None if shift is None else shift.f64,
                        act, y=ref)
    assert_close(got, ref, L.dtype, L.k * L.k, f"nhwc {L.label()}")
    if ctot:
        assert np.all(got[:, :off] == -9.0) and np.all(got[:, off + L.OC:] == -9.0)


def test_nhwc_misaligned_input_takes_generic_kernel():
    """An x that is not 16-byte aligned cannot be a tensor-map base: the call
    runs on the generic kernel and gives the same values."""
    th = torch()
    L = WL.Layer(N=2, C=32, H=20, W=20, k=3, s=1, p=1)
    inp, x = nhwc_inputs(L)
    buf = th.empty(x.numel() + 1, dtype=x.dtype, device="cuda")
    xs = buf[1:].view(x.shape)
    xs.copy_(x)
    _, got = nhwc_run(L, 0, 0, "none", xs, inp)
    _, ref = nhwc_run(L, 0, 0, "none", x, inp)
    assert_close(got, ref, L.dtype, 9, "misaligned nhwc")
    assert_close(got, oracle.fwd(oconv(L), inp.x.f64, inp.w.f64), L.dtype, 9, "misaligned nhwc vs oracle")


def test_nhwc_matches_nchw_forward_bitwise_where_sums_agree():
    """A delta filter makes every output one product, so the channels-last
    and NCHW kernels must agree bit for bit (a check of the layout mapping,
    independent of summation order)."""
    th = torch()
    L = WL.Layer(N=2, C=64, H=23, W=23, k=5, s=2, p=2, dtype="bf16")
    inp, x = nhwc_inputs(L)
    w = np.zeros((L.OC, 5, 5))
    w[:, 1, 3] = np.linspace(0.5, 2.0, L.OC)
    wt = synth.Tensor(w, w.shape, "bf16")
    inp.w = wt
    d, got = nhwc_run(L, 0, 0, "none", x, inp)
    y = empty_dev((L.N, L.OC, L.Ho, L.Wo), "bf16")
    B.dwconv2d_fwd(d, to_dev(inp.x), to_dev(wt), None, y)
    th.cuda.synchronize()
    assert np.array_equal(got, to_f64(y))


def test_nhwc_full_size_mobilenet_layer_sampled():
    """A full-size MobileNet layer in channels-last form (64 x 128 x 56 x 56
    fp32, 3x3 stride 1), compared with the oracle on sampled samples and
    channels."""
    L = WL.Layer(N=64, C=128, H=56, W=56, k=3, s=1, p=1)
    inp, x = nhwc_inputs(L)
    d, got = nhwc_run(L, 0, 0, "none", x, inp)
    assert B.dwconv2d_plan_name(d, 4) == "nhwc"
    nsel, csel = [0, 31, 63], [0, 37, 127]
    cv = oconv(L, N=len(nsel), C=len(csel))
    ref = oracle.fwd(cv, inp.x.f64[np.ix_(nsel, csel)], inp.w.f64[csel])
    assert_close(got[np.ix_(nsel, csel)], ref, "f32", 9, "mobilenet nhwc")


# ------------------------------------------------- depthwise-separable block
# (layer, cout, out_c_offset, out_c_total, dw act, pw act, expected kernel)
SEP_CASES = [
    (WL.Layer(N=2, C=64, H=14, W=14, k=3, s=1, p=1, dtype="bf16"), 64, 0, 0, "relu6", "relu6", "septc"),
    (WL.Layer(N=3, C=128, H=17, W=19, k=3, s=2, p=1, dtype="f16"), 40, 0, 0, "relu", "none", "septc"),
    (WL.Layer(N=2, C=64, H=7, W=7, k=3, s=1, p=1, dtype="bf16"), 256, 0, 0, "relu6", "relu", "septc"),
    (WL.Layer(N=2, C=128, H=9, W=9, k=5, s=1, p=2, dtype="f16"), 300, 0, 0, "none", "relu6", "septc"),
    (WL.Layer(N=1, C=64, H=30, W=30, k=5, s=2, p=2, dtype="bf16"), 96, 0, 0, "relu6", "none", "septc"),
    (WL.Layer(N=5, C=64, H=4, W=4, k=3, s=1, p=1, dtype="bf16"), 32, 0, 0, "relu", "relu", "septc"),
    (WL.Layer(N=2, C=64, H=56, W=56, k=3, s=1, p=1, dtype="bf16"), 128, 8, 136, "relu6", "relu6", "septc"),
    (WL.Layer(N=2, C=64, H=23, W=23, k=3, s=1, p=1, dtype="f16"), 48, 3, 55, "relu6", "none", "septc"),
    (WL.Layer(N=2, C=24, H=15, W=15, k=3, s=1, p=1), 20, 0, 0, "relu6", "relu", "generic"),
    (WL.Layer(N=2, C=48, H=12, W=12, k=3, s=2, p=1, dtype="bf16"), 64, 0, 0, "relu", "relu6", "generic"),
    (WL.Layer(N=2, C=16, H=10, W=10, k=3, s=1, p=1, m=2, dtype="f16"), 24, 0, 0, "none", "none", "generic"),
    (WL.Layer(N=2, C=64, H=13, W=13, k=3, s=1, p=2, d=2, dtype="bf16"), 32, 0, 0, "relu", "relu", "generic"),
]
SEP_IDS = ["k3s1_bf16_14", "k3s2_f16_cout40", "k3_bf16_7x7_pack2", "k5s1_f16_cout300", "k5s2_bf16",
           "bf16_4x4_pack8", "slice_aligned", "slice_unaligned", "f32_generic", "C48_generic",
           "m2_generic", "d2_generic"]


def sep_run(L, cout, off, ctot, a1, a2, seed=0):
    th = torch()
    inp, x = nhwc_inputs(L, seed)
    s1, h1 = WL.make_scale_shift(L, seed)
    wp, s2, h2 = WL.make_pointwise(L, cout, seed)
    d = B.make_desc(**L.desc_kwargs(), out_c_offset=off, out_c_total=ctot)
    y = empty_dev((L.N, L.Ho, L.Wo, ctot or cout), L.dtype, fill=-5.0)
    B.dwconv2d_separable_nhwc(d, x, to_dev(inp.w), cout, to_dev(wp), y, dw_scale=to_dev(s1), dw_shift=to_dev(h1),
                              dw_act=a1, pw_scale=to_dev(s2), pw_shift=to_dev(h2), pw_act=a2)
    th.cuda.synchronize()
    got = np.ascontiguousarray(to_f64(y).transpose(0, 3, 1, 2))
    return d, got, (inp, s1, h1, wp, s2, h2)


@pytest.mark.parametrize("L,cout,off,ctot,a1,a2,family", SEP_CASES, ids=SEP_IDS)
def test_separable_block_vs_oracle(L, cout, off, ctot, a1, a2, family):
    d, got, (inp, s1, h1, wp, s2, h2) = sep_run(L, cout, off, ctot, a1, a2)
    assert B.dwconv2d_separable_plan_name(d, cout) == family
    ref = oracle.separable(oconv(L), inp.x.f64, inp.w.f64, s1.f64, h1.f64, a1, wp.f64, s2.f64, h2.f64, a2)
    assert_close(got[:, off:off + cout], ref, L.dtype, L.k * L.k + L.OC, f"separable {L.label()}")
    if ctot:
        assert np.all(got[:, :off] == -5.0) and np.all(got[:, off + cout:] == -5.0)


def test_separable_block_full_size_mobilenet_sampled():
    """A full-size MobileNet block (64 x 128 x 56 x 56 bf16, 3x3, 1x1 to 128
    channels), compared with the oracle on three whole samples."""
    L = WL.Layer(N=64, C=128, H=56, W=56, k=3, s=1, p=1, dtype="bf16")
    d, got, (inp, s1, h1, wp, s2, h2) = sep_run(L, 128, 0, 0, "relu6", "relu6")
    assert B.dwconv2d_separable_plan_name(d, 128) == "septc"
    nsel = [0, 33, 63]
    ref = oracle.separable(oconv(L, N=3), inp.x.f64[nsel], inp.w.f64, s1.f64, h1.f64, "relu6", wp.f64, s2.f64,
                           h2.f64, "relu6")
    assert_close(got[nsel], ref, "bf16", 9 + 128, "mobilenet separable block")


def test_separable_block_deterministic_and_misaligned_weights_fall_back():
    """Two runs agree bit for bit; a pointwise weight pointer that is not
    16-byte aligned cannot be a tensor-map base and runs the generic kernel,
    within tolerance of the same oracle."""
    th = torch()
    L = WL.Layer(N=2, C=64, H=20, W=20, k=3, s=1, p=1, dtype="bf16")
    _, a, args = sep_run(L, 64, 0, 0, "relu6", "relu")
    _, b, _ = sep_run(L, 64, 0, 0, "relu6", "relu")
    assert np.array_equal(a, b)
    inp, s1, h1, wp, s2, h2 = args
    _, x = nhwc_inputs(L)
    wpd = to_dev(wp)
    buf = th.empty(wpd.numel() + 1, dtype=wpd.dtype, device="cuda")
    wmis = buf[1:].view(wpd.shape)
    wmis.copy_(wpd)
    d = B.make_desc(**L.desc_kwargs())
    y = empty_dev((L.N, L.Ho, L.Wo, 64), "bf16")
    B.dwconv2d_separable_nhwc(d, x, to_dev(inp.w), 64, wmis, y, dw_scale=to_dev(s1), dw_shift=to_dev(h1),
                              dw_act="relu6", pw_scale=to_dev(s2), pw_shift=to_dev(h2), pw_act="relu")
    th.cuda.synchronize()
    got = np.ascontiguousarray(to_f64(y).transpose(0, 3, 1, 2))
    ref = oracle.separable(oconv(L), inp.x.f64, inp.w.f64, s1.f64, h1.f64, "relu6", wp.f64, s2.f64, h2.f64, "relu")
    assert_close(got, ref, "bf16", 9 + 64, "misaligned pointwise weights")


def test_no_bounded_wait_gave_up_in_fused_kernels():
    assert B.dwconv_device_timeouts() == 0
