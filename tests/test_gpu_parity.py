"""GPU parity: libdwconv (through its C ABI) against the fp64 oracle.

Small shapes are compared element by element over whole tensors; the full
workload sizes run in the launch configuration the benchmark times and are
compared on sampled planes / channels that the oracle computes exactly.
Tolerances: fp32 normwise max|g-r|/max|r| <= 1e-5 sqrt(taps); fp16/bf16
elementwise |g-r| <= 1e-2 + 2e-2 |r| (fp32 accumulation inside).
"""
import zlib
import math
import os

import numpy as np
import pytest

import oracle
from depthwise_convolution_dwconv2d_gb300 import binding as B
from depthwise_convolution_dwconv2d_gb300 import synth, workloads as WL
from dw_testutil import assert_close, empty_dev, oconv, to_dev, to_f64, torch, ws_for
from oracle import Conv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    th = pytest.importorskip("torch")
    if not th.cuda.is_available():
        pytest.skip("no CUDA device")
    from depthwise_convolution_dwconv2d_gb300 import build
    build.build()
    B.load()


def desc_of(L, off=0, c_total=0):
    return B.make_desc(**L.desc_kwargs(), out_c_offset=off, out_c_total=c_total)


def run_all(L, inp, want_b=None):
    """fwd, bwd_data and bwd_weight (+ bias grad) on the GPU; float64 results."""
    th = torch()
    d = desc_of(L)
    x, w, gy = to_dev(inp.x), to_dev(inp.w), to_dev(inp.gy)
    b = to_dev(inp.b) if inp.b is not None else None
    y = empty_dev((L.N, L.OC, L.Ho, L.Wo), L.dtype)
    B.dwconv2d_fwd(d, x, w, b, y)
    gx = empty_dev((L.N, L.C, L.H, L.W), L.dtype)
    B.dwconv2d_bwd_data(d, gy, w, gx, 0)
    gw = empty_dev((L.OC, L.k, L.k), L.dtype)
    want_b = L.bias if want_b is None else want_b
    gb = empty_dev((L.OC,), L.dtype) if want_b else None
    ws, nbytes = ws_for(d)
    B.dwconv2d_bwd_weight(d, x, gy, gw, gb, ws, nbytes)
    th.cuda.synchronize()
    return to_f64(y), to_f64(gx), to_f64(gw), (to_f64(gb) if gb is not None else None)


def check_full(L, inp, label=""):
    y, gx, gw, gb = run_all(L, inp)
    cv = oconv(L)
    b64 = inp.b.f64 if inp.b is not None else None
    taps = L.k * L.k
    assert_close(y, oracle.fwd(cv, inp.x.f64, inp.w.f64, b64), L.dtype, taps, f"{label} fwd")
    assert_close(gx, oracle.bwd_data(cv, inp.gy.f64, inp.w.f64), L.dtype, taps * L.m, f"{label} bwd_data")
    rgw, rgb = oracle.bwd_weight(cv, inp.x.f64, inp.gy.f64, want_w=True, want_b=L.bias)
    assert_close(gw, rgw, L.dtype, taps, f"{label} bwd_weight")
    if L.bias:
        assert_close(gb, rgb, L.dtype, 1, f"{label} bias grad")


def check_sampled(L, inp, nsel, csel, label=""):
    """Full-size GPU run; oracle on the planes (nsel x csel) for fwd / bwd_data
    and on whole channels csel (all N) for bwd_weight."""
    y, gx, gw, gb = run_all(L, inp)
    m = L.m
    ocsel = [c * m + j for c in csel for j in range(m)]
    xs = inp.x.f64[np.ix_(nsel, csel)]
    ws = inp.w.f64[ocsel]
    gys = inp.gy.f64[np.ix_(nsel, ocsel)]
    bs = inp.b.f64[ocsel] if inp.b is not None else None
    cv = oconv(L, N=len(nsel), C=len(csel))
    taps = L.k * L.k
    assert_close(y[np.ix_(nsel, ocsel)], oracle.fwd(cv, xs, ws, bs), L.dtype, taps, f"{label} fwd")
    assert_close(gx[np.ix_(nsel, csel)], oracle.bwd_data(cv, gys, ws), L.dtype, taps * m, f"{label} bwd_data")
    cvw = oconv(L, C=len(csel))
    rgw, rgb = oracle.bwd_weight(cvw, inp.x.f64[:, csel], inp.gy.f64[:, ocsel], want_w=True, want_b=L.bias)
    assert_close(gw[ocsel], rgw, L.dtype, taps, f"{label} bwd_weight")
    if L.bias:
        assert_close(gb[ocsel], rgb, L.dtype, 1, f"{label} bias grad")


# ---------------------------------------------------------------- workloads
def test_pr1_full():
    L = WL.pr1()[0]
    check_full(L, WL.make_inputs(L), "pr1")


@pytest.mark.parametrize("L", WL.mobilenet(), ids=lambda L: L.name)
def test_mobilenet_full_size_sampled(L):
    inp = WL.make_inputs(L)
    check_sampled(L, inp, [0, 31, 63], [0, 1, L.C // 2 + 1, L.C - 1], L.name)


@pytest.mark.parametrize("L", WL.mobilenet(N=3), ids=lambda L: L.name)
def test_mobilenet_small_batch_full(L):
    check_full(L, WL.make_inputs(L), L.name)


def test_multiplier_full_size():
    L = WL.multiplier()[0]
    inp = WL.make_inputs(L)
    check_sampled(L, inp, [0, 64, 127], [0, 77, 255], L.name)


_LK_CACHE = {}


def _largek_inputs(L):
    """x and grad_out depend only on (H, dtype) here (stride 1, pad k//2); keep
    the most recent pair instead of redrawing 100M values per kernel size."""
    key = (L.H, L.dtype)
    if key not in _LK_CACHE:
        _LK_CACHE.clear()
        _LK_CACHE[key] = WL.make_inputs(WL.Layer(N=L.N, C=L.C, H=L.H, W=L.W, k=1, p=0, dtype=L.dtype))
    base = _LK_CACHE[key]
    w = synth.normal_tensor((L.OC, L.k, L.k), L.dtype, 0, synth.STREAM_W, std=1.0 / L.k)
    return WL.Inputs(base.x, w, None, base.gy)


@pytest.mark.parametrize("L", WL.largek(), ids=lambda L: L.name)
def test_largek_full_size_sampled(L):
    # edge and interior samples and channels: the persistent kernels' units
    # straddle plane groups, so the middle of the tensor is checked too
    check_sampled(L, _largek_inputs(L), [0, 31, 63], [0, 1, 191, 383], L.name)


def run_multi(M, xs, wsx, gy_t):
    th = torch()
    brs, ctot = M.branches()
    descs = [B.make_desc(**L.desc_kwargs(), out_c_offset=i * M.C, out_c_total=ctot)
             for i, L in enumerate(brs)]
    x = to_dev(xs)
    wd = [to_dev(w) for w in wsx]
    y = empty_dev((M.N, ctot, M.H, M.W), M.dtype)
    B.dwconv2d_fwd_multi(descs, x, wd, None, y)
    gy = to_dev(gy_t)
    gx = empty_dev((M.N, M.C, M.H, M.W), M.dtype)
    B.dwconv2d_bwd_data_multi(descs, gy, wd, gx)
    th.cuda.synchronize()
    return brs, ctot, to_f64(y), to_f64(gx)


@pytest.mark.parametrize("M", [WL.multidil(), WL.Multi(N=1, C=5, H=37, W=29, dtype="f32"),
                               WL.Multi(N=2, C=3, H=20, W=21, dilations=(1, 2), dtype="f16")],
                         ids=["multidil_full", "multi_small_f32", "multi_2br_f16"])
def test_multi_branch(M):
    brs, ctot = M.branches()
    L0 = brs[0]
    inp = WL.make_inputs(L0, gy_channels=ctot)
    wsx = [inp.w] + [synth.normal_tensor((M.C, M.k, M.k), M.dtype, 0, synth.STREAM_W + 16 * i, std=M.w_std)
                     for i in range(1, len(brs))]
    brs, ctot, y, gx = run_multi(M, inp.x, wsx, inp.gy)
    cvs = [oconv(L, off=i * M.C, c_total=ctot) for i, L in enumerate(brs)]
    ry = oracle.fwd_multi(cvs, inp.x.f64, [w.f64 for w in wsx])
    assert_close(y, ry, M.dtype, 9, "multi fwd")
    rgx = oracle.bwd_data_multi(cvs, inp.gy.f64, [w.f64 for w in wsx])
    assert_close(gx, rgx, M.dtype, 9 * len(brs), "multi bwd_data")
    # weight gradient of each branch through the single-branch entry point
    th = torch()
    x, gyd = to_dev(inp.x), to_dev(inp.gy)
    for i, L in enumerate(brs):
        d = B.make_desc(**L.desc_kwargs(), out_c_offset=i * M.C, out_c_total=ctot)
        gw = empty_dev((M.C, M.k, M.k), M.dtype)
        ws, nb = ws_for(d)
        B.dwconv2d_bwd_weight(d, x, gyd, gw, None, ws, nb)
        th.cuda.synchronize()
        rgw, _ = oracle.bwd_weight(cvs[i], inp.x.f64, inp.gy.f64)
        assert_close(to_f64(gw), rgw, M.dtype, 9, f"multi bwd_weight branch {i}")


# ---------------------------------------------------------------- sweep
def sweep_cases():
    rng = np.random.default_rng(7)
    cases = []
    ks = [1, 2, 3, 4, 5, 6, 7, 31]
    for i in range(60):
        k = ks[i % len(ks)]
        kw = k if i % 3 else max(1, ks[(i + 3) % len(ks)] % 8)
        s = [1, 2, 3][i % 3]
        d = [1, 1, 2, 3, 5][i % 5]
        m = [1, 2, 3][(i // 3) % 3]
        dtype = ["f32", "f16", "bf16"][(i // 2) % 3]
        H = int(rng.integers(1, 40)) + d * (k - 1)
        W = int(rng.integers(1, 45)) + d * (kw - 1)
        if k == 31:
            d = 1
            H, W = int(rng.integers(20, 70)), int(rng.integers(20, 70))
        ph = int(rng.integers(0, k // 2 * d + 1))
        pw = int(rng.integers(0, kw // 2 * d + 1))
        N, C = int(rng.integers(1, 4)), int(rng.integers(1, 6))
        cases.append(dict(N=N, C=C, H=H, W=W, kh=k, kw=kw, s=s, sw=max(1, s - (i % 2)), d=d,
                          dw=1 if i % 4 == 0 else d, ph=ph, pw=pw, m=m, dtype=dtype, bias=bool(i % 2)))
    return cases


@pytest.mark.parametrize("cs", sweep_cases(), ids=lambda c: "k{kh}x{kw}s{s}{sw}d{d}{dw}p{ph}{pw}m{m}{dtype}N{N}C{C}H{H}W{W}".format(**c))
def test_sweep_vs_oracle(cs):
    th = torch()
    cv = Conv(N=cs["N"], C=cs["C"], H=cs["H"], W=cs["W"], kh=cs["kh"], kw=cs["kw"], sh=cs["s"],
              sw=cs["sw"], ph=cs["ph"], pw=cs["pw"], dh=cs["d"], dw=cs["dw"], m=cs["m"])
    if cv.Ho < 1 or cv.Wo < 1:
        pytest.skip("empty output")
    dt = cs["dtype"]
    seed = zlib.crc32(repr(sorted(cs.items())).encode()) % 1000
    x = synth.uniform_tensor((cv.N, cv.C, cv.H, cv.W), dt, seed, 0)
    w = synth.normal_tensor((cv.OC, cv.kh, cv.kw), dt, seed, 1, std=1 / math.sqrt(cv.kh * cv.kw))
    b = synth.normal_tensor((cv.OC,), dt, seed, 2) if cs["bias"] else None
    gy = synth.normal_tensor((cv.N, cv.OC, cv.Ho, cv.Wo), dt, seed, 3)
    d = B.make_desc(cv.N, cv.C, cv.H, cv.W, (cv.kh, cv.kw), (cv.sh, cv.sw), (cv.ph, cv.pw),
                    (cv.dh, cv.dw), cv.m, dt)
    xd, wd, gyd = to_dev(x), to_dev(w), to_dev(gy)
    bd = to_dev(b) if b is not None else None
    y = empty_dev((cv.N, cv.OC, cv.Ho, cv.Wo), dt)
    B.dwconv2d_fwd(d, xd, wd, bd, y)
    gx = empty_dev((cv.N, cv.C, cv.H, cv.W), dt)
    B.dwconv2d_bwd_data(d, gyd, wd, gx, 0)
    gw = empty_dev((cv.OC, cv.kh, cv.kw), dt)
    gb = empty_dev((cv.OC,), dt) if b is not None else None
    ws, nb = ws_for(d)
    B.dwconv2d_bwd_weight(d, xd, gyd, gw, gb, ws, nb)
    th.cuda.synchronize()
    taps = cv.kh * cv.kw
    assert_close(to_f64(y), oracle.fwd(cv, x.f64, w.f64, None if b is None else b.f64), dt, taps, "fwd")
    assert_close(to_f64(gx), oracle.bwd_data(cv, gy.f64, w.f64), dt, taps * cv.m, "bwd_data")
    rgw, rgb = oracle.bwd_weight(cv, x.f64, gy.f64, want_w=True, want_b=b is not None)
    assert_close(to_f64(gw), rgw, dt, taps, "bwd_weight")
    if b is not None:
        assert_close(to_f64(gb), rgb, dt, 1, "bias grad")


# ---------------------------------------------------------------- properties
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("k,s,d", [(3, 1, 1), (3, 2, 1), (5, 1, 2), (31, 1, 1), (7, 2, 1)])
def test_delta_kernel_bit_exact(dtype, k, s, d):
    """A delta filter copies the shifted input: exact in every dtype."""
    th = torch()
    L = WL.Layer(N=2, C=6, H=37, W=45, k=k, s=s, p=d * (k // 2), d=d, dtype=dtype)
    x = synth.normal_tensor((L.N, L.C, L.H, L.W), dtype, 3, 0)
    wv = np.zeros((L.OC, k, k))
    for oc in range(L.OC):
        wv[oc, oc % k, (2 * oc) % k] = 1.0
    w = synth.Tensor(wv, wv.shape, dtype)
    y = empty_dev((L.N, L.OC, L.Ho, L.Wo), dtype)
    B.dwconv2d_fwd(desc_of(L), to_dev(x), to_dev(w), None, y)
    th.cuda.synchronize()
    ref = oracle.fwd(oconv(L), x.f64, w.f64)
    assert np.array_equal(to_f64(y), ref)


@pytest.mark.parametrize("L", [WL.mobilenet(N=4)[1], WL.mobilenet(N=4)[0],
                               WL.Layer(N=2, C=8, H=33, W=35, k=5, p=2, m=2, bias=True, dtype="bf16"),
                               WL.Layer(N=2, C=4, H=40, W=40, k=13, p=6, dtype="f16"),
                               WL.Layer(N=3, C=4, H=40, W=36, k=21, p=10, bias=True, dtype="f32"),
                               WL.Layer(N=2, C=3, H=34, W=34, k=31, p=15, dtype="f32")],
                         ids=["s1", "s2", "m2bf16", "k13f16", "k21f32", "k31f32"])
def test_slice_guard_bands_and_accumulate(L):
    """Channels outside the slice stay bit-identical; accumulate adds."""
    th = torch()
    inp = WL.make_inputs(L, gy_channels=L.OC + 5)
    ctot, off = L.OC + 5, 3
    d = desc_of(L, off, ctot)
    x, w = to_dev(inp.x), to_dev(inp.w)
    b = to_dev(inp.b) if inp.b is not None else None
    y = empty_dev((L.N, ctot, L.Ho, L.Wo), L.dtype, fill=-7.5)
    B.dwconv2d_fwd(d, x, w, b, y)
    yh = to_f64(y)
    assert np.all(yh[:, :off] == -7.5) and np.all(yh[:, off + L.OC:] == -7.5)
    cv = oconv(L, off=off, c_total=ctot)
    ry = oracle.fwd(cv, inp.x.f64, inp.w.f64, inp.b.f64 if inp.b is not None else None)
    assert_close(yh[:, off:off + L.OC], ry[:, off:off + L.OC], L.dtype, L.k * L.k, "slice fwd")
    gy = to_dev(inp.gy)
    gx = empty_dev((L.N, L.C, L.H, L.W), L.dtype, fill=0.5)
    B.dwconv2d_bwd_data(d, gy, w, gx, 1)
    rgx = oracle.bwd_data(cv, inp.gy.f64, inp.w.f64) + 0.5
    assert_close(to_f64(gx), rgx, L.dtype, L.k * L.k * L.m, "accumulate bwd_data")
    gw = empty_dev((L.OC, L.k, L.k), L.dtype)
    ws, nb = ws_for(d)
    B.dwconv2d_bwd_weight(d, x, gy, gw, None, ws, nb)
    th.cuda.synchronize()
    rgw, _ = oracle.bwd_weight(cv, inp.x.f64, inp.gy.f64)
    assert_close(to_f64(gw), rgw, L.dtype, L.k * L.k, "slice bwd_weight")


@pytest.mark.parametrize("L", [WL.mobilenet(N=8)[1], WL.mobilenet(N=8)[7], WL.multiplier(N=4)[0],
                               WL.Layer(N=4, C=16, H=48, W=48, k=27, p=13, dtype="f32")],
                         ids=["mb56", "mb7s2", "mult", "k27"])
def test_determinism(L):
    inp = WL.make_inputs(L)
    a = run_all(L, inp)
    b = run_all(L, inp)
    for u, v in zip(a, b):
        if u is not None:
            assert np.array_equal(u, v)


def test_empty_batch_and_workspace_zero_case():
    th = torch()
    L = WL.Layer(N=0, C=4, H=9, W=9)
    d = desc_of(L)
    w = empty_dev((4, 3, 3), "f32", fill=1.0)
    gw = empty_dev((4, 3, 3), "f32", fill=3.0)
    gb = empty_dev((4,), "f32", fill=3.0)
    ws, nb = ws_for(d)
    B.dwconv2d_fwd(d, None, w, None, None)
    B.dwconv2d_bwd_weight(d, None, None, gw, gb, ws, nb)
    th.cuda.synchronize()
    assert np.all(to_f64(gw) == 0) and np.all(to_f64(gb) == 0)


def test_generic_and_planned_kernels_agree():
    """The planner's kernels and the generic kernels agree within tolerance."""
    L = WL.mobilenet(N=4)[1]
    inp = WL.make_inputs(L)
    a = run_all(L, inp)
    os.environ["DWCONV_FORCE_ALGO"] = "generic"
    try:
        b = run_all(L, inp)
    finally:
        del os.environ["DWCONV_FORCE_ALGO"]
    for u, v in zip(a, b):
        if u is not None:
            assert_close(u, v, L.dtype, 9, "planned vs generic")


def test_no_bounded_wait_gave_up():
    """Every tile copy the suite waited for arrived (no timeouts counted)."""
    assert B.dwconv_device_timeouts() == 0


@pytest.mark.parametrize("L", [WL.Layer(N=3, C=5, H=21, W=19, k=7, p=3, bias=True, dtype="f32"),
                               WL.Layer(N=2, C=3, H=30, W=33, k=13, p=6, dtype="bf16"),
                               WL.Layer(N=3, C=7, H=17, W=16, k=31, p=15, bias=True, dtype="f16"),
                               WL.Layer(N=2, C=6, H=12, W=12, k=9, p=2, dtype="f32")],
                         ids=["k7f32", "k13bf16", "k31f16", "k9p2"])
def test_large_kernels_planes_straddle_samples(L):
    """Large kernels where a CTA's planes span two samples (C not a multiple
    of the planes per CTA), with bias and non-"same" padding."""
    check_full(L, WL.make_inputs(L), L.label())


def _large_direct_cases():
    """Every odd filter size 9..31 on the direct large kernels: ragged planes
    (widths that are not multiples of the 8-column blocks), planes above and
    below 32 rows (two- and four-row blocks), "same" and other paddings,
    every storage type, bias on some."""
    cases = []
    for i, k in enumerate(range(9, 32, 2)):
        H = [12, 37, 20, 45, 33, 19][i % 6] + (k if i % 2 else 0) // 3
        W = [16, 13, 41, 24, 35, 9][(i + 1) % 6] + k // 4
        p = k // 2 if i % 3 else max(0, k // 2 - 3)
        dt = ["f32", "f16", "bf16"][i % 3]
        cases.append(WL.Layer(N=2 + i % 2, C=3 + i % 3, H=H, W=W, k=k, p=p, bias=i % 2 == 1, dtype=dt,
                              name=f"k{k}H{H}W{W}p{p}{dt}"))
    return cases


@pytest.mark.parametrize("L", _large_direct_cases(), ids=lambda L: L.name)
def test_large_direct_every_odd_filter(L):
    """The direct large kernels (16-bit forward and grad-input kept off the
    tensor cores) against the oracle, including the 17/19/23/25/29 sizes."""
    os.environ["DWCONV_FORCE_ALGO"] = "direct"
    try:
        d = desc_of(L)
        assert [B.dwconv2d_plan_name(d, q) for q in range(3)] == ["large"] * 3
        check_full(L, WL.make_inputs(L), L.label())
    finally:
        del os.environ["DWCONV_FORCE_ALGO"]


BANDED_WGRAD = [
    WL.Layer(N=3, C=2, H=112, W=112, k=15, p=7, bias=True, dtype="f32", name="k15H112_f32"),
    WL.Layer(N=2, C=3, H=128, W=120, k=21, p=10, dtype="f32", name="k21H128W120_f32"),
    WL.Layer(N=5, C=2, H=100, W=97, k=19, p=3, dtype="bf16", name="k19H100W97p3_bf16"),
    WL.Layer(N=2, C=3, H=112, W=100, k=27, p=13, bias=True, dtype="f32", name="k27H112W100_f32"),
    WL.Layer(N=3, C=2, H=120, W=72, k=31, p=9, dtype="f16", name="k31H120W72p9_f16"),
]


@pytest.mark.parametrize("L", BANDED_WGRAD, ids=lambda L: L.name)
def test_large_weight_gradient_banded_planes(L):
    """The packed large weight gradient (13 taps and up) on planes it cuts into
    bands of output rows (112..128 rows), with bias, a ragged odd width and
    non-"same" padding, against the oracle."""
    os.environ["DWCONV_FORCE_ALGO"] = "direct"
    try:
        assert B.dwconv2d_plan_name(desc_of(L), 2) == "large"
        check_full(L, WL.make_inputs(L), L.label())
    finally:
        del os.environ["DWCONV_FORCE_ALGO"]


ODD_BATCH_WGRAD = [
    WL.Layer(N=1, C=3, H=40, W=40, k=31, p=15, dtype="f32", name="N1_k31"),
    WL.Layer(N=9, C=40, H=32, W=32, k=31, p=15, bias=True, dtype="f32", name="N9C40_k31"),
    WL.Layer(N=7, C=6, H=36, W=36, k=21, p=10, dtype="f32", name="N7_k21"),
    WL.Layer(N=3, C=5, H=20, W=44, k=13, p=6, bias=True, dtype="f32", name="N3_k13W44"),
]


@pytest.mark.parametrize("L", ODD_BATCH_WGRAD, ids=lambda L: L.name)
def test_packed_weight_gradient_odd_batches(L):
    """The packed fp32 weight gradient walks samples in pairs over chunks of
    an even number of samples; with an odd batch the last chunk ends in a
    pair whose second sample is missing (zero-filled). One sample, nine
    samples in chunks of two, seven, and three, against the oracle."""
    assert B.dwconv2d_plan_name(desc_of(L), 2) == "large"
    check_full(L, WL.make_inputs(L), L.label())


def test_large_direct_accumulate_into_gx():
    """The stride-1 grad-input of the direct large kernels adds into gx when
    asked (accumulate = 1)."""
    th = torch()
    L = WL.Layer(N=2, C=3, H=40, W=21, k=17, p=8, dtype="f32")
    inp = WL.make_inputs(L)
    d = desc_of(L)
    gy, w = to_dev(inp.gy), to_dev(inp.w)
    base = synth.normal_tensor((L.N, L.C, L.H, L.W), "f32", 5, 0)
    gx = to_dev(base)
    B.dwconv2d_bwd_data(d, gy, w, gx, 1)
    th.cuda.synchronize()
    ref = base.f64 + oracle.bwd_data(oconv(L), inp.gy.f64, inp.w.f64)
    assert_close(to_f64(gx), ref, "f32", L.k * L.k, "accumulated gx")


CLIFF_CASES = [
    WL.Layer(N=3, C=5, H=56, W=56, k=3, s=3, p=1, bias=True, dtype="f32", name="k3s3p1_f32"),
    WL.Layer(N=2, C=4, H=29, W=31, k=3, s=3, p=0, dtype="bf16", name="k3s3p0_bf16"),
    WL.Layer(N=3, C=5, H=40, W=36, k=5, s=1, p=6, d=3, bias=True, dtype="f32", name="k5d3_f32"),
    WL.Layer(N=2, C=3, H=33, W=27, k=5, s=1, p=6, d=3, dtype="f16", name="k5d3_f16"),
    WL.Layer(N=3, C=4, H=56, W=56, k=7, s=2, p=3, dtype="f32", name="k7s2_f32"),
    WL.Layer(N=2, C=3, H=30, W=34, k=7, s=2, p=3, bias=True, dtype="bf16", name="k7s2_bf16"),
]


@pytest.mark.parametrize("L", CLIFF_CASES, ids=lambda L: L.name)
def test_tile_kernels_for_stride3_dilation3_and_7x7_stride2(L):
    """3x3 stride 3, 5x5 dilation 3 and the 7x7 stride-2 weight gradient run
    on the tile kernels (not the generic one-output-per-thread kernels)."""
    d = desc_of(L)
    assert [B.dwconv2d_plan_name(d, q) for q in range(3)] == ["tile"] * 3
    check_full(L, WL.make_inputs(L), L.label())


# ------------------------------------------------ tensor-core large kernels
IBG_CASES = [
    WL.Layer(N=3, C=5, H=32, W=32, k=31, p=15, bias=True, dtype="f16"),
    WL.Layer(N=20, C=3, H=48, W=48, k=13, p=6, dtype="bf16"),
    WL.Layer(N=2, C=4, H=17, W=16, k=9, p=4, bias=True, dtype="f16"),
    WL.Layer(N=2, C=3, H=24, W=24, k=11, p=2, dtype="bf16"),
    WL.Layer(N=130, C=2, H=16, W=16, k=15, p=7, dtype="bf16"),
    WL.Layer(N=1, C=3, H=64, W=64, k=27, p=13, dtype="f16"),
]
IBG_IDS = ["k31f16_T8", "k13bf16_W48", "k9f16_raggedM", "k11bf16_p2", "k15bf16_N130", "k27f16_W64"]


@pytest.mark.parametrize("L", IBG_CASES, ids=IBG_IDS)
def test_ibgemm_vs_oracle(L):
    """Implicit batched GEMM on the tensor cores: several M tiles per plane, a
    ragged last tile, K steps that straddle input rows (W = 48), a ragged batch
    (zero-filled samples), non-"same" padding and a batch above 128."""
    d = desc_of(L)
    assert B.dwconv2d_plan_name(d, 0) == "ibgemm"
    if L.p == L.k // 2:
        assert B.dwconv2d_plan_name(d, 1) == "ibgemm"
    check_full(L, WL.make_inputs(L), L.label())


@pytest.mark.parametrize("L", [IBG_CASES[0], IBG_CASES[1]], ids=IBG_IDS[:2])
def test_ibgemm_and_direct_agree(L):
    """The tensor-core kernels and the direct large-kernel ones agree."""
    inp = WL.make_inputs(L)
    a = run_all(L, inp)
    os.environ["DWCONV_FORCE_ALGO"] = "direct"
    try:
        assert B.dwconv2d_plan_name(desc_of(L), 0) == "large"
        b = run_all(L, inp)
    finally:
        del os.environ["DWCONV_FORCE_ALGO"]
    for u, v in zip(a[:2], b[:2]):
        assert_close(u, v, L.dtype, L.k * L.k, "ibgemm vs direct")


def test_ibgemm_misaligned_input_falls_back():
    """An input pointer off the 16-byte grid runs on the direct kernels."""
    th = torch()
    L = IBG_CASES[2]
    inp = WL.make_inputs(L)
    d = desc_of(L)
    n = L.N * L.C * L.H * L.W
    xbuf = empty_dev((n + 8,), L.dtype)
    xv = xbuf[1:1 + n].view(L.N, L.C, L.H, L.W)
    xv.copy_(to_dev(inp.x))
    w, b = to_dev(inp.w), to_dev(inp.b)
    y = empty_dev((L.N, L.C, L.Ho, L.Wo), L.dtype)
    B.dwconv2d_fwd(d, xv, w, b, y)
    th.cuda.synchronize()
    assert_close(to_f64(y), oracle.fwd(oconv(L), inp.x.f64, inp.w.f64, inp.b.f64), L.dtype, L.k * L.k,
                 "misaligned fwd")


def test_no_bounded_wait_gave_up_after_ibgemm():
    assert B.dwconv_device_timeouts() == 0


TCW_CASES = [
    WL.Layer(N=5, C=3, H=32, W=32, k=31, p=15, bias=True, dtype="f16"),
    WL.Layer(N=7, C=5, H=24, W=16, k=9, p=4, dtype="bf16"),
    WL.Layer(N=3, C=4, H=17, W=24, k=13, p=2, bias=True, dtype="f16"),
    WL.Layer(N=2, C=3, H=40, W=40, k=17, p=8, dtype="bf16"),
    WL.Layer(N=11, C=2, H=16, W=16, k=15, p=7, bias=True, dtype="bf16"),
    WL.Layer(N=2, C=3, H=64, W=64, k=27, p=13, dtype="f16"),
]
TCW_IDS = ["k31f16_b", "k9bf16_W16", "k13f16_p2", "k17bf16", "k15bf16_N11", "k27f16_64"]


@pytest.mark.parametrize("L", TCW_CASES, ids=TCW_IDS)
def test_tensor_core_weight_gradient_vs_oracle(L):
    """Large-filter fp16 / bf16 weight gradient on the tensor cores: "same"
    and other paddings, planes taller than wide, batch chunks of several
    samples, several channels, bias gradient."""
    d = desc_of(L)
    if L.Wo % 8 == 0:
        assert B.dwconv2d_plan_name(d, 2) == "tcwgrad"
    check_full(L, WL.make_inputs(L), L.label())


def test_tensor_core_weight_gradient_reads_its_slice():
    """The weight gradient reads grad_out from a channel slice of a wider
    tensor (offset 3 of 11 channels)."""
    th = torch()
    L = WL.Layer(N=3, C=4, H=24, W=24, k=11, p=5, bias=True, dtype="f16")
    inp = WL.make_inputs(L, gy_channels=11)
    d = desc_of(L, off=3, c_total=11)
    assert B.dwconv2d_plan_name(d, 2) == "tcwgrad"
    x, gy = to_dev(inp.x), to_dev(inp.gy)
    gw = empty_dev((L.OC, L.k, L.k), L.dtype)
    gb = empty_dev((L.OC,), L.dtype)
    ws, nbytes = ws_for(d)
    B.dwconv2d_bwd_weight(d, x, gy, gw, gb, ws, nbytes)
    th.cuda.synchronize()
    rgw, rgb = oracle.bwd_weight(oconv(L, off=3, c_total=11), inp.x.f64, inp.gy.f64, want_w=True, want_b=True)
    assert_close(to_f64(gw), rgw, L.dtype, L.k * L.k, "sliced gw")
    assert_close(to_f64(gb), rgb, L.dtype, 1, "sliced gb")


def test_tensor_core_weight_gradient_deterministic_and_matches_direct():
    """Bitwise repeatable, and within the fp16 tolerance of the direct
    (FMA) weight gradient."""
    th = torch()
    L = TCW_CASES[0]
    inp = WL.make_inputs(L)
    d = desc_of(L)
    x, gy = to_dev(inp.x), to_dev(inp.gy)
    outs = []
    for force in (None, None, "direct"):
        if force:
            os.environ["DWCONV_FORCE_ALGO"] = force
        try:
            gw = empty_dev((L.OC, L.k, L.k), L.dtype)
            ws, nbytes = ws_for(d)
            B.dwconv2d_bwd_weight(d, x, gy, gw, None, ws, nbytes)
            th.cuda.synchronize()
            outs.append(to_f64(gw))
        finally:
            if force:
                del os.environ["DWCONV_FORCE_ALGO"]
    assert np.array_equal(outs[0], outs[1])
    assert_close(outs[0], outs[2], L.dtype, L.k * L.k, "tensor-core vs direct gw")


def test_tensor_core_weight_gradient_misaligned_input_falls_back():
    """An x pointer off the 16-byte grid runs on the direct kernels."""
    th = torch()
    L = TCW_CASES[1]
    inp = WL.make_inputs(L)
    d = desc_of(L)
    n = L.N * L.C * L.H * L.W
    xbuf = empty_dev((n + 8,), L.dtype)
    xv = xbuf[1:1 + n].view(L.N, L.C, L.H, L.W)
    xv.copy_(to_dev(inp.x))
    gw = empty_dev((L.OC, L.k, L.k), L.dtype)
    ws, nbytes = ws_for(d)
    B.dwconv2d_bwd_weight(d, xv, to_dev(inp.gy), gw, None, ws, nbytes)
    th.cuda.synchronize()
    rgw, _ = oracle.bwd_weight(oconv(L), inp.x.f64, inp.gy.f64)
    assert_close(to_f64(gw), rgw, L.dtype, L.k * L.k, "misaligned gw")


def test_no_bounded_wait_gave_up_after_tensor_core_wgrad():
    assert B.dwconv_device_timeouts() == 0


# ------------------------------------------------------ small-plane kernels
PLANE_CASES = [
    WL.Layer(N=3, C=5, H=14, W=14, k=3, s=1, p=1, bias=True, dtype="f32"),
    WL.Layer(N=5, C=3, H=15, W=13, k=3, s=2, p=1, dtype="f32"),
    WL.Layer(N=2, C=4, H=7, W=7, k=3, s=2, p=1, dtype="bf16"),
    WL.Layer(N=3, C=2, H=28, W=28, k=3, s=2, p=1, bias=True, dtype="f16"),
    WL.Layer(N=2, C=3, H=9, W=16, k=3, s=1, p=0, dtype="f32"),
    WL.Layer(N=2, C=3, H=10, W=11, k=3, s=1, p=2, dtype="f32"),
    WL.Layer(N=17, C=3, H=10, W=11, k=3, s=2, p=2, bias=True, dtype="f32"),
    WL.Layer(N=3, C=5, H=40, W=12, k=3, s=1, p=1, bias=True, dtype="f32"),
]
PLANE_IDS = ["14s1", "15x13s2", "7s2bf16", "28s2f16", "w16p0", "p2s1", "p2s2N17", "tall40x12"]


@pytest.mark.parametrize("L", PLANE_CASES, ids=PLANE_IDS)
def test_plane_kernels_vs_oracle(L):
    """One warp per group of small planes: odd sizes, stride 2, padding 0 and
    2, ragged batches, all dtypes, bias. The planner uses them for the forward
    on rows of 9..16, the stride-1 grad-input on rows of 9..16 and the
    weight gradient on output rows of at most 16."""
    d = desc_of(L)
    narrow = 8 < L.W <= 16
    assert (B.dwconv2d_plan_name(d, 0) == "plane") == narrow
    assert (B.dwconv2d_plan_name(d, 1) == "plane") == (narrow and L.s == 1)
    assert B.dwconv2d_plan_name(d, 2) == "plane"
    check_full(L, WL.make_inputs(L), L.label())


def test_plane_wgrad_unit_with_empty_group():
    """62 samples, 128 channels of 14x14: the weight gradient's units are two
    sample groups of two samples (16 chunks of 4 samples, so 16 * 128 * 10
    fp32 partials); the last chunk holds samples 60, 61 only, so its second
    group is empty and must not overwrite the unit's partial."""
    L = WL.Layer(N=62, C=128, H=14, W=14, k=3, s=1, p=1, bias=True, dtype="f32")
    d = desc_of(L)
    assert B.dwconv2d_plan_name(d, 2) == "plane"
    _, nbytes = ws_for(d)
    assert nbytes >= 16 * L.OC * 10 * 4
    assert nbytes < 17 * L.OC * 10 * 4
    check_full(L, WL.make_inputs(L), L.label())


def test_plane_tall_strided_planes():
    """64 x 16 planes at stride 2: the forward's tile buffers do not fit a
    CTA's shared memory, so it runs on the tile kernel; the weight gradient
    runs on the plane kernel with four-warp CTAs."""
    L = WL.Layer(N=2, C=3, H=64, W=16, k=3, s=2, p=1, bias=True, dtype="f32")
    d = desc_of(L)
    assert B.dwconv2d_plan_name(d, 0) != "plane"
    assert B.dwconv2d_plan_name(d, 2) == "plane"
    check_full(L, WL.make_inputs(L), L.label())


@pytest.mark.parametrize("L", [PLANE_CASES[0], PLANE_CASES[1]], ids=PLANE_IDS[:2])
def test_plane_slices_and_accumulate(L):
    """Output slice written in place, grad_out read from the slice, grad-input accumulates."""
    th = torch()
    inp = WL.make_inputs(L, gy_channels=L.OC + 4)
    ctot, off = L.OC + 4, 2
    d = desc_of(L, off, ctot)
    assert B.dwconv2d_plan_name(d, 0) == "plane"
    x, w = to_dev(inp.x), to_dev(inp.w)
    b = to_dev(inp.b) if inp.b is not None else None
    y = empty_dev((L.N, ctot, L.Ho, L.Wo), L.dtype, fill=-3.0)
    B.dwconv2d_fwd(d, x, w, b, y)
    yh = to_f64(y)
    assert np.all(yh[:, :off] == -3.0) and np.all(yh[:, off + L.OC:] == -3.0)
    cv = oconv(L, off=off, c_total=ctot)
    ry = oracle.fwd(cv, inp.x.f64, inp.w.f64, inp.b.f64 if inp.b is not None else None)
    assert_close(yh[:, off:off + L.OC], ry[:, off:off + L.OC], L.dtype, 9, "plane slice fwd")
    gy = to_dev(inp.gy)
    gx = empty_dev((L.N, L.C, L.H, L.W), L.dtype, fill=0.25)
    B.dwconv2d_bwd_data(d, gy, w, gx, 1)
    th.cuda.synchronize()
    rgx = oracle.bwd_data(cv, inp.gy.f64, inp.w.f64) + 0.25
    assert_close(to_f64(gx), rgx, L.dtype, 9, "plane accumulate bwd_data")
    gw = empty_dev((L.OC, L.k, L.k), L.dtype)
    ws, nb = ws_for(d)
    B.dwconv2d_bwd_weight(d, x, gy, gw, None, ws, nb)
    th.cuda.synchronize()
    rgw, _ = oracle.bwd_weight(cv, inp.x.f64, inp.gy.f64)
    assert_close(to_f64(gw), rgw, L.dtype, 9, "plane slice bwd_weight")


def test_no_bounded_wait_gave_up_at_end():
    assert B.dwconv_device_timeouts() == 0
