"""Filter-cache (kernel-im2col) path of the tensor-core large-kernel forward
and grad-input against the fp64 oracle: the cache built once per filter, row
widths 8..64, one and several tile groups per channel, batches split into
chunks of 64 samples with a ragged last chunk, ragged tiles, non-square
filters with unequal vertical padding, output slices, accumulation, and
agreement with the uncached tensor-core kernels."""
import numpy as np
import pytest

import oracle
from depthwise_convolution_dwconv2d_gb300 import binding as B
from depthwise_convolution_dwconv2d_gb300 import synth, workloads as WL
from dw_testutil import assert_close, empty_dev, oconv, to_dev, to_f64, torch
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


def cache_for(d, pass_, w):
    th = torch()
    nbytes = B.dwconv2d_filter_cache_size(d, pass_)
    assert nbytes > 0
    cache = th.empty(nbytes // 2, dtype=th.float16, device="cuda")
    B.dwconv2d_filter_cache_build(d, pass_, w, cache)
    return cache


def run_cached(L, inp, d, gy_t=None, y_shape=None):
    """Cached fwd and bwd_data on the GPU; float64 results."""
    th = torch()
    x, w = to_dev(inp.x), to_dev(inp.w)
    b = to_dev(inp.b) if inp.b is not None else None
    gy = to_dev(inp.gy) if gy_t is None else gy_t
    y = empty_dev(y_shape or (L.N, L.OC, L.Ho, L.Wo), L.dtype, fill=0)
    B.dwconv2d_fwd_cached(d, x, cache_for(d, 0, w), b, y)
    gx = empty_dev((L.N, L.C, L.H, L.W), L.dtype)
    B.dwconv2d_bwd_data_cached(d, gy, cache_for(d, 1, w), gx, 0)
    th.cuda.synchronize()
    return to_f64(y), to_f64(gx)


CASES = [
    WL.Layer(N=3, C=5, H=32, W=32, k=31, p=15, bias=True, dtype="f16"),
    WL.Layer(N=20, C=3, H=16, W=16, k=13, p=6, dtype="bf16"),
    WL.Layer(N=2, C=4, H=17, W=8, k=9, p=4, bias=True, dtype="f16"),
    WL.Layer(N=2, C=3, H=64, W=64, k=21, p=10, dtype="f16"),
    WL.Layer(N=130, C=2, H=32, W=32, k=15, p=7, dtype="bf16"),
    WL.Layer(N=300, C=2, H=8, W=8, k=11, p=5, bias=True, dtype="bf16"),
    WL.Layer(N=5, C=3, H=45, W=32, k=21, p=10, dtype="f16"),
    WL.Layer(N=33, C=2, H=96, W=64, k=13, p=6, bias=True, dtype="bf16"),
    WL.Layer(N=1, C=3, H=32, W=32, k=27, p=13, bias=True, dtype="f16"),
    WL.Layer(N=1, C=2, H=16, W=64, k=21, p=10, dtype="bf16"),
]
IDS = ["k31f16_W32", "k13bf16_W16", "k9f16_W8_raggedM", "k21f16_W64_groups", "k15bf16_N130_chunks",
       "k11bf16_N300", "k21f16_H45", "k13bf16_W64_H96", "k27f16_N1", "k21bf16_N1_W64"]


def check(L, inp, label):
    d = B.make_desc(**L.desc_kwargs())
    y, gx = run_cached(L, inp, d)
    cv = oconv(L)
    taps = L.k * L.k
    b64 = inp.b.f64 if inp.b is not None else None
    assert_close(y, oracle.fwd(cv, inp.x.f64, inp.w.f64, b64), L.dtype, taps, f"{label} cached fwd")
    assert_close(gx, oracle.bwd_data(cv, inp.gy.f64, inp.w.f64), L.dtype, taps, f"{label} cached bwd_data")


@pytest.mark.parametrize("L", CASES, ids=IDS)
def test_cached_vs_oracle(L):
    check(L, WL.make_inputs(L), L.label())


def test_cached_non_square_filter_and_unequal_vertical_padding():
    """kh != kw, pad_h != (kh - 1) / 2 (Ho != H); only the row width must match."""
    th = torch()
    N, C, H, W, kh, kw, ph, pw = 3, 4, 40, 32, 21, 9, 3, 4
    cv = Conv(N=N, C=C, H=H, W=W, kh=kh, kw=kw, sh=1, sw=1, ph=ph, pw=pw, dh=1, dw=1, m=1)
    Ho = H + 2 * ph - kh + 1
    x = synth.uniform_tensor((N, C, H, W), "f16", 7, synth.STREAM_X)
    w = synth.normal_tensor((C, kh, kw), "f16", 7, synth.STREAM_W, std=0.1)
    b = synth.normal_tensor((C,), "f16", 7, synth.STREAM_B, std=0.3)
    gy = synth.normal_tensor((N, C, Ho, W), "f16", 7, synth.STREAM_GY)
    d = B.make_desc(N, C, H, W, (kh, kw), 1, (ph, pw), dtype="f16")
    wd = to_dev(w)
    y = empty_dev((N, C, Ho, W), "f16")
    B.dwconv2d_fwd_cached(d, to_dev(x), cache_for(d, 0, wd), to_dev(b), y)
    gx = empty_dev((N, C, H, W), "f16")
    B.dwconv2d_bwd_data_cached(d, to_dev(gy), cache_for(d, 1, wd), gx, 0)
    th.cuda.synchronize()
    assert_close(to_f64(y), oracle.fwd(cv, x.f64, w.f64, b.f64), "f16", kh * kw, "non-square fwd")
    assert_close(to_f64(gx), oracle.bwd_data(cv, gy.f64, w.f64), "f16", kh * kw, "non-square bwd_data")


def test_cached_slices_guard_bands_and_accumulate():
    """y slice of a wider tensor (other channels untouched), gy read from a
    slice, gx accumulated into."""
    th = torch()
    L = WL.Layer(N=4, C=3, H=32, W=32, k=17, p=8, bias=True, dtype="bf16")
    off, ctot = 2, 7
    inp = WL.make_inputs(L, gy_channels=ctot)
    d = B.make_desc(**L.desc_kwargs(), out_c_offset=off, out_c_total=ctot)
    w = to_dev(inp.w)
    y = empty_dev((L.N, ctot, L.Ho, L.Wo), "bf16", fill=5.0)
    B.dwconv2d_fwd_cached(d, to_dev(inp.x), cache_for(d, 0, w), to_dev(inp.b), y)
    gx0 = synth.normal_tensor((L.N, L.C, L.H, L.W), "bf16", 9, synth.STREAM_X)
    gx = to_dev(gx0)
    B.dwconv2d_bwd_data_cached(d, to_dev(inp.gy), cache_for(d, 1, w), gx, 1)
    th.cuda.synchronize()
    yh = to_f64(y)
    cv = oconv(L, off=off, c_total=ctot)
    ref = oracle.fwd(cv, inp.x.f64, inp.w.f64, inp.b.f64)
    sl = slice(off, off + L.C)
    assert_close(yh[:, sl], ref[:, sl], "bf16", L.k * L.k, "sliced fwd")
    assert np.all(yh[:, :off] == 5.0) and np.all(yh[:, off + L.C:] == 5.0)
    rgx = oracle.bwd_data(cv, inp.gy.f64, inp.w.f64) + gx0.f64
    assert_close(to_f64(gx), rgx, "bf16", L.k * L.k, "accumulated bwd_data")


def test_cached_matches_uncached_and_is_deterministic():
    th = torch()
    L = CASES[0]
    inp = WL.make_inputs(L, seed=5)
    d = B.make_desc(**L.desc_kwargs())
    x, w, b = to_dev(inp.x), to_dev(inp.w), to_dev(inp.b)
    cache = cache_for(d, 0, w)
    outs = []
    for _ in range(2):
        y = empty_dev((L.N, L.C, L.Ho, L.Wo), L.dtype)
        B.dwconv2d_fwd_cached(d, x, cache, b, y)
        outs.append(y)
    y0 = empty_dev((L.N, L.C, L.Ho, L.Wo), L.dtype)
    assert B.dwconv2d_plan_name(d, 0) == "ibgemm"
    B.dwconv2d_fwd(d, x, w, b, y0)
    th.cuda.synchronize()
    assert th.equal(outs[0], outs[1])
    assert_close(to_f64(outs[0]), to_f64(y0), L.dtype, L.k * L.k, "cached vs uncached")


def test_cache_rebuild_follows_the_filter():
    """A cache rebuilt for a new filter gives that filter's result; one cache
    serves another batch size and height of the same layer."""
    th = torch()
    L = WL.Layer(N=2, C=3, H=32, W=32, k=31, p=15, dtype="f16")
    i1, i2 = WL.make_inputs(L, seed=1), WL.make_inputs(L, seed=2)
    d = B.make_desc(**L.desc_kwargs())
    cache = cache_for(d, 0, to_dev(i1.w))
    B.dwconv2d_filter_cache_build(d, 0, to_dev(i2.w), cache)
    y = empty_dev((L.N, L.C, L.Ho, L.Wo), "f16")
    B.dwconv2d_fwd_cached(d, to_dev(i1.x), cache, None, y)
    L2 = WL.Layer(N=7, C=3, H=20, W=32, k=31, p=15, dtype="f16")
    x2 = WL.make_x(L2, seed=4)
    d2 = B.make_desc(**L2.desc_kwargs())
    assert B.dwconv2d_filter_cache_size(d2, 0) == B.dwconv2d_filter_cache_size(d, 0)
    y2 = empty_dev((L2.N, L2.C, L2.Ho, L2.Wo), "f16")
    B.dwconv2d_fwd_cached(d2, to_dev(x2), cache, None, y2)
    th.cuda.synchronize()
    assert_close(to_f64(y), oracle.fwd(oconv(L), i1.x.f64, i2.w.f64, None), "f16", L.k * L.k, "rebuilt cache")
    assert_close(to_f64(y2), oracle.fwd(oconv(L2), x2.f64, i2.w.f64, None), "f16", L.k * L.k, "other N and H")


_FULL = {}


def _full_inputs(L):
    """x and grad_out of a full-size layer depend only on (H, dtype) here;
    keep the most recent pair."""
    key = (L.H, L.dtype)
    if key not in _FULL:
        _FULL.clear()
        _FULL[key] = WL.make_inputs(WL.Layer(N=L.N, C=L.C, H=L.H, W=L.W, k=1, p=0, dtype=L.dtype))
    return _FULL[key]


@pytest.mark.parametrize("L", [L for L in WL.largek_infer() if L.H in (32, 64) and (L.H == 32 or L.k <= 21)],
                         ids=lambda L: L.name)
def test_cached_full_size_sampled(L):
    """The benchmark's full-size layers (64 x 384) in the launch configuration
    the bench times: cached forward and grad-input, oracle on sampled planes
    (edge and interior samples and channels: the persistent units straddle
    channels and tile groups)."""
    th = torch()
    d = B.make_desc(**L.desc_kwargs())
    assert B.dwconv2d_filter_cache_size(d, 0) > 0
    inp = _full_inputs(L)
    w = synth.normal_tensor((L.OC, L.k, L.k), L.dtype, 0, synth.STREAM_W, std=1.0 / L.k)
    wd = to_dev(w)
    y = empty_dev((L.N, L.C, L.Ho, L.Wo), L.dtype)
    B.dwconv2d_fwd_cached(d, to_dev(inp.x), cache_for(d, 0, wd), None, y)
    gx = empty_dev((L.N, L.C, L.H, L.W), L.dtype)
    B.dwconv2d_bwd_data_cached(d, to_dev(inp.gy), cache_for(d, 1, wd), gx, 0)
    th.cuda.synchronize()
    nsel, csel = [0, 31, 63], [0, 1, 191, 383]
    cv = oconv(L, N=len(nsel), C=len(csel))
    xs = inp.x.f64[np.ix_(nsel, csel)]
    gys = inp.gy.f64[np.ix_(nsel, csel)]
    ws = w.f64[csel]
    taps = L.k * L.k
    assert_close(to_f64(y)[np.ix_(nsel, csel)], oracle.fwd(cv, xs, ws, None), L.dtype, taps, f"{L.name} cached fwd")
    assert_close(to_f64(gx)[np.ix_(nsel, csel)], oracle.bwd_data(cv, gys, ws), L.dtype, taps,
                 f"{L.name} cached bwd_data")


def test_no_bounded_wait_gave_up_after_cached_calls():
    assert B.dwconv_device_timeouts() == 0
