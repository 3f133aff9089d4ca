"""Pins for the fp64 oracle: each check ties it to something other than itself.

The pages print no output values, so the pins are the mathematics the
definition fixes (forward as in "Spatial Depthwise Convolution on the GPU
#3057", the forward binding with stride, padding, dilation, depth multiplier
and bias; the sliding window of the MegEngine article, "From convolution to
matrix multiplication"; the concatenated channel slices of the
DynamicConvolutionOperator README, "Solution"):

* brute force: the operator assembled as an explicit sparse matrix, one tap at
  a time with numpy fancy indexing (no nested output loop), on tiny shapes
  over every combination of stride, dilation, padding, multiplier;
* a float64 library cross-check (torch.nn.functional.conv2d with groups=C and
  autograd) -- used only to validate the oracle;
* a delta kernel reproduces the shifted, zero-padded input bit-exactly;
* an all-ones kernel equals a summed-area-table box sum (exact integers);
* a separable kernel equals a row pass then a column pass (exact dyadics);
* stride, dilation and multiplier reduce to simpler calls;
* adjoint identities for bwd_data and bwd_weight, an exact finite difference,
  an impulse input, and the bias gradient as a plain sum;
* channel slices outside [off, off + C*m) are left untouched.
"""
import itertools

import numpy as np
import pytest

import oracle
from oracle import Conv

RNG = np.random.default_rng(12345)


def rand(*shape):
    return RNG.standard_normal(shape)


def conv_cases():
    out = []
    for (kh, kw), s, d, m in itertools.product([(1, 1), (3, 3), (2, 3), (5, 5), (3, 1)],
                                               [1, 2, 3], [1, 2], [1, 2]):
        for ph, pw in [(0, 0), (kh // 2 * d, kw // 2 * d), (1, 2)]:
            cv = Conv(N=2, C=2, H=7, W=6, kh=kh, kw=kw, sh=s, sw=max(1, s - 1),
                      ph=ph, pw=pw, dh=d, dw=1 + (d > 1 and kw > 1), m=m)
            if cv.Ho >= 1 and cv.Wo >= 1:
                out.append(cv)
    return out


CASES = conv_cases()


def assemble_matrix(cv: Conv, w):
    """Dense matrix A with y_flat = A @ x_flat (slice of y only, no bias).

    Built tap by tap: for tap (a, b) of output channel oc, output (oh, ow)
    reads input (oh*sh - ph + a*dh, ow*sw - pw + b*dw) when that is inside.
    """
    Ho, Wo = cv.Ho, cv.Wo
    A = np.zeros((cv.N * cv.OC * Ho * Wo, cv.N * cv.C * cv.H * cv.W))
    oh, ow = np.meshgrid(np.arange(Ho), np.arange(Wo), indexing="ij")
    for n in range(cv.N):
        for oc in range(cv.OC):
            c = oc // cv.m
            for a in range(cv.kh):
                for b in range(cv.kw):
                    ih = oh * cv.sh - cv.ph + a * cv.dh
                    iw = ow * cv.sw - cv.pw + b * cv.dw
                    ok = (ih >= 0) & (ih < cv.H) & (iw >= 0) & (iw < cv.W)
                    rows = ((n * cv.OC + oc) * Ho + oh[ok]) * Wo + ow[ok]
                    cols = ((n * cv.C + c) * cv.H + ih[ok]) * cv.W + iw[ok]
                    np.add.at(A, (rows, cols), w[oc, a, b])
    return A


@pytest.mark.parametrize("cv", CASES[::3], ids=lambda c: f"k{c.kh}x{c.kw}s{c.sh}{c.sw}p{c.ph}{c.pw}d{c.dh}{c.dw}m{c.m}")
def test_brute_force_matrix(cv):
    x, w, b = rand(cv.N, cv.C, cv.H, cv.W), rand(cv.OC, cv.kh, cv.kw), rand(cv.OC)
    g = rand(cv.N, cv.OC, cv.Ho, cv.Wo)
    A = assemble_matrix(cv, w)
    y = oracle.fwd(cv, x, w, b)
    ref = (A @ x.ravel()).reshape(y.shape) + b[None, :, None, None]
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    gx = oracle.bwd_data(cv, g, w)
    np.testing.assert_allclose(gx.ravel(), A.T @ g.ravel(), rtol=1e-12, atol=1e-12)
    # weight gradient: impulse response in w, gw[e] = <A(e_w) x, g>
    gw, gb = oracle.bwd_weight(cv, x, g, want_w=True, want_b=True)
    ref_gw = np.zeros_like(w)
    for idx in itertools.product(range(cv.OC), range(cv.kh), range(cv.kw)):
        e = np.zeros_like(w)
        e[idx] = 1.0
        ref_gw[idx] = g.ravel() @ (assemble_matrix(cv, e) @ x.ravel())
    np.testing.assert_allclose(gw, ref_gw, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gb, g.sum(axis=(0, 2, 3)), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("cv", CASES, ids=lambda c: f"k{c.kh}x{c.kw}s{c.sh}{c.sw}p{c.ph}{c.pw}d{c.dh}{c.dw}m{c.m}")
def test_torch_float64_crosscheck(cv):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    x, w, b = rand(cv.N, cv.C, cv.H, cv.W), rand(cv.OC, cv.kh, cv.kw), rand(cv.OC)
    g = rand(cv.N, cv.OC, cv.Ho, cv.Wo)
    tx = torch.tensor(x, requires_grad=True)
    tw = torch.tensor(w.reshape(cv.OC, 1, cv.kh, cv.kw), requires_grad=True)
    tb = torch.tensor(b, requires_grad=True)
    ty = F.conv2d(tx, tw, tb, stride=(cv.sh, cv.sw), padding=(cv.ph, cv.pw),
                  dilation=(cv.dh, cv.dw), groups=cv.C)
    ty.backward(torch.tensor(g))
    np.testing.assert_allclose(oracle.fwd(cv, x, w, b), ty.detach().numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.bwd_data(cv, g, w), tx.grad.numpy(), rtol=1e-12, atol=1e-12)
    gw, gb = oracle.bwd_weight(cv, x, g, want_w=True, want_b=True)
    np.testing.assert_allclose(gw, tw.grad.numpy().reshape(w.shape), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gb, tb.grad.numpy(), rtol=1e-12, atol=1e-12)


def padded(x, ph, pw, extra=64):
    return np.pad(x, ((0, 0), (0, 0), (ph + extra, ph + extra), (pw + extra, pw + extra)))


@pytest.mark.parametrize("cv", [c for c in CASES if c.kh * c.kw > 1][::2],
                         ids=lambda c: f"k{c.kh}x{c.kw}s{c.sh}{c.sw}p{c.ph}{c.pw}d{c.dh}{c.dw}m{c.m}")
def test_delta_kernel_shifts_input_exactly(cv):
    x = rand(cv.N, cv.C, cv.H, cv.W)
    E = 64
    xp = padded(x, cv.ph, cv.pw, E)
    for a, b in [(0, 0), (cv.kh - 1, cv.kw - 1), (cv.kh // 2, 0)]:
        w = np.zeros((cv.OC, cv.kh, cv.kw))
        w[:, a, b] = 1.0
        y = oracle.fwd(cv, x, w)
        r0 = E + a * cv.dh  # padded row index of oh = 0 for tap a
        c0 = E + b * cv.dw
        sh = xp[:, :, r0:r0 + cv.sh * cv.Ho:cv.sh, c0:c0 + cv.sw * cv.Wo:cv.sw]
        ref = np.repeat(sh, cv.m, axis=1)
        assert np.array_equal(y, ref)


@pytest.mark.parametrize("k,s,p", [(3, 1, 1), (5, 2, 2), (4, 1, 0), (7, 3, 1), (3, 2, 0)])
def test_ones_kernel_is_box_sum(k, s, p):
    cv = Conv(N=2, C=3, H=11, W=9, kh=k, kw=k, sh=s, sw=s, ph=p, pw=p)
    x = RNG.integers(-50, 50, size=(cv.N, cv.C, cv.H, cv.W)).astype(np.float64)
    y = oracle.fwd(cv, x, np.ones((cv.OC, k, k)))
    xp = np.pad(x, ((0, 0), (0, 0), (p, p), (p, p)))
    S = np.zeros((cv.N, cv.C, xp.shape[2] + 1, xp.shape[3] + 1))
    S[:, :, 1:, 1:] = xp.cumsum(2).cumsum(3)
    r = np.arange(cv.Ho)[:, None] * s
    c = np.arange(cv.Wo)[None, :] * s
    box = S[:, :, r + k, c + k] - S[:, :, r, c + k] - S[:, :, r + k, c] + S[:, :, r, c]
    assert np.array_equal(y, box)


@pytest.mark.parametrize("kh,kw,s,d,p", [(3, 3, 1, 1, 1), (5, 3, 2, 1, 2), (3, 5, 1, 2, 2), (7, 7, 2, 3, 4)])
def test_separable_kernel_is_two_1d_passes(kh, kw, s, d, p):
    cv = Conv(N=1, C=2, H=13, W=12, kh=kh, kw=kw, sh=s, sw=s, ph=p, pw=p, dh=d, dw=d)
    x = RNG.integers(-8, 8, size=(cv.N, cv.C, cv.H, cv.W)) / 4.0
    u = RNG.integers(-4, 4, size=(cv.C, kh)) / 2.0
    v = RNG.integers(-4, 4, size=(cv.C, kw)) / 2.0
    w = u[:, :, None] * v[:, None, :]
    y = oracle.fwd(cv, x, w)
    xp = np.pad(x, ((0, 0), (0, 0), (p, p), (p, p)))
    rowpass = sum(v[None, :, b, None, None] * xp[:, :, :, b * d:b * d + s * cv.Wo:s] for b in range(kw))
    ref = sum(u[None, :, a, None, None] * rowpass[:, :, a * d:a * d + s * cv.Ho:s, :] for a in range(kh))
    assert np.array_equal(y, ref)


def test_unit_kernel_is_scale():
    cv = Conv(N=2, C=4, H=5, W=6, kh=1, kw=1)
    x = rand(2, 4, 5, 6)
    w = rand(4, 1, 1)
    assert np.array_equal(oracle.fwd(cv, x, w), x * w[None, :, :, :])


@pytest.mark.parametrize("s,d,p", [(2, 1, 1), (3, 2, 2), (2, 3, 0)])
def test_stride_is_subsampled_stride1(s, d, p):
    base = dict(N=2, C=3, H=15, W=14, kh=3, kw=3, ph=p, pw=p, dh=d, dw=d)
    x, w = rand(2, 3, 15, 14), rand(3, 3, 3)
    y1 = oracle.fwd(Conv(**base), x, w)
    ys = oracle.fwd(Conv(**base, sh=s, sw=s), x, w)
    assert np.array_equal(ys, y1[:, :, ::s, ::s])


@pytest.mark.parametrize("k,d", [(3, 2), (3, 5), (5, 3), (2, 4)])
def test_dilation_is_zero_inserted_kernel(k, d):
    x, w = rand(1, 2, 19, 17), rand(2, k, k)
    K = d * (k - 1) + 1
    wz = np.zeros((2, K, K))
    wz[:, ::d, ::d] = w
    p = (K - 1) // 2
    yd = oracle.fwd(Conv(N=1, C=2, H=19, W=17, kh=k, kw=k, dh=d, dw=d, ph=p, pw=p), x, w)
    yz = oracle.fwd(Conv(N=1, C=2, H=19, W=17, kh=K, kw=K, ph=p, pw=p), x, wz)
    assert np.array_equal(yd, yz)


@pytest.mark.parametrize("m", [2, 3])
def test_multiplier_is_repeated_input(m):
    x, w, b = rand(2, 3, 9, 8), rand(3 * m, 3, 3), rand(3 * m)
    ym = oracle.fwd(Conv(N=2, C=3, H=9, W=8, ph=1, pw=1, m=m), x, w, b)
    y1 = oracle.fwd(Conv(N=2, C=3 * m, H=9, W=8, ph=1, pw=1), np.repeat(x, m, axis=1), w, b)
    assert np.array_equal(ym, y1)
    # bwd_data with a multiplier sums the m filters of each input channel
    g = rand(2, 3 * m, 9, 8)
    gx1 = oracle.bwd_data(Conv(N=2, C=3 * m, H=9, W=8, ph=1, pw=1), g, w)
    gxm = oracle.bwd_data(Conv(N=2, C=3, H=9, W=8, ph=1, pw=1, m=m), g, w)
    np.testing.assert_allclose(gxm, gx1.reshape(2, 3, m, 9, 8).sum(axis=2), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("cv", CASES[1::4], ids=lambda c: f"k{c.kh}x{c.kw}s{c.sh}{c.sw}p{c.ph}{c.pw}d{c.dh}{c.dw}m{c.m}")
def test_adjoint_identities(cv):
    x, w = rand(cv.N, cv.C, cv.H, cv.W), rand(cv.OC, cv.kh, cv.kw)
    g = rand(cv.N, cv.OC, cv.Ho, cv.Wo)
    lhs = np.vdot(oracle.fwd(cv, x, w), g)
    assert abs(lhs - np.vdot(x, oracle.bwd_data(cv, g, w))) <= 1e-12 * max(1.0, abs(lhs)) * 10
    gw, _ = oracle.bwd_weight(cv, x, g)
    assert abs(lhs - np.vdot(w, gw)) <= 1e-12 * max(1.0, abs(lhs)) * 10


def test_weight_gradient_finite_difference():
    cv = Conv(N=2, C=3, H=9, W=10, kh=3, kw=5, sh=2, sw=1, ph=1, pw=2, dh=2, dw=1, m=2)
    x, w = rand(2, 3, 9, 10), rand(6, 3, 5)
    g = rand(2, 6, cv.Ho, cv.Wo)
    gw, _ = oracle.bwd_weight(cv, x, g)
    L = lambda ww: np.vdot(oracle.fwd(cv, x, ww), g)
    for idx in [(0, 0, 0), (3, 1, 2), (5, 2, 4), (2, 0, 3)]:
        e = np.zeros_like(w)
        e[idx] = 1.0   # L is linear in w, so step 1 is exact up to rounding
        fd = (L(w + e) - L(w - e)) / 2.0
        assert abs(fd - gw[idx]) <= 1e-11 * max(1.0, abs(gw[idx]))


def test_impulse_input_gives_gradient_window():
    cv = Conv(N=2, C=2, H=8, W=9, kh=3, kw=3, sh=1, sw=1, ph=1, pw=1, m=2)
    g = rand(2, 4, cv.Ho, cv.Wo)
    n, c, i, j = 1, 1, 4, 3
    x = np.zeros((2, 2, 8, 9))
    x[n, c, i, j] = 1.0
    gw, _ = oracle.bwd_weight(cv, x, g)
    for oc in range(4):
        for a in range(3):
            for b in range(3):
                want = g[n, oc, i + 1 - a, j + 1 - b] if oc // 2 == c else 0.0
                assert gw[oc, a, b] == want


def test_slice_leaves_other_channels_untouched():
    cv = Conv(N=2, C=3, H=6, W=7, ph=1, pw=1, m=2, off=5, c_total=13)
    x, w, b = rand(2, 3, 6, 7), rand(6, 3, 3), rand(6)
    y = np.full((2, 13, cv.Ho, cv.Wo), 7.25)
    oracle.fwd(cv, x, w, b, y=y)
    assert np.all(y[:, :5] == 7.25) and np.all(y[:, 11:] == 7.25)
    dense = oracle.fwd(Conv(N=2, C=3, H=6, W=7, ph=1, pw=1, m=2), x, w, b)
    assert np.array_equal(y[:, 5:11], dense)
    # the backward passes read the same slice of gy
    g = rand(2, 13, cv.Ho, cv.Wo)
    dcv = Conv(N=2, C=3, H=6, W=7, ph=1, pw=1, m=2)
    assert np.array_equal(oracle.bwd_data(cv, g, w), oracle.bwd_data(dcv, g[:, 5:11].copy(), w))
    gw, gb = oracle.bwd_weight(cv, x, g, want_b=True)
    gw2, gb2 = oracle.bwd_weight(dcv, x, g[:, 5:11].copy(), want_b=True)
    assert np.array_equal(gw, gw2) and np.array_equal(gb, gb2)


def test_multi_branch_is_concat_and_sum():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    N, C, H, W = 1, 2, 12, 11
    brs = [Conv(N=N, C=C, H=H, W=W, ph=d, pw=d, dh=d, dw=d, off=i * C, c_total=3 * C)
           for i, d in enumerate((1, 3, 5))]
    x = rand(N, C, H, W)
    ws = [rand(C, 3, 3) for _ in brs]
    bs = [rand(C) for _ in brs]
    y = oracle.fwd_multi(brs, x, ws, bs)
    tx = torch.tensor(x, requires_grad=True)
    parts = [F.conv2d(tx, torch.tensor(ws[i][:, None]), torch.tensor(bs[i]), padding=d,
                      dilation=d, groups=C) for i, d in enumerate((1, 3, 5))]
    ty = torch.cat(parts, dim=1)
    np.testing.assert_allclose(y, ty.detach().numpy(), rtol=1e-12, atol=1e-12)
    g = rand(*y.shape)
    ty.backward(torch.tensor(g))
    np.testing.assert_allclose(oracle.bwd_data_multi(brs, g, ws), tx.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_zero_batch_and_degenerate_output():
    cv = Conv(N=0, C=3, H=5, W=5, ph=1, pw=1)
    y = oracle.fwd(cv, np.zeros((0, 3, 5, 5)), rand(3, 3, 3))
    assert y.shape == (0, 3, 5, 5)
    # kernel exactly as large as the padded input: a 1x1 output
    cv = Conv(N=1, C=1, H=3, W=3, kh=5, kw=5, ph=1, pw=1)
    assert (cv.Ho, cv.Wo) == (1, 1)
    x = rand(1, 1, 3, 3)
    w = rand(1, 5, 5)
    assert abs(oracle.fwd(cv, x, w)[0, 0, 0, 0] - np.sum(w[0, 1:4, 1:4] * x[0, 0])) < 1e-12


# ---- fused forward epilogue -------------------------------------------------

@pytest.mark.parametrize("act", ["none", "relu", "relu6"])
@pytest.mark.parametrize("cv", [CASES[1], CASES[40], CASES[-5]],
                         ids=lambda c: f"k{c.kh}x{c.kw}s{c.sh}{c.sw}p{c.ph}{c.pw}d{c.dh}{c.dw}m{c.m}")
def test_epilogue_is_batch_norm_then_activation(cv, act):
    """A folded inference batch norm plus activation equals torch's float64
    conv2d -> batch_norm(eval) -> relu / hardtanh(0, 6) on the same values."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(cv.kh * 100 + cv.sh * 10 + cv.m)
    x, w, b = 3.0 * rng.standard_normal((cv.N, cv.C, cv.H, cv.W)), rng.standard_normal((cv.OC, cv.kh, cv.kw)), \
        rng.standard_normal(cv.OC)
    gamma, beta, mean = rng.standard_normal(cv.OC), rng.standard_normal(cv.OC), rng.standard_normal(cv.OC)
    var, eps = rng.uniform(0.5, 2.0, cv.OC), 1e-5
    scale = gamma / np.sqrt(var + eps)
    shift = beta - mean * scale
    ty = F.conv2d(torch.tensor(x), torch.tensor(w.reshape(cv.OC, 1, cv.kh, cv.kw)), torch.tensor(b),
                  stride=(cv.sh, cv.sw), padding=(cv.ph, cv.pw), dilation=(cv.dh, cv.dw), groups=cv.C)
    ty = F.batch_norm(ty, torch.tensor(mean), torch.tensor(var), torch.tensor(gamma), torch.tensor(beta),
                      training=False, eps=eps)
    if act == "relu":
        ty = F.relu(ty)
    elif act == "relu6":
        ty = F.hardtanh(ty, 0.0, 6.0)
    got = oracle.fwd_epilogue(cv, x, w, b, scale, shift, act)
    np.testing.assert_allclose(got, ty.numpy(), rtol=1e-12, atol=1e-12)


def test_epilogue_identity_and_activation_cases():
    """No scale, shift or activation is the plain forward (bit-exact); a
    negated delta kernel with ReLU gives max(-x, 0); ReLU6 of a constant plane
    of 7 under the same kernel and shift 13 gives 6 everywhere."""
    cv = Conv(N=2, C=3, H=5, W=6, kh=3, kw=3, ph=1, pw=1, m=2, off=1, c_total=8)
    x, w = rand(cv.N, cv.C, cv.H, cv.W), rand(cv.OC, 3, 3)
    y0 = oracle.fwd(cv, x, w)
    assert np.array_equal(oracle.fwd_epilogue(cv, x, w), y0)
    neg = np.zeros((cv.OC, 3, 3))
    neg[:, 1, 1] = -1.0
    y = oracle.fwd_epilogue(cv, x, neg, act="relu")
    want = np.maximum(-np.repeat(x, cv.m, axis=1), 0.0)
    assert np.array_equal(y[:, 1:1 + cv.OC], want)
    assert not y[:, 0].any() and not y[:, 1 + cv.OC:].any()
    y6 = oracle.fwd_epilogue(cv, np.full(x.shape, 7.0), neg, shift=np.full(cv.OC, 13.0), act="relu6")
    assert np.array_equal(y6[:, 1:1 + cv.OC], np.full((cv.N, cv.OC, cv.H, cv.W), 6.0))
    # ReLU6 of a ramp through the identity kernel: clipped below and above
    ramp = np.linspace(-4.0, 10.0, cv.N * cv.C * cv.H * cv.W).reshape(x.shape)
    yr = oracle.fwd_epilogue(cv, ramp, -neg, act="relu6")
    assert np.array_equal(yr[:, 1:1 + cv.OC], np.clip(np.repeat(ramp, cv.m, axis=1), 0.0, 6.0))
    # scale only: channel oc multiplied by scale[oc], exactly for powers of two
    sc = 2.0 ** np.arange(cv.OC)
    ys = oracle.fwd_epilogue(cv, x, w, scale=sc)
    assert np.array_equal(ys[:, 1:1 + cv.OC], y0[:, 1:1 + cv.OC] * sc[None, :, None, None])


# ---- depthwise-separable block ----------------------------------------------

@pytest.mark.parametrize("cv,cout", [(Conv(N=2, C=6, H=9, W=8, kh=3, kw=3, ph=1, pw=1), 10),
                                     (Conv(N=1, C=4, H=11, W=11, kh=3, kw=3, sh=2, sw=2, ph=1, pw=1), 3),
                                     (Conv(N=2, C=3, H=8, W=7, kh=5, kw=5, ph=2, pw=2, m=2), 5)],
                         ids=["s1", "s2", "k5m2"])
def test_separable_block_is_torch_sequence(cv, cout):
    """The block equals torch's float64 depthwise conv2d -> batch_norm(eval)
    -> ReLU6 -> 1x1 conv2d -> batch_norm(eval) -> ReLU on the same values."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(cv.C * 10 + cout)
    x = 3.0 * rng.standard_normal((cv.N, cv.C, cv.H, cv.W))
    wd, wp = rng.standard_normal((cv.OC, cv.kh, cv.kw)), rng.standard_normal((cout, cv.OC))
    bn = lambda c: (rng.standard_normal(c), rng.standard_normal(c), rng.standard_normal(c),
                    rng.uniform(0.5, 2.0, c))
    g1, b1, m1, v1 = bn(cv.OC)
    g2, b2, m2, v2 = bn(cout)
    eps = 1e-5
    s1 = g1 / np.sqrt(v1 + eps)
    s2 = g2 / np.sqrt(v2 + eps)
    T = torch.tensor
    z = F.conv2d(T(x), T(wd.reshape(cv.OC, 1, cv.kh, cv.kw)), stride=(cv.sh, cv.sw), padding=(cv.ph, cv.pw),
                 dilation=(cv.dh, cv.dw), groups=cv.C)
    z = F.hardtanh(F.batch_norm(z, T(m1), T(v1), T(g1), T(b1), training=False, eps=eps), 0.0, 6.0)
    y = F.conv2d(z, T(wp.reshape(cout, cv.OC, 1, 1)))
    y = F.relu(F.batch_norm(y, T(m2), T(v2), T(g2), T(b2), training=False, eps=eps))
    got = oracle.separable(cv, x, wd, s1, b1 - m1 * s1, "relu6", wp, s2, b2 - m2 * s2, "relu")
    np.testing.assert_allclose(got, y.numpy(), rtol=1e-12, atol=1e-12)


def test_separable_block_special_cases():
    """Identity pointwise weights give the depthwise stage unchanged (bit for
    bit); a row of ones sums the channels exactly (dyadic values); a
    permutation moves whole channels."""
    cv = Conv(N=2, C=5, H=7, W=6, kh=3, kw=3, ph=1, pw=1)
    x = np.round(RNG.standard_normal((cv.N, cv.C, cv.H, cv.W)) * 64) / 64
    wd = np.round(RNG.standard_normal((cv.C, 3, 3)) * 16) / 16
    z = oracle.fwd_epilogue(cv, x, wd, act="relu")
    assert np.array_equal(oracle.separable(cv, x, wd, dw_act="relu", w_pw=np.eye(cv.C)), z)
    ones = np.ones((1, cv.C))
    assert np.array_equal(oracle.separable(cv, x, wd, dw_act="relu", w_pw=ones)[:, 0], z.sum(axis=1))
    perm = np.eye(cv.C)[[3, 0, 4, 1, 2]]
    assert np.array_equal(oracle.separable(cv, x, wd, w_pw=perm), oracle.fwd(cv, x, wd)[:, [3, 0, 4, 1, 2]])
    # the second epilogue acts per output channel of the pointwise step
    sc = np.array([2.0, -1.0])
    y = oracle.separable(cv, x, wd, w_pw=np.vstack([ones, ones]), pw_scale=sc, pw_shift=np.array([0.5, 0.25]),
                         pw_act="relu")
    s = oracle.fwd(cv, x, wd).sum(axis=1)
    assert np.array_equal(y[:, 0], np.maximum(2.0 * s + 0.5, 0.0))
    assert np.array_equal(y[:, 1], np.maximum(-s + 0.25, 0.0))
