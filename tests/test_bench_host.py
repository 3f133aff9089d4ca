"""Host-side work counts of the bench, against closed forms (no GPU).

The roofline counts valid taps (padded taps multiply zeros and need not be
computed); the dense count (every output times every tap) is reported beside
it. For a same-padded odd filter the valid taps of one axis are
sum_o [min(k, n + p - o) - max(0, p - o)], so the 2-D valid/dense ratio is
that sum squared over (n * k)^2.
"""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _layer(bench, workload, label):
    return next(i for i in bench.build_workload(workload) if i.label() == label)


def _ratio(bench, item):
    valid = sum(c[2] for c in bench.layer_calls(item))
    return valid / bench.dense_fma(item)


@pytest.mark.parametrize("H,k", [(32, 31), (48, 21), (64, 31), (64, 13)])
def test_large_kernel_valid_over_dense(bench, H, k):
    p = k // 2
    axis = sum(min(k, H + p - o) - max(0, p - o) for o in range(H))
    # 32 x 32, k = 31: 752 of 992 taps per axis -> 0.575; 64 x 64: 1744 of 1984 -> 0.773
    assert _ratio(bench, _layer(bench, "largek", f"lk_H{H}_k{k}_f32")) == pytest.approx((axis / (H * k)) ** 2, rel=1e-12)


def test_known_ratios(bench):
    assert _ratio(bench, _layer(bench, "largek", "lk_H32_k31_f32")) == pytest.approx(0.5747, abs=1e-4)
    assert _ratio(bench, _layer(bench, "largek", "lk_H64_k31_f32")) == pytest.approx(0.7727, abs=1e-4)
    # 3x3 stride 2 pad 1 on 7 x 7 (4 x 4 outputs): output o reads inputs 2o-1 .. 2o+1, so per
    # axis 2 + 3 + 3 + 2 = 10 of 12 taps are inside the plane (input -1 and input 7 are not)
    assert _ratio(bench, _layer(bench, "mobilenet", "mb_C1024_H7_s2")) == pytest.approx((10 / 12) ** 2, rel=1e-12)
    # 5 x 5, pad 2 on 28 x 28: per axis 28 * 5 - 2 * (1 + 2) = 134 of 140
    assert _ratio(bench, _layer(bench, "multiplier", "mult_C256_H28_k5_m2")) == pytest.approx((134 / 140) ** 2,
                                                                                            rel=1e-12)


def test_dense_counts_every_pass(bench):
    L = _layer(bench, "mobilenet", "mb_C128_H56_s1")
    # fwd, bwd_data and bwd_weight each touch N * C * Ho * Wo * 9 taps
    assert bench.dense_fma(L) == 3 * 64 * 128 * 56 * 56 * 9
