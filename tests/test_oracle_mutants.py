"""Planted mistakes: each mutant of the oracle must fail the pin suite.

A mutant is a copy of oracle/dwconv_oracle.c with one plausible slip (a
wrong sign, a flipped or transposed kernel, a dropped term, a wrong channel
mapping, a dropped divisibility test), compiled to a temporary library and
loaded by the pin tests through DWCONV_ORACLE_LIB. The mistakes live only in
the temporary copy, on the CPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "dwconv_oracle.c")

MUTANTS = {
    "fwd_pad_sign": ("const int64_t ih = oh * d->sh - d->ph + a * d->dh;\n          if (ih < 0 || ih >= d->H) continue;\n          for",
                     "const int64_t ih = oh * d->sh + d->ph + a * d->dh;\n          if (ih < 0 || ih >= d->H) continue;\n          for"),
    "fwd_kernel_flipped": ("acc += wp[a * d->kw + b] * xp[ih * d->W + iw];",
                           "acc += wp[(d->kh - 1 - a) * d->kw + (d->kw - 1 - b)] * xp[ih * d->W + iw];"),
    "fwd_channel_map": ("const int64_t n = t / OC, oc = t % OC, c = oc / d->m;",
                        "const int64_t n = t / OC, oc = t % OC, c = oc % d->C;"),
    "fwd_bias_dropped": ("if (bias) acc += bias[oc];", ""),
    "fwd_slice_offset_dropped": ("kw;\n    double* yp = y + (n * d->c_total + d->off + oc) * Ho * Wo;",
                                 "kw;\n    double* yp = y + (n * d->c_total + oc) * Ho * Wo;"),
    "bwd_data_no_divisibility": ("if (num_h < 0 || num_h % d->sh != 0) continue;",
                                 "if (num_h < 0) continue;"),
    "bwd_data_dilation_sign": ("const int64_t num_w = iw + d->pw - b * d->dw;",
                               "const int64_t num_w = iw + d->pw + b * d->dw - 2 * d->pw;"),
    "bwd_weight_tap_transposed": ("gw[(oc * d->kh + a) * d->kw + b] = acc;",
                                  "gw[(oc * d->kw + b) * d->kh + a] = acc;"),
    "bwd_weight_stride_dropped": ("const int64_t iw = ow * d->sw - d->pw + b * d->dw;\n                if",
                                  "const int64_t iw = ow - d->pw + b * d->dw;\n                if"),
    "epi_shift_inside_scale": ("double v = sc * yp[i] + sh;", "double v = sc * (yp[i] + sh);"),
    "epi_relu6_uncapped": ("if (act == 2) v = v < 6.0 ? v : 6.0;", ""),
    "epi_scale_by_input_channel": ("const double sc = scale ? scale[oc] : 1.0;",
                                   "const double sc = scale ? scale[oc / d->m] : 1.0;"),
    "pw_weight_transposed": ("const double wv = wp[co * cin + ci];", "const double wv = wp[ci * cout + co];"),
    "pw_channel_dropped": ("for (int64_t ci = 0; ci < cin; ++ci) {\n      const double wv",
                           "for (int64_t ci = 1; ci < cin; ++ci) {\n      const double wv"),
    "bias_grad_short": ("for (int64_t i = 0; i < Ho * Wo; ++i) acc += gyp[i];",
                        "for (int64_t i = 1; i < Ho * Wo; ++i) acc += gyp[i];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", str(lib), str(mpath)],
                   check=True, capture_output=True)
    env = dict(os.environ, DWCONV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_oracle_golden.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
