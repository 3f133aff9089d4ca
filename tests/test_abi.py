"""The C-ABI library on the host: it builds, loads, exports every symbol the
header declares, and rejects bad arguments before any launch (no GPU needed:
each call below fails validation, so nothing is enqueued)."""
import ctypes
import os
import re

import pytest

from depthwise_convolution_dwconv2d_gb300 import binding as B
from depthwise_convolution_dwconv2d_gb300 import build as BLD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dwconv.h")


@pytest.fixture(scope="module")
def lib():
    BLD.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(dwconv\w+)\s*\(", text, flags=re.M)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(B.SYMBOLS)


def test_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {B.lib_path()}").read()
    for name in declared_functions():
        assert re.search(rf"\bT {name}\b", out), f"{name} not exported"


def test_desc_layout():
    assert ctypes.sizeof(B.Desc) == 88
    assert B.Desc.out_c_offset.offset == 72 and B.Desc.dtype.offset == 68


def test_output_shape(lib):
    assert B.dwconv2d_output_shape(B.make_desc(64, 128, 56, 56, 3, 1, 1)) == (56, 56)
    assert B.dwconv2d_output_shape(B.make_desc(64, 64, 112, 112, 3, 2, 1)) == (56, 56)
    assert B.dwconv2d_output_shape(B.make_desc(64, 1024, 7, 7, 3, 2, 1)) == (4, 4)
    assert B.dwconv2d_output_shape(B.make_desc(2, 64, 256, 256, 3, 1, 5, 5)) == (256, 256)
    assert B.dwconv2d_output_shape(B.make_desc(1, 1, 5, 5, 2, 2, 0, 2)) == (2, 2)
    assert B.dwconv2d_output_shape(B.make_desc(1, 1, 3, 7, (5, 3), (1, 2), (1, 0))) == (1, 3)


def status_of(fn, *args):
    try:
        fn(*args)
    except B.DwconvError as e:
        return e.status
    return 0


INVALID, UNSUPPORTED, MISALIGNED, WORKSPACE = 1, 2, 3, 4
P = 0x10000  # a well-aligned fake address: validation fails before any use


@pytest.mark.parametrize("desc,want", [
    (B.make_desc(1, 0, 8, 8), INVALID),                 # C < 1
    (B.make_desc(-1, 3, 8, 8), INVALID),                # N < 0
    (B.make_desc(1, 3, 0, 8), INVALID),                 # H < 1
    (B.make_desc(1, 3, 8, 8, 0), INVALID),              # kernel < 1
    (B.make_desc(1, 3, 8, 8, 3, 0), INVALID),           # stride < 1
    (B.make_desc(1, 3, 8, 8, 3, 1, -1), INVALID),       # pad < 0
    (B.make_desc(1, 3, 8, 8, 3, 1, 1, 0), INVALID),     # dilation < 1
    (B.make_desc(1, 3, 2, 2, 5, 1, 0), INVALID),        # Ho < 1
    (B.make_desc(1, 3, 8, 8, multiplier=0), INVALID),
    (B.make_desc(1, 3, 8, 8, out_c_offset=2, out_c_total=4), INVALID),   # slice overflows
    (B.make_desc(1, 3, 8, 8, out_c_offset=-1, out_c_total=9), INVALID),
    (B.make_desc(1, 3, 8, 8, dtype=7), UNSUPPORTED),
    (B.make_desc(1, 3, 300, 300, 256, 1, 128), UNSUPPORTED),  # kernel > 255
])
def test_bad_descriptors_rejected(lib, desc, want):
    assert status_of(B.dwconv2d_fwd, desc, P, P, None, P, 0) == want
    assert status_of(B.dwconv2d_bwd_data, desc, P, P, P, 0, 0) == want
    assert status_of(B.dwconv2d_bwd_weight, desc, P, P, P, None, P, 1 << 30, 0) == want
    assert B.dwconv2d_bwd_weight_workspace_size(desc) == 0
    assert B.dwconv2d_plan_name(desc, 0) == "invalid"


def test_null_and_misaligned_pointers(lib):
    d = B.make_desc(2, 3, 8, 8, 3, 1, 1)
    assert status_of(B.dwconv2d_fwd, d, None, P, None, P, 0) == INVALID
    assert status_of(B.dwconv2d_fwd, d, P, None, None, P, 0) == INVALID
    assert status_of(B.dwconv2d_fwd, d, P, P, None, None, 0) == INVALID
    assert status_of(B.dwconv2d_fwd, d, P + 2, P, None, P, 0) == MISALIGNED
    assert status_of(B.dwconv2d_fwd, d, P, P, P + 1, P, 0) == MISALIGNED
    h = B.make_desc(2, 3, 8, 8, 3, 1, 1, dtype="bf16")
    assert status_of(B.dwconv2d_fwd, h, P + 1, P, None, P, 0) == MISALIGNED
    assert status_of(B.dwconv2d_bwd_data, d, P, P, P, 2, 0) == INVALID   # accumulate not 0/1
    assert status_of(B.dwconv2d_bwd_data, d, P, P, P + 2, 0, 0) == MISALIGNED


def test_epilogue_argument_checks(lib):
    d = B.make_desc(2, 3, 8, 8, 3, 1, 1)
    fe = B.dwconv2d_fwd_epilogue
    assert status_of(fe, d, P, P, None, None, None, 3, P, 0) == INVALID     # unknown activation
    assert status_of(fe, d, P, P, None, None, None, -1, P, 0) == INVALID
    assert status_of(fe, d, P, P, None, P + 2, None, "relu", P, 0) == MISALIGNED   # scale
    assert status_of(fe, d, P, P, None, None, P + 1, "relu6", P, 0) == MISALIGNED  # shift
    assert status_of(fe, d, None, P, None, P, P, "relu", P, 0) == INVALID
    assert status_of(fe, d, P, P, None, P, P, "relu", None, 0) == INVALID
    # empty batch: a valid no-op once the filter pointers check out
    e = B.make_desc(0, 3, 8, 8, 3, 1, 1)
    assert status_of(fe, e, None, P, None, P, P, "relu", None, 0) == 0


def test_epilogue_plan_avoids_kernels_without_one(lib):
    """Pass 3 (forward with a fused epilogue) never names the small-plane or
    tensor-core forward kernels, which have no epilogue."""
    small = B.make_desc(64, 512, 14, 14, 3, 1, 1)
    assert B.dwconv2d_plan_name(small, 0) == "plane"
    assert B.dwconv2d_plan_name(small, 3) == "tile"
    big = B.make_desc(64, 384, 32, 32, 31, 1, 15, dtype="f16")
    assert B.dwconv2d_plan_name(big, 0) == "ibgemm"
    assert B.dwconv2d_plan_name(big, 3) == "large"
    mb = B.make_desc(64, 128, 56, 56, 3, 1, 1)
    assert B.dwconv2d_plan_name(mb, 3) == B.dwconv2d_plan_name(mb, 0) == "tile"
    odd = B.make_desc(2, 3, 9, 9, 4, 1, 1)
    assert B.dwconv2d_plan_name(odd, 3) == "generic"
    assert B.dwconv2d_plan_name(odd, 5) == "invalid"


def test_nhwc_argument_checks_and_routing(lib):
    d = B.make_desc(2, 32, 8, 8, 3, 1, 1)
    fn = B.dwconv2d_fwd_nhwc
    assert status_of(fn, d, P, P, None, P, None, None, 7) == INVALID          # unknown activation
    assert status_of(fn, d, P, None, None, P) == INVALID
    assert status_of(fn, d, P, P, None, None) == INVALID
    assert status_of(fn, d, P + 2, P, None, P) == MISALIGNED
    assert status_of(fn, d, P, P, None, P, P + 1, None, "relu") == MISALIGNED
    assert status_of(fn, B.make_desc(0, 32, 8, 8, 3, 1, 1), None, P, None, None) == 0
    # tiled kernel: 3/5/7 square, stride 1 or 2, dilation 1, m = 1, C*es % 16 == 0
    assert B.dwconv2d_plan_name(B.make_desc(64, 128, 56, 56, 3, 1, 1), 4) == "nhwc"
    assert B.dwconv2d_plan_name(B.make_desc(64, 64, 112, 112, 3, 2, 1, dtype="bf16"), 4) == "nhwc"
    assert B.dwconv2d_plan_name(B.make_desc(8, 36, 30, 30, 7, 2, 3), 4) == "nhwc"
    assert B.dwconv2d_plan_name(B.make_desc(8, 6, 30, 30, 3, 1, 1), 4) == "generic"        # 24-byte pixels
    assert B.dwconv2d_plan_name(B.make_desc(8, 12, 30, 30, 3, 1, 1, dtype="f16"), 4) == "generic"
    assert B.dwconv2d_plan_name(B.make_desc(8, 32, 30, 30, 3, 1, 2, 2), 4) == "generic"    # dilation
    assert B.dwconv2d_plan_name(B.make_desc(8, 32, 30, 30, 3, 3, 1), 4) == "generic"       # stride 3
    assert B.dwconv2d_plan_name(B.make_desc(8, 32, 30, 30, 3, 1, 1, multiplier=2), 4) == "generic"
    assert B.dwconv2d_plan_name(B.make_desc(8, 32, 30, 30, 9, 1, 4), 4) == "generic"


def test_separable_argument_checks_and_routing(lib):
    d = B.make_desc(2, 64, 8, 8, 3, 1, 1, dtype="bf16")
    fn = B.dwconv2d_separable_nhwc
    assert status_of(fn, d, P, P, 0, P, P) == INVALID                       # cout < 1
    assert status_of(fn, d, P, P, 32, P, P, None, None, 5) == INVALID       # unknown activation
    assert status_of(fn, d, P, P, 32, P, P, None, None, 0, None, None, -2) == INVALID
    assert status_of(fn, d, P, P, 32, None, P) == INVALID                   # no pointwise weights
    assert status_of(fn, d, P, P, 32, P + 1, P) == MISALIGNED
    assert status_of(fn, d, P, P, 32, P, P, P + 1) == MISALIGNED            # dw_scale
    slice_over = B.make_desc(2, 64, 8, 8, 3, 1, 1, dtype="bf16", out_c_offset=10, out_c_total=40)
    assert status_of(fn, slice_over, P, P, 32, P, P) == INVALID
    assert B.dwconv2d_separable_plan_name(slice_over, 30) == "septc"        # 10 + 30 <= 40
    assert B.dwconv2d_separable_plan_name(slice_over, 31) == "invalid"
    assert status_of(fn, B.make_desc(0, 64, 8, 8, 3, 1, 1, dtype="bf16"), None, P, 32, P, None) == 0
    # tensor-core kernel: 16-bit, 3x3 / 5x5, stride 1 / 2, dilation 1, m = 1, C % 64 == 0
    sp = B.dwconv2d_separable_plan_name
    assert sp(B.make_desc(64, 128, 56, 56, 3, 1, 1, dtype="bf16"), 128) == "septc"
    assert sp(B.make_desc(64, 512, 14, 14, 3, 2, 1, dtype="f16"), 1024) == "septc"
    assert sp(B.make_desc(8, 64, 30, 30, 5, 2, 2, dtype="bf16"), 96) == "septc"
    assert sp(B.make_desc(8, 64, 30, 30, 3, 1, 1), 96) == "generic"                     # fp32
    assert sp(B.make_desc(8, 96, 30, 30, 3, 1, 1, dtype="bf16"), 96) == "generic"       # C % 64
    assert sp(B.make_desc(8, 64, 30, 30, 7, 1, 3, dtype="bf16"), 96) == "generic"       # 7x7
    assert sp(B.make_desc(8, 64, 30, 30, 3, 1, 2, 2, dtype="bf16"), 96) == "generic"    # dilation
    assert sp(B.make_desc(8, 64, 30, 30, 3, 1, 1, multiplier=2, dtype="bf16"), 96) == "generic"
    # the generic kernel stages one pixel's C*m fp32 values in at most 96 KB
    assert sp(B.make_desc(1, 24577, 4, 4, 3, 1, 1), 8) == "invalid"


def test_workspace_checks(lib):
    d = B.make_desc(4, 8, 16, 16, 3, 1, 1)
    need = B.dwconv2d_bwd_weight_workspace_size(d)
    assert need > 0 and need % 256 == 0
    assert status_of(B.dwconv2d_bwd_weight, d, P, P, P, None, None, need, 0) == WORKSPACE
    assert status_of(B.dwconv2d_bwd_weight, d, P, P, P, None, P, need - 1, 0) == WORKSPACE
    assert status_of(B.dwconv2d_bwd_weight, d, P, P, P, None, P + 8, need, 0) == MISALIGNED
    # nothing requested: a valid no-op that touches nothing
    assert status_of(B.dwconv2d_bwd_weight, d, None, None, None, None, None, 0, 0) == 0


def test_empty_batch_is_noop(lib):
    d = B.make_desc(0, 3, 8, 8, 3, 1, 1)
    assert status_of(B.dwconv2d_fwd, d, None, P, None, None, 0) == 0
    assert status_of(B.dwconv2d_bwd_data, d, None, P, None, 0, 0) == 0


def test_multi_branch_validation(lib):
    mk = lambda d, off: B.make_desc(2, 4, 16, 16, 3, 1, d, d, out_c_offset=off, out_c_total=12)
    ok = [mk(1, 0), mk(3, 4), mk(5, 8)]
    # unequal output size
    bad_size = [mk(1, 0), B.make_desc(2, 4, 16, 16, 3, 1, 0, 1, out_c_offset=4, out_c_total=12)]
    assert status_of(B.dwconv2d_fwd_multi, bad_size, P, [P, P], None, P, 0) == INVALID
    # overlapping slices
    assert status_of(B.dwconv2d_fwd_multi, [mk(1, 0), mk(3, 2)], P, [P, P], None, P, 0) == INVALID
    # too many branches / none
    assert status_of(B.dwconv2d_fwd_multi, ok * 3, P, [P] * 9, None, P, 0) == INVALID
    assert status_of(B.dwconv2d_bwd_data_multi, [], P, [], P, 0) == INVALID
    # differing c_total
    odd = [mk(1, 0), B.make_desc(2, 4, 16, 16, 3, 1, 3, 3, out_c_offset=4, out_c_total=13)]
    assert status_of(B.dwconv2d_bwd_data_multi, odd, P, [P, P], P, 0) == INVALID


def test_status_strings(lib):
    for s in range(6):
        assert B.dwconv_status_string(s)
    assert B.dwconv_status_string(99) == "unknown status"


def test_plan_names(lib):
    assert B.dwconv2d_plan_name(B.make_desc(64, 128, 56, 56, 3, 1, 1), 0) in ("generic", "tile", "large")
    assert B.dwconv2d_plan_name(B.make_desc(64, 128, 56, 56, 3, 1, 1), 5) == "invalid"
    assert B.dwconv2d_plan_name(B.make_desc(64, 128, 56, 56, 3, 1, 1), -1) == "invalid"


def test_packed_weight_gradient_chunks_hold_whole_pairs(lib):
    """Host planning of the packed fp32 large weight gradient (no GPU needed):
    about eight (channel, chunk) units per resident CTA (two per SM on 152
    SMs), chunks of an even number of samples so that only the batch's last
    sample can sit in a half-empty pair; the workspace holds chunks x OC x
    (k*k + 1) fp32 partials."""
    K = 31
    for N, C in [(16, 384), (64, 384), (33, 384), (9, 64), (7, 64), (1, 64), (2, 64), (200, 64)]:
        d = B.make_desc(N, C, 32, 32, K, 1, K // 2, 1, 1, "f32")
        assert B.dwconv2d_plan_name(d, 2) == "large"
        per_chunk = C * (K * K + 1) * 4  # C a multiple of 64: a whole number of 256-byte blocks
        ws = B.dwconv2d_bwd_weight_workspace_size(d)
        assert ws % per_chunk == 0
        chunks = ws // per_chunk
        want = max(1, min((152 * 2 * 8 + C - 1) // C, N))
        nb = (N + want - 1) // want
        nb += nb & 1
        assert chunks == (N + nb - 1) // nb, (N, C, chunks)
        assert nb % 2 == 0 and (chunks - 1) * nb < N <= chunks * nb


def test_plane_routing_and_chunking(lib):
    """Host planning of the small-plane family (no GPU needed): the forward and
    stride-1 grad-input take it on rows of 9..16, the weight gradient on
    output rows of at most 16; its weight-gradient chunks cover the batch
    (1 <= chunks <= N) and size the workspace as chunks x OC x (k*k + 1)
    fp32 partials."""
    mk = lambda N, C, H, s: B.make_desc(N, C, H, H, 3, s, 1)
    assert B.dwconv2d_plan_name(mk(64, 512, 14, 1), 0) == "plane"
    assert B.dwconv2d_plan_name(mk(64, 512, 14, 1), 1) == "plane"
    assert B.dwconv2d_plan_name(mk(64, 512, 14, 2), 0) == "plane"
    assert B.dwconv2d_plan_name(mk(64, 512, 14, 2), 1) == "tile"  # strided grad-input
    assert B.dwconv2d_plan_name(mk(64, 256, 28, 2), 2) == "plane"  # output rows of 14
    assert B.dwconv2d_plan_name(mk(64, 256, 28, 1), 2) == "tile"  # output rows of 28
    assert B.dwconv2d_plan_name(mk(64, 256, 28, 1), 0) == "tile"  # rows of 28
    # tall stride-2 planes: the forward's eight-warp tile buffers would need
    # about 300 KB of shared memory, so it goes to the tile kernel; the weight
    # gradient's fit with four warps per CTA
    tall = B.make_desc(2, 3, 64, 16, 3, 2, 1)
    assert B.dwconv2d_plan_name(tall, 0) != "plane"
    assert B.dwconv2d_plan_name(tall, 2) == "plane"
    for N, C, H, s in [(64, 512, 14, 1), (64, 512, 14, 2), (64, 1024, 7, 2), (64, 256, 28, 2), (62, 128, 14, 1),
                       (1, 32, 14, 1), (17, 32, 11, 2)]:
        d = mk(N, C, H, s)
        assert B.dwconv2d_plan_name(d, 2) == "plane"
        ws = B.dwconv2d_bwd_weight_workspace_size(d)
        per_chunk = C * (3 * 3 + 1) * 4  # C a multiple of 32: a whole number of 256-byte blocks
        assert ws % per_chunk == 0
        chunks = ws // per_chunk
        assert 1 <= chunks <= N, (N, C, H, s, chunks)


def test_tile_routing_respects_band_limits(lib):
    """A shape whose narrowest tile band would exceed the tile planner's
    48 KB shared-memory limit is routed to the generic kernels by the host
    planner, instead of failing at launch. Worked cases (fp32):
    - 3x3, dilation 5, padding 5, rows of 400: the forward's narrowest band
      is 20 output rows = 30 input rows x a 416-element pitch x 4 B
      = 49,920 B;
    - 3x3, padding 1, multiplier 2, rows of 1024: the stride-1 grad-input
      stages 2 grad_out planes of 6 rows x 1032 elements x 4 B = 49,536 B."""
    assert B.dwconv2d_plan_name(B.make_desc(2, 4, 16, 400, 3, 1, 5, 5), 0) == "generic"
    assert B.dwconv2d_plan_name(B.make_desc(2, 4, 16, 1024, 3, 1, 1, 1, 2), 1) == "generic"
    # the same filters on narrower rows stay on the tile kernels
    assert B.dwconv2d_plan_name(B.make_desc(2, 4, 16, 256, 3, 1, 5, 5), 0) == "tile"
    assert B.dwconv2d_plan_name(B.make_desc(2, 4, 16, 512, 3, 1, 1, 1, 2), 1) == "tile"
    # the fused multi-dilation path fits its 96 KB bands up to its 512-wide rows
    ds = [B.make_desc(2, 8, 16, 512, 3, 1, d, d, out_c_offset=8 * i, out_c_total=24)
          for i, d in enumerate((1, 3, 5))]
    assert B.dwconv2d_multi_plan_name(ds) == "tile"


def test_large_weight_gradient_routing_respects_shared_memory(lib):
    """The scalar large-filter weight gradient (below 13 taps) stages two fp32
    (x tile + grad_out plane) stages; from 112 x 112 planes it would need
    more than its 220 KB limit (k = 9 at 112 x 112: 2 x (123 rows x 132 +
    112 x 112) floats = 230 KB), so those shapes take the generic weight
    gradient while the forward and grad-input stay on the large kernels. The
    packed kernel (13 taps and up) cuts a plane into bands of output rows
    until they fit, so it serves them."""
    big = B.make_desc(4, 8, 112, 112, 9, 1, 4)
    assert B.dwconv2d_plan_name(big, 0) == "large"
    assert B.dwconv2d_plan_name(big, 2) == "generic"
    for k in (17, 31):
        banded = B.make_desc(4, 8, 112, 112, k, 1, k // 2)
        assert B.dwconv2d_plan_name(banded, 2) == "large"
    fits = B.make_desc(4, 8, 96, 96, 31, 1, 15)
    assert B.dwconv2d_plan_name(fits, 2) == "large"


def test_every_odd_large_filter_has_a_specialised_plan(lib):
    """Every odd filter size from 7 to 31 at the large-kernel sweep's sizes
    (64 x 384 x {32, 48, 64}^2, stride 1, pad k // 2) plans to a specialised
    family for all three passes: the direct large kernels for fp32 (the tile
    kernels for 7), the tensor-core kernels for the fp16 forward, grad-input
    and weight gradient from 9 up."""
    for k in range(7, 32, 2):
        for h in (32, 48, 64):
            d32 = B.make_desc(64, 384, h, h, k, 1, k // 2, 1, 1, "f32")
            d16 = B.make_desc(64, 384, h, h, k, 1, k // 2, 1, 1, "f16")
            want = "tile" if k == 7 else "large"
            assert [B.dwconv2d_plan_name(d32, p) for p in range(3)] == [want] * 3, (k, h)
            p16 = [B.dwconv2d_plan_name(d16, p) for p in range(3)]
            assert p16[:2] == (["tile"] * 2 if k == 7 else ["ibgemm"] * 2), (k, h, p16)
            assert p16[2] == ("tile" if k == 7 else "tcwgrad"), (k, h, p16)


def test_filter_cache_sizes_and_argument_checks(lib):
    """Cache sizes of the large-kernel layers (C x strips x W rows of 128
    bytes; 38 strips for 31x31 at width 32, 44 at width 16, 23 for 21x21 at
    width 64), shapes without a cached form (31x31 at width 64: its 35
    strips of 8 KB do not fit in shared memory), and the checks before any
    launch."""
    size = B.dwconv2d_filter_cache_size
    for W, k, strips in ((32, 31, 38), (16, 31, 44), (64, 21, 23), (32, 13, 22)):
        for pass_ in (0, 1):
            assert size(B.make_desc(64, 384, W, W, k, 1, k // 2, dtype="f16"), pass_) == 384 * strips * W * 128
    d = B.make_desc(64, 384, 32, 32, 31, 1, 15, dtype="bf16")
    # independent of N and H
    assert size(B.make_desc(1, 384, 7, 32, 31, 1, 15, dtype="bf16"), 0) == size(d, 0)
    assert size(B.make_desc(0, 384, 32, 32, 31, 1, 15, dtype="bf16"), 0) == size(d, 0)
    assert size(B.make_desc(300, 384, 32, 32, 31, 1, 15, dtype="bf16"), 0) == size(d, 0)
    for bad in (B.make_desc(64, 384, 32, 32, 31, 1, 15),                      # fp32
                B.make_desc(64, 384, 48, 48, 31, 1, 15, dtype="f16"),         # 48 does not divide 64
                B.make_desc(64, 384, 24, 24, 11, 1, 2, dtype="f16"),          # Wo != W
                B.make_desc(64, 384, 32, 32, 31, 2, 15, dtype="f16"),         # stride 2
                B.make_desc(64, 384, 32, 32, 31, 1, 15, 2, dtype="f16"),      # dilation 2
                B.make_desc(8, 16, 32, 32, 31, 1, 15, multiplier=2, dtype="f16"),
                B.make_desc(8, 16, 4, 4, 3, 1, 1, dtype="f16"),               # width 4
                B.make_desc(64, 384, 64, 64, 31, 1, 15, dtype="f16"),         # strips do not fit
                B.make_desc(64, 384, 64, 64, 27, 1, 13, dtype="bf16")):
        assert size(bad, 0) == 0 and size(bad, 1) == 0
    assert size(d, 2) == 0 and size(d, -1) == 0
    need = size(d, 0)
    build, fc, bc = B.dwconv2d_filter_cache_build, B.dwconv2d_fwd_cached, B.dwconv2d_bwd_data_cached
    assert status_of(build, d, 2, P, P, need, 0) == INVALID
    assert status_of(build, d, 0, P, None, need, 0) == WORKSPACE
    assert status_of(build, d, 0, P, P, need - 1, 0) == WORKSPACE
    assert status_of(build, d, 0, P, P + 8, need, 0) == MISALIGNED
    assert status_of(build, d, 0, P + 1, P, need, 0) == MISALIGNED
    assert status_of(build, d, 0, None, P, need, 0) == INVALID
    f32 = B.make_desc(64, 384, 32, 32, 31, 1, 15)
    assert status_of(build, f32, 0, P, P, 1 << 30, 0) == UNSUPPORTED
    assert status_of(fc, f32, P, P, None, P, 1 << 30, 0) == UNSUPPORTED
    assert status_of(fc, d, P, None, None, P, need, 0) == WORKSPACE
    assert status_of(fc, d, P, P, None, P, need - 2, 0) == WORKSPACE
    assert status_of(fc, d, P + 8, P, None, P, need, 0) == MISALIGNED     # x on the 16-byte grid
    assert status_of(fc, d, P, P, P + 1, P, need, 0) == MISALIGNED        # bias
    assert status_of(fc, d, P, P, None, None, need, 0) == INVALID
    big = B.make_desc(64, 384, 64, 64, 31, 1, 15, dtype="bf16")
    assert status_of(fc, big, P, P, None, P, 1 << 30, 0) == UNSUPPORTED
    assert status_of(build, big, 0, P, P, 1 << 30, 0) == UNSUPPORTED
    assert status_of(bc, d, P, P, P, 2, need, 0) == INVALID                 # accumulate not 0 / 1
    assert status_of(bc, d, P, P, P + 1, 0, need, 0) == MISALIGNED
    assert status_of(bc, d, P + 8, P, P, 0, need, 0) == MISALIGNED
    # empty batch: a valid no-op once the cache checks out
    e = B.make_desc(0, 384, 32, 32, 31, 1, 15, dtype="bf16")
    assert status_of(fc, e, None, P, None, None, need, 0) == 0
    assert status_of(bc, e, None, P, None, 0, need, 0) == 0
