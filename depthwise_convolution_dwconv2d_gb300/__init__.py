"""libdwconv: depthwise 2-D convolution on GB300 (sm_103a), forward,
backward-data and backward-weight, behind a C ABI (include/dwconv.h).

The Python surface is the binding in ``binding`` (same names as the C entry
points). ``build.build()`` compiles the CUDA library in-tree. ``synth`` draws
seeded synthetic inputs and holds no convolution arithmetic.
"""
from .binding import (  # noqa: F401
    DTYPES, Desc, DwconvError, ESIZE, SYMBOLS, dwconv2d_bwd_data, dwconv2d_bwd_data_multi,
    dwconv2d_bwd_weight, dwconv2d_bwd_weight_noalloc, dwconv2d_bwd_weight_workspace_size, dwconv2d_fwd, dwconv2d_fwd_multi,
    dwconv2d_multi_plan_name, dwconv2d_output_shape, dwconv2d_plan_name, dwconv_device_timeouts, dwconv_fma_probe, dwconv_status_string, lib_path,
    load, make_desc)
