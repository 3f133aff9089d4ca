"""Every entry point under CUDA-graph capture.

The library enqueues only kernel launches on the caller's stream (no
allocation, copy, synchronisation or legacy-stream work), so a step of calls
can be captured once and replayed. For each workload of the bench, at a small
batch, the step's calls run eagerly, then are captured into one graph on a
non-default stream and replayed into the same output buffers (first filled
with a sentinel); every output must match the eager run bit for bit (the
entry points are deterministic). The families covered are those the bench
uses: tile, plane, large direct (fp32 pairs), tensor-core IBGEMM and weight
gradient, the fused multi-branch kernels, NHWC with epilogue, the separable
block and the filter-cache forward.
"""
import importlib.util
import os

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (workload, batch, layer labels kept: None = all)
CASES = [
    ("pr1", 1, None),
    ("mobilenet", 4, None),
    ("largek", 8, ["lk_H32_k7_f32", "lk_H32_k31_f32", "lk_H48_k21_f32", "lk_H32_k7_f16", "lk_H32_k31_f16",
                   "lk_H64_k27_f16"]),
    ("multidil", 1, None),
    ("multiplier", 4, None),
    ("infer", 4, None),
    ("separable", 4, None),
    ("largek_infer", 8, ["lki_H32_k31_f16", "lki_H64_k21_f16", "lki_H64_k31_f16"]),
]


@pytest.fixture(scope="module")
def bench():
    th = pytest.importorskip("torch")
    if not th.cuda.is_available():
        pytest.skip("no CUDA device")
    from depthwise_convolution_dwconv2d_gb300 import binding as B, build
    build.build()
    B.load()
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name,batch,keep", CASES, ids=[c[0] for c in CASES])
def test_step_graph_replay_matches_eager(bench, name, batch, keep):
    import torch

    dev = torch.device("cuda", 0)
    items = bench.build_workload(name)
    if keep is not None:
        items = [i for i in items if i.label() in keep]
        assert len(items) == len(keep)
    items = [type(i)(**{**i.__dict__, "N": batch}) for i in items]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        calls, groups = bench.setup_workload(name, items, dev, stream, bench.HostCache(), {})
        outs = [t for g in groups for t, _ in g[2]]
        for c in calls:
            c[6]()
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs]
    assert any(bool(t.abs().sum() > 0) for t in eager)
    families = sorted({c[2] for c in calls})

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            c[6]()
    for t in outs:
        t.fill_(7.0)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    for i, (t, e) in enumerate(zip(outs, eager)):
        assert torch.equal(t.view(torch.uint8), e.view(torch.uint8)), (name, i, families)
    # a second replay after the outputs were overwritten again
    for t in outs:
        t.fill_(-1.0)
    g.replay()
    torch.cuda.synchronize()
    for i, (t, e) in enumerate(zip(outs, eager)):
        assert torch.equal(t.view(torch.uint8), e.view(torch.uint8)), (name, i, families)
    del g
