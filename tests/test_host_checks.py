"""Host-side bounds checks of the kernels' planners (no GPU).

Each program under tests/host/ compiles a kernel family's planner with nvcc
(host code only runs) and replays, for hundreds of shapes, the index
arithmetic the kernel's threads perform against the planned layout:
  * check_pair.cu: the packed fp32 large forward / grad-input: staging
    writes and window / filter reads inside each plane-pair block, every
    output row of a band covered once;
  * check_pwgrad.cu: the packed fp32 large weight gradient: staging and
    window reads inside the stage, the thread -> tap-block map a bijection,
    sample chunks of whole pairs covering the batch;
  * check_ibc.cu: the filter-cache tensor-core kernel: shared- and
    tensor-memory plan, the cache's strip taps, the K steps and strip
    offsets of every tile, and the whole GEMM walk equal to a direct integer
    correlation;
  * check_ibgemm.cu: the uncached tensor-core forward / grad-input: memory
    plan, K steps covering every input position a tile reads, and the
    builders' 16-byte filter pieces (bounds, alignment, values) walked
    against a direct integer correlation.
Each prints one line per plan and exits non-zero on any failure.
"""
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HOST = os.path.join(ROOT, "tests", "host")
CSRC = os.path.join(ROOT, "depthwise_convolution_dwconv2d_gb300", "csrc")
PROGRAMS = ["check_pair", "check_pwgrad", "check_ibc", "check_ibgemm"]


@pytest.fixture(scope="module")
def built(tmp_path_factory):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not found")
    out = tmp_path_factory.mktemp("host_checks")

    def build(name):
        exe = str(out / name)
        cmd = [nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
               "-I", os.path.join(ROOT, "include"), "-I", CSRC, os.path.join(HOST, name + ".cu"),
               os.path.join(CSRC, "tma.cu"), "-o", exe, "-lcuda"]
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
        return name, exe, r

    with ThreadPoolExecutor(len(PROGRAMS)) as ex:
        res = list(ex.map(build, PROGRAMS))
    exes = {}
    for name, exe, r in res:
        assert r.returncode == 0, f"{name}: {r.stderr[-3000:]}"
        exes[name] = exe
    return exes


@pytest.mark.parametrize("name", PROGRAMS)
def test_planner_index_bounds(built, name):
    r = subprocess.run([built[name]], capture_output=True, text=True, timeout=600)
    tail = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else ""
    assert r.returncode == 0, f"{name}: {tail}\n" + "\n".join(
        ln for ln in r.stdout.splitlines() if ln.startswith("FAIL"))[:3000]
    assert "fails: 0" in tail or "fails 0" in tail, tail
