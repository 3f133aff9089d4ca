"""The give-up path of the library's bounded waits, exercised on purpose.

Every wait of the staging and tensor-core pipelines on an mbarrier is
bounded; when a wait runs out, the kernel counts it in the device counter
that dwconv_device_timeouts reads and returns instead of hanging. Here a
one-CTA self-test kernel waits a few hundred polls on a barrier that nothing
will ever complete (no copy and no tensor-core operation targets it, so
nothing is in flight), gives up through the same routine and returns; the
counter must grow by exactly one per launch and the context must stay
usable. The parity suite's checks that the counter is still 0 run earlier
(this file is collected after test_gpu_parity.py).
"""
import pytest

from depthwise_convolution_dwconv2d_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    th = pytest.importorskip("torch")
    if not th.cuda.is_available():
        pytest.skip("no CUDA device")
    from depthwise_convolution_dwconv2d_gb300 import build
    build.build()
    B.load()


def test_bounded_wait_gives_up_counts_and_returns():
    import torch
    before = B.dwconv_device_timeouts()
    B.dwconv_wait_selftest(256)
    torch.cuda.synchronize()
    assert B.dwconv_device_timeouts() == before + 1
    B.dwconv_wait_selftest(64)
    B.dwconv_wait_selftest(64)
    torch.cuda.synchronize()
    assert B.dwconv_device_timeouts() == before + 3
    # the context is still usable: an ordinary allocation and kernel run
    t = torch.ones(1024, device="cuda")
    assert float(t.sum()) == 1024.0


def test_wait_selftest_rejects_out_of_range_polls():
    with pytest.raises(B.DwconvError) as e:
        B.dwconv_wait_selftest(0)
    assert e.value.status == 1
    with pytest.raises(B.DwconvError) as e:
        B.dwconv_wait_selftest(1 << 20)
    assert e.value.status == 1
