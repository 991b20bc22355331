"""Failure detection without a GPU fault: a bounded wait that runs out (a
barrier nothing arrives at) reports a timeout through the device error
word, the kernel returns, and the context stays usable."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def v():
    from collective_reduction_virtual_gb300 import build
    build.build()
    import collective_reduction_virtual_gb300 as vc
    return vc


def test_bounded_wait_times_out_and_reports(v):
    assert v.device_errors(clear=True) == 0
    assert v.vcoll_selftest_wait_timeout(20_000) == v.OK  # 20 ms
    assert v.device_errors(clear=True) & v.DEVICE_ERR_TIMEOUT
    assert v.device_errors() == 0
    # the context still works: a normal collective right after
    ins = [torch.ones(1000, device="cuda") * (u + 1) for u in range(4)]
    out = v.allreduce(ins, op="sum")
    assert torch.equal(out[0], torch.full((1000,), 10.0, device="cuda"))
    assert v.device_errors() == 0


def test_selftest_rejects_bad_limits(v):
    assert v.vcoll_selftest_wait_timeout(0) == v.ERR_INVALID_ARG
    assert v.vcoll_selftest_wait_timeout(2_000_000) == v.ERR_INVALID_ARG
