"""Failure detection on the GPU without a fault: the bounded mbarrier wait
every kernel here uses is made to run out (a wait that nothing satisfies, with
a budget of about a millisecond).  The kernel returns, the device status word
reports the timeout to the host once and is cleared, and the context stays
usable: a prefill afterwards still matches the oracle."""
import pytest
import torch

from selective_state_space_131_b300 import inputs
from tests.gpu_util import TOL, dev, gpu_scan, max_rel, oracle_scan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m3():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from selective_state_space_131_b300 import m3scan
    return m3scan


def test_bounded_wait_runs_out_and_reports(m3):
    assert m3.m3_device_status() == m3.M3_OK            # start from a clear word
    assert m3.m3_selftest_wait_timeout(2_000_000) == m3.M3_OK
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_ERR_DEVICE    # the timeout, reported once
    assert m3.m3_device_status() == m3.M3_OK            # and cleared


def test_context_stays_usable_after_a_timeout(m3):
    assert m3.m3_selftest_wait_timeout(1_000_000) == m3.M3_OK
    assert m3.m3_device_status() == m3.M3_ERR_DEVICE
    shape = inputs.ScanShape(batch=2, seqlen=130, heads=3, headdim=64, dstate=64, rank=1, chunk=64, dtype="bf16")
    inp = inputs.make_scan_inputs(shape, 77)
    y, fs = gpu_scan(m3, dev(inp), shape.chunk)
    torch.cuda.synchronize()
    assert m3.m3_device_status() == m3.M3_OK
    yr, fr = oracle_scan(inp)
    assert max_rel(y.float().cpu(), yr) <= TOL["bf16"] and max_rel(fs.cpu(), fr) <= TOL["bf16"]
