"""The bounded on-device wait, made to run out on purpose.

Every wait of the scans for a bulk copy into shared memory is bounded; when
it gives up, the kernel sets the library's device error word and carries on,
and mamba_device_status() reports MAMBA_ERR_TIMEOUT.  A copy that never lands
cannot be produced safely, so the test hook (include/mamba_scan_testing.h)
waits with the same code on an mbarrier that nothing ever arrives on.  No GPU
fault, no hang: the wait ends after a few hundred polls.
"""
import pytest

from parity_util import TOL, gpu_scan, oracle_scan, rel_err, to_device
from selective_state_space_140_b300 import abi, workloads

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_is_reported_and_the_context_stays_usable(cuda):
    abi.mamba_device_status()  # start from a clear error word
    abi.mamba_test_bounded_wait(256)
    assert abi.mamba_device_status() == 7  # MAMBA_ERR_TIMEOUT
    assert abi.mamba_device_status() == 0  # reading cleared it
    x = workloads.make_scan_inputs(2, 20, 300, 16, "f32", seed=40, d_mode="normal")
    y, h = gpu_scan(to_device(x, cuda))
    assert abi.mamba_device_status() == 0
    yr, hr = oracle_scan(x)
    assert rel_err(y.cpu().numpy(), yr) <= TOL["f32"]
    assert rel_err(h.cpu().numpy(), hr) <= TOL["f32"]
