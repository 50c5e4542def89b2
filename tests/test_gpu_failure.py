"""Failure detection without a GPU fault: a bounded wait runs out, the kernel
records the time-out and returns, the host reads it, and the context stays
usable.  The wait is on a barrier that nothing ever completes (no copy is in
flight), limited to a few milliseconds."""
import pytest
import torch

import far_gen
from gpu_helpers import check_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def far():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import mixed_precision_residual_gb300 as far

    return far


def test_wait_timeout_is_reported_and_cleared(far):
    assert far.device_status() == 0
    far.selftest_wait_timeout(5000)  # 5 ms
    assert far.device_status() == far.FAR_ERR_TIMEOUT
    assert far.device_status() == 0  # read-and-clear


def test_context_usable_after_timeout(far):
    far.selftest_wait_timeout(2000)
    assert far.device_status() == far.FAR_ERR_TIMEOUT
    d = far_gen.custom_inputs("bf16", "bf16", 64, 4096, seed=1)
    check_both(far, d, "after a time-out")


def test_selftest_argument_range(far):
    with pytest.raises(far.FarError):
        far.selftest_wait_timeout(0)
