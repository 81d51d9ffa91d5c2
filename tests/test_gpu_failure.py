"""Failure detection without a GPU fault: a bounded wait that runs out reports
CB_ERR_TIMEOUT through the device error word and the context stays usable."""
import time

import pytest
import torch

from continuous_batching_ragged_gb300 import native
from continuous_batching_ragged_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports(native_lib):
    from continuous_batching_ragged_gb300 import api
    api.cb_check_device_errors()                     # start from a clean word
    t0 = time.perf_counter()
    status = native_lib.cb_selftest_bounded_wait(50, int(torch.cuda.current_stream().cuda_stream))
    assert status == native.CB_OK
    with pytest.raises(native.CBError) as e:
        api.cb_check_device_errors()
    elapsed = time.perf_counter() - t0
    assert e.value.status == native.CB_ERR_TIMEOUT
    assert 0.04 < elapsed < 5.0                      # it waited about the limit, then gave up
    api.cb_check_device_errors()                     # the word was cleared
    # the context is still usable: a normal step runs and is correct
    from gpu_harness import DeviceStep, assert_tolerance, oracle_packed, to_np
    b = W.make_batch([40, 0], [1, 130], num_heads=2, head_dim=128, block_size=16, dtype="bf16", seed=5)
    assert_tolerance(to_np(DeviceStep(b).run()), oracle_packed(b))


def test_bounded_wait_rejects_bad_limits(native_lib):
    assert native_lib.cb_selftest_bounded_wait(0, None) == native.CB_ERR_INVALID
    assert native_lib.cb_selftest_bounded_wait(20000, None) == native.CB_ERR_INVALID
