"""Failure detection on the device without a fault (GPU).

Every pipeline wait in the kernels is bounded; when one gives up it records
Q4_0_ERR_DEVICE_TIMEOUT in the device error word and the kernel returns.
The self-check makes one wait run out on purpose (an mbarrier nothing
arrives on, 20 ms limit) and checks that the status comes back and that the
context still computes correctly afterwards.
"""
import pytest
import torch

import oracle
from gpu_common import check_full, lib, wq_dev, x_dev
from q4_weight_only_gb300 import synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    q4 = lib()
    assert q4.device_error() == q4.OK
    assert q4.selftest_wait_timeout(20000) == q4.ERR_DEVICE_TIMEOUT
    assert q4.device_error() == q4.OK          # reading clears the word
    w, x = synth.small_case(77, 3, 300, 1024)
    wq = oracle.get().quantize(w)
    check_full(q4.matmul(x_dev(x), wq_dev(wq), 300, 1024), x, wq, 300, 1024)
    assert q4.device_error() == q4.OK


def test_selftest_rejects_bad_limit():
    q4 = lib()
    with pytest.raises(q4.Q4Error):
        q4.selftest_wait_timeout(0)
