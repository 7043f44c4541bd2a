"""The failure path of the bounded waits, on the GPU without a fault: a probe
kernel's wait on a barrier that nothing completes gives up after its limit
(about one second), records a timeout in the device status word and returns.
The host then reads LA_ERR_TIMEOUT, and the context keeps working."""
import time

import pytest
import torch

import oracle
import recurrent_lm_gb300 as la
from recurrent_lm_gb300 import inputs
from helpers import TOL, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_bounded_wait_reports_timeout_and_context_survives():
    la.check_device_status()  # start from a clear status word
    t0 = time.perf_counter()
    la.debug_timeout_probe()
    with pytest.raises(la.LAError) as e:
        la.check_device_status()
    elapsed = time.perf_counter() - t0
    assert e.value.status == la.LA_ERR_TIMEOUT
    assert 0.2 < elapsed < 30.0, elapsed  # the wait gave up at its limit, not at once and not never
    la.check_device_status()  # the check cleared the word
    # the context still runs the kernels correctly
    q, k, v, _, _ = inputs.qkv(1, 2, 200, seed=950, dtype=torch.bfloat16)
    y, s, z = la.prefill(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    la.check_device_status()
    yr, sr, zr = oracle.prefill(q, k, v)
    assert_close("y", y, yr, TOL[torch.bfloat16])
    assert_close("s", s, sr, TOL[torch.bfloat16])
