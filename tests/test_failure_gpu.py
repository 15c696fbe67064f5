"""Failure path of the kernels' bounded waits, made to run on purpose without any GPU fault.

dwc_testing_stall_next_row_launch() makes the first CTA of the next row-kernel launch issue
none of its input copies (so no copy is ever in flight); its compute warps then wait until
the wait limit runs out, record the timeout in the device status word and end.  The test
shortens the limit to 1 ms, checks that the call returns promptly, that dwc_device_status()
reports DWC_ERR_TIMEOUT, and that the next ordinary call on the same context is correct and
reports DWC_OK."""
import time

import numpy as np
import pytest
import torch

import depthwise_convolution_nhwc_gb300 as dwc
from depthwise_convolution_nhwc_gb300.inputs import Case
from parity_util import TOL, normalized_error

pytestmark = pytest.mark.gpu

DWC_OK, DWC_ERR_TIMEOUT = 0, 6


def test_timed_out_wait_is_reported_and_the_context_stays_usable():
    import oracle
    lib = dwc.load_library()
    case = Case(2, 14, 14, 64, 7, 7, 1, 3, "f32", "normal", 11)
    assert dwc.path("fwd", None, None, None, case.N, case.H, case.W, case.C, case.FH, case.FW,
                    case.stride, case.pad, 0) == 1   # the row-streaming kernel serves it
    x, w = case.x().cuda(), case.w().cuda()
    assert dwc.device_status() == DWC_OK
    prev = dwc.set_wait_limit_ns(1_000_000)
    try:
        lib.dwc_testing_stall_next_row_launch()
        t0 = time.perf_counter()
        dwc.fwd(x, w, case.stride, case.pad)
        status = dwc.device_status()
        elapsed = time.perf_counter() - t0
    finally:
        dwc.set_wait_limit_ns(prev)
    assert status == DWC_ERR_TIMEOUT
    assert elapsed < 1.0, elapsed          # the 1 ms limit, not the 2 s default, ended it
    assert dwc.device_status() == DWC_OK   # reading the status cleared it

    y = dwc.fwd(x, w, case.stride, case.pad)
    assert dwc.device_status() == DWC_OK
    xn, wn = x.cpu().double().numpy(), w.cpu().double().numpy()
    ref = oracle.fwd(xn, wn, case.stride, case.pad)
    den = oracle.fwd(np.abs(xn), np.abs(wn), case.stride, case.pad)
    assert normalized_error(y.cpu().numpy(), ref, den) <= TOL[case.dtype]
