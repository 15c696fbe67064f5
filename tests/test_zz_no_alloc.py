"""dwc_bwd_filter_noalloc: the filter gradient for callers that cannot allocate device
memory (a fixed memory budget, a host that only hands over input and output buffers, or a
code path where an allocation's implicit synchronisation is not allowed).  Its workspace is
a fixed array inside the library, so its results must equal dwc_bwd_filter's with a
caller-allocated workspace, call after call, although every call reuses the same array.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process (it builds and loads the
library itself)."""
import numpy as np
import pytest
import torch

import depthwise_convolution_nhwc_gb300 as dwc
from depthwise_convolution_nhwc_gb300.inputs import Case
from parity_util import TOL, normalized_error

pytestmark = pytest.mark.gpu

DT = {"f32": 0, "bf16": 1, "f16": 2}


@pytest.fixture(scope="module")
def lib():
    dwc.build()
    return dwc.load_library()


def noalloc(lib, x, dy, case, out):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.dwc_bwd_filter_noalloc(x.data_ptr(), dy.data_ptr(), out.data_ptr(), case.N,
                                      case.H, case.W, case.C, case.FH, case.FW, case.stride,
                                      case.pad, DT[case.dtype], stream)


def test_noalloc_matches_workspace_version_on_consecutive_calls(lib):
    cases = [Case(8, 28, 28, 256, 13, 13, 1, 6, "f32", "normal", 41),
             Case(4, 56, 56, 128, 7, 7, 1, 3, "bf16", "normal", 42),
             Case(2, 15, 17, 24, 5, 5, 2, 2, "f32", "normal", 43)]   # general kernels
    for case in cases:
        x, dy = case.x().cuda(), case.dy().cuda()
        ref = dwc.bwd_filter(x, dy, (case.FH, case.FW), case.stride, case.pad)
        denom = dwc.bwd_filter(x.abs(), dy.abs(), (case.FH, case.FW), case.stride, case.pad)
        torch.cuda.synchronize()
        for _ in range(2):   # two calls in a row share the same scratch array
            out = torch.full((case.FH, case.FW, case.C), float("nan"), device="cuda")
            assert noalloc(lib, x, dy, case, out) == 0
            torch.cuda.synchronize()
            err = normalized_error(out.cpu().numpy(), ref.cpu().numpy(), denom.cpu().numpy())
            assert err <= TOL[case.dtype], (case, err)
    assert dwc.device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # 31x31 filters over 16384 channels need more than the fixed 32 MiB of scratch
    case = Case(64, 56, 56, 16384, 31, 31, 1, 15, "f32", "normal", 44)
    need = lib.dwc_bwd_filter_workspace_size(case.N, case.H, case.W, case.C, case.FH, case.FW,
                                             case.stride, case.pad, DT[case.dtype])
    assert need > 32 * 1024 * 1024
    code = lib.dwc_bwd_filter_noalloc(16, 16, 16, case.N, case.H, case.W, case.C, case.FH,
                                      case.FW, case.stride, case.pad, DT[case.dtype], None)
    assert code == 2  # DWC_ERR_UNSUPPORTED, nothing launched


def test_noalloc_reports_argument_errors_like_the_workspace_version(lib):
    assert lib.dwc_bwd_filter_noalloc(16, 16, 16, 1, 8, 8, 16, 3, 3, 0, 1, 0, None) == 1
    assert lib.dwc_bwd_filter_noalloc(None, 16, 16, 1, 8, 8, 16, 3, 3, 1, 1, 0, None) == 1
