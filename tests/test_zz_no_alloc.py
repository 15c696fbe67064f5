"""dwc_bwd_filter_noalloc: the filter gradient for callers that cannot allocate device
memory (a fixed memory budget, a host that only hands over input and output buffers, or a
code path where an allocation's implicit synchronisation is not allowed).  Its workspace is
a fixed array inside the library, so its results must equal dwc_bwd_filter's with a
caller-allocated workspace bit for bit (the same deterministic kernels run on the same
inputs), call after call, although every call reuses the same array.

Between two calls of one problem a call with other inputs of the same shape refills the
array's slots with other values, so a partial sum that a call failed to write would change
the repeated result.  One problem is also checked against the fp64 oracle.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process (it builds and loads the
library itself)."""
from dataclasses import replace

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


def noalloc(lib, x, dy, case):
    out = torch.full((case.FH, case.FW, case.C), float("nan"), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    code = lib.dwc_bwd_filter_noalloc(x.data_ptr(), dy.data_ptr(), out.data_ptr(), case.N,
                                      case.H, case.W, case.C, case.FH, case.FW, case.stride,
                                      case.pad, DT[case.dtype], stream)
    assert code == 0, (case, code)
    return out


@pytest.mark.parametrize("case", [
    Case(8, 28, 28, 256, 13, 13, 1, 6, "f32", "normal", 41),
    Case(4, 56, 56, 128, 7, 7, 1, 3, "bf16", "normal", 42),
    Case(2, 15, 17, 24, 5, 5, 2, 2, "f32", "normal", 43),    # general kernels
], ids=lambda c: f"{c.dtype}-{c.N}x{c.H}x{c.W}x{c.C}-{c.FH}x{c.FW}-s{c.stride}")
def test_noalloc_equals_workspace_version_on_consecutive_calls(lib, case):
    other = replace(case, seed=case.seed + 100)
    x, dy = case.x().cuda(), case.dy().cuda()
    xo, dyo = other.x().cuda(), other.dy().cuda()
    F = (case.FH, case.FW)
    ref = dwc.bwd_filter(x, dy, F, case.stride, case.pad)
    ref_o = dwc.bwd_filter(xo, dyo, F, case.stride, case.pad)
    first = noalloc(lib, x, dy, case)
    between = noalloc(lib, xo, dyo, other)   # other values in the same scratch slots
    second = noalloc(lib, x, dy, case)
    torch.cuda.synchronize()
    assert dwc.device_status() == 0
    assert torch.equal(first, ref)
    assert torch.equal(between, ref_o)
    assert torch.equal(second, ref)


def test_noalloc_matches_the_oracle(lib):
    import oracle
    case = Case(3, 20, 24, 64, 7, 7, 1, 3, "f32", "normal", 45)
    x, dy = case.x(), case.dy()
    got = noalloc(lib, x.cuda(), dy.cuda(), case)
    torch.cuda.synchronize()
    xn, dyn = x.double().numpy(), dy.double().numpy()
    ref = oracle.bwd_filter(xn, dyn, (case.FH, case.FW), case.stride, case.pad)
    den = oracle.bwd_filter(abs(xn), abs(dyn), (case.FH, case.FW), case.stride, case.pad)
    assert normalized_error(got.cpu().numpy(), ref, den) <= TOL[case.dtype]


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
    # argument errors come before the size limit: a null pointer on a shape that does not
    # fit the scratch array is still DWC_ERR_INVALID_ARG, a misaligned one DWC_ERR_ALIGNMENT
    assert lib.dwc_bwd_filter_noalloc(None, 16, 16, 64, 56, 56, 16384, 31, 31, 1, 15, 0,
                                      None) == 1
    assert lib.dwc_bwd_filter_noalloc(18, 16, 16, 64, 56, 56, 16384, 31, 31, 1, 15, 0,
                                      None) == 3
