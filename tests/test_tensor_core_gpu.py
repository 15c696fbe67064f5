"""Parity of the tensor-core forward / backward-data kernels for 16-bit inputs against the
fp64 oracle, with the kernel family forced (dwc_testing_prefer_family) so that every shape
below runs on the kernel under test, whatever the automatic choice would be.

The tcgen05 kernel (family 2) tiles 128 virtual output rows that run through several
images, N output columns per column tile, groups of 2 or 4 channels and ring items of 1
to 4 filter rows, with one filter row per MMA or two (dwc_testing_tc_row_pairs: every case
runs in both forms); the cases cover
several images per tile, tall images cut into 128-row bands, several column tiles, stripe
filters, filters from 1 to 51 taps, pads from 0 to beyond (F-1)/2, channel counts that take
every channel-group size, and both output types.  The warp-level MMA kernel (family 4) keeps
its own cases."""
import numpy as np
import pytest
import torch

import depthwise_convolution_nhwc_gb300 as dwc
import oracle
from depthwise_convolution_nhwc_gb300.inputs import WORKLOADS, Case
from parity_util import TOL, normalized_error

pytestmark = pytest.mark.gpu

CODE = {"f32": 0, "bf16": 1, "f16": 2}


@pytest.fixture(scope="module")
def lib():
    dwc.build()
    lib = dwc.load_library()
    yield lib
    assert lib.dwc_testing_prefer_family(0) >= 0
    assert lib.dwc_testing_tc_row_pairs(0) >= 0


def C_(N, H, W, C, F, p=None, FW=None, seed=31):
    FW = F if FW is None else FW
    return Case(N, H, W, C, F, FW, 1, (F - 1) // 2 if p is None else p, "bf16", "normal", seed)


TC_CASES = [
    C_(1, 6, 32, 16, 27, p=13),       # filter larger than the map
    C_(2, 9, 20, 8, 15),              # two images per 128-row tile
    C_(5, 11, 13, 24, 9),             # several images per tile, last tile partial
    C_(1, 140, 20, 16, 15),           # tall image: 128-row bands
    C_(1, 4, 300, 16, 9),             # several column tiles
    C_(2, 17, 19, 64, 3),             # small filter
    C_(1, 20, 60, 32, 17),
    C_(1, 30, 45, 16, 41),
    C_(1, 20, 60, 16, 51, p=25),      # largest filter
    C_(2, 9, 9, 16, 9, p=0),          # no padding
    C_(2, 9, 9, 16, 9, p=8),          # padding beyond (F-1)/2
    C_(1, 12, 30, 8, 7, FW=21, p=3),  # stripe filters
    C_(1, 40, 24, 16, 31, FW=5, p=2),
    C_(1, 13, 50, 8, 1, FW=13, p=0),
    C_(3, 7, 7, 40, 31),              # 40 channels, map below the filter
    C_(2, 56, 56, 16, 31),            # the large-kernel stage shape, few channels
    C_(1, 1, 1, 8, 3),                # single pixel
    # groups of 4 channels with ring items of 3 or 4 filter rows, the last item shorter
    C_(8, 28, 28, 64, 13),            # items of 4 rows (13 = 3 x 4 + 1)
    C_(8, 56, 56, 64, 17),            # items of 3 rows (17 = 5 x 3 + 2)
    C_(16, 30, 40, 64, 11),           # items of 4 rows, N = 48 columns
    # even filter heights (stripe filters): the last pair of filter rows is full
    C_(2, 20, 30, 16, 8, FW=9, p=4),
    C_(1, 33, 40, 8, 12, FW=5, p=2),
]


def oracle_pair(case, name, x, w, dy):
    s, p = case.stride, case.pad
    if name == "fwd":
        return oracle.fwd(x, w, s, p), oracle.fwd(np.abs(x), np.abs(w), s, p)
    return (oracle.bwd_data(dy, w, (case.H, case.W), s, p),
            oracle.bwd_data(np.abs(dy), np.abs(w), (case.H, case.W), s, p))


def run_family(lib, family, case, out16=False, pairs=0):
    prev = lib.dwc_testing_prefer_family(family)
    prev_pairs = lib.dwc_testing_tc_row_pairs(pairs)
    try:
        args = (case.N, case.H, case.W, case.C, case.FH, case.FW, case.stride, case.pad,
                CODE[case.dtype])
        fams = [dwc.path(n, None, None, None, *args) for n in ("fwd", "bwd_data")]
        x, w, dy = case.x(), case.w(), case.dy()
        od = x.dtype if out16 else None
        y = dwc.fwd(x.cuda(), w.cuda(), case.stride, case.pad, out_dtype=od)
        dx = dwc.bwd_data(dy.cuda(), w.cuda(), (case.H, case.W), case.stride, case.pad,
                          out_dtype=od)
        torch.cuda.synchronize()
    finally:
        lib.dwc_testing_prefer_family(prev)
        lib.dwc_testing_tc_row_pairs(prev_pairs)
    assert dwc.device_status() == 0
    return fams, x, w, dy, {"fwd": y, "bwd_data": dx}


ROWS = {1: "single_rows", 2: "row_pairs"}


@pytest.mark.parametrize("pairs", [1, 2], ids=ROWS.get)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: f"n{c.N}_{c.H}x{c.W}_c{c.C}_f{c.FH}x{c.FW}_p{c.pad}")
def test_tcgen05_kernel_full_tensors(lib, case, dtype, pairs):
    case = Case(**{**case.__dict__, "dtype": dtype})
    fams, x, w, dy, got = run_family(lib, 2, case, pairs=pairs)
    assert fams == [2, 2], fams
    xn, wn, dyn = (t.double().numpy() for t in (x, w, dy))
    for name, g in got.items():
        ref, den = oracle_pair(case, name, xn, wn, dyn)
        err = normalized_error(g.cpu().numpy(), ref, den)
        assert err <= TOL[dtype], f"{name} {case}: normalized error {err:.3e}"


@pytest.mark.parametrize("pairs", [1, 2], ids=ROWS.get)
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", [TC_CASES[1], TC_CASES[3], TC_CASES[6], TC_CASES[11]],
                         ids=lambda c: f"n{c.N}_{c.H}x{c.W}_c{c.C}_f{c.FH}x{c.FW}")
def test_tcgen05_kernel_16bit_outputs_are_the_fp32_outputs_rounded(lib, case, dtype, pairs):
    case = Case(**{**case.__dict__, "dtype": dtype})
    _, _, _, _, g16 = run_family(lib, 2, case, out16=True, pairs=pairs)
    _, _, _, _, g32 = run_family(lib, 2, case, pairs=pairs)
    for name in g16:
        assert g16[name].dtype == case.x().dtype
        assert torch.equal(g16[name].cpu(), g32[name].cpu().to(g16[name].dtype)), name


def test_tcgen05_kernel_is_deterministic(lib):
    case = Case(2, 20, 40, 16, 21, 21, 1, 10, "bf16", "normal", 5)
    _, _, _, _, a = run_family(lib, 2, case)
    _, _, _, _, b = run_family(lib, 2, case)
    for name in a:
        assert torch.equal(a[name], b[name]), name


@pytest.mark.parametrize("name", ["bf16_n32_56x56_c128_f31", "bf16_n64_28x28_c256_f13"])
def test_tcgen05_kernel_full_workload_sampled(lib, name):
    """The large-kernel and backward workloads at full size on the tcgen05 kernel, in the
    launch configuration the benchmark times, checked on sampled outputs."""
    case = WORKLOADS[name]
    fams, x, w, dy, got = run_family(lib, 2, case)
    assert fams == [2, 2]
    rng = np.random.default_rng(3)
    xn, wn, dyn = (t.double().numpy() for t in (x, w, dy))
    s, p = case.stride, case.pad
    for pname, g in got.items():
        flat = g.cpu().numpy().ravel()
        idx = np.concatenate([rng.integers(0, flat.size, 2048), [0, flat.size - 1]])
        if pname == "fwd":
            ref, den = oracle.fwd_at(xn, wn, idx, s, p), oracle.fwd_at(np.abs(xn), np.abs(wn), idx, s, p)
        else:
            ref = oracle.bwd_data_at(dyn, wn, (case.H, case.W), idx, s, p)
            den = oracle.bwd_data_at(np.abs(dyn), np.abs(wn), (case.H, case.W), idx, s, p)
        err = normalized_error(flat[idx], ref, den)
        assert err <= TOL[case.dtype], f"{pname} {name}: normalized error {err:.3e}"


# The tcgen05 filter gradient (forced with family 2): the square-filter cases above that are
# not small maps (those take the small-map filter gradient first).  They cover several
# column tiles of 64 (300-wide rows), filter heights that are not a multiple of 4, filters
# to 51 taps, pads beyond (F-1)/2 and none, and tall images.
FG_CASES = [c for c in TC_CASES if c.FH == c.FW]


def run_fgrad(lib, case, family):
    prev = lib.dwc_testing_prefer_family(family)
    try:
        fam = dwc.path("bwd_filter", None, None, None, case.N, case.H, case.W, case.C, case.FH,
                       case.FW, case.stride, case.pad, CODE[case.dtype])
        x, dy = case.x(), case.dy()
        dw = dwc.bwd_filter(x.cuda(), dy.cuda(), (case.FH, case.FW), case.stride, case.pad)
        torch.cuda.synchronize()
    finally:
        lib.dwc_testing_prefer_family(prev)
    assert dwc.device_status() == 0
    return fam, x, dy, dw


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", FG_CASES, ids=lambda c: f"n{c.N}_{c.H}x{c.W}_c{c.C}_f{c.FH}_p{c.pad}")
def test_tcgen05_filter_gradient_full_tensors(lib, case, dtype):
    case = Case(**{**case.__dict__, "dtype": dtype})
    fam, x, dy, dw = run_fgrad(lib, case, 2)
    if fam != 2:
        pytest.skip("a small map: the small-map filter gradient serves it")
    xn, dyn = x.double().numpy(), dy.double().numpy()
    f_hw = (case.FH, case.FW)
    ref = oracle.bwd_filter(xn, dyn, f_hw, case.stride, case.pad)
    den = oracle.bwd_filter(np.abs(xn), np.abs(dyn), f_hw, case.stride, case.pad)
    err = normalized_error(dw.cpu().numpy(), ref, den)
    assert err <= TOL[dtype], f"{case}: normalized error {err:.3e}"


def test_tcgen05_filter_gradient_is_deterministic_and_matches_the_warp_mma_kernel(lib):
    """Every dw element is one thread's fixed-order sum of one unit's accumulator diagonal:
    two runs are bit-identical; the warp-level MMA kernel agrees within the 16-bit tolerance."""
    case = Case(3, 30, 70, 64, 27, 27, 1, 13, "bf16", "normal", 17)
    fam, x, dy, a = run_fgrad(lib, case, 2)
    assert fam == 2
    _, _, _, b = run_fgrad(lib, case, 2)
    assert torch.equal(a, b)
    fam4, _, _, c = run_fgrad(lib, case, 4)
    assert fam4 == 4
    den = oracle.bwd_filter(np.abs(x.double().numpy()), np.abs(dy.double().numpy()),
                            (case.FH, case.FW), 1, case.pad)
    assert normalized_error(a.cpu().numpy(), c.cpu().double().numpy(), den) <= TOL["bf16"]


MMA_CASES = [C_(2, 19, 26, 32, 15), C_(1, 20, 60, 16, 31), C_(1, 5, 223, 8, 13)]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", MMA_CASES, ids=lambda c: f"n{c.N}_{c.H}x{c.W}_c{c.C}_f{c.FH}")
def test_warp_mma_kernel_full_tensors(lib, case, dtype):
    case = Case(**{**case.__dict__, "dtype": dtype})
    fams, x, w, dy, got = run_family(lib, 4, case)
    assert fams == [4, 4], fams
    xn, wn, dyn = (t.double().numpy() for t in (x, w, dy))
    for name, g in got.items():
        ref, den = oracle_pair(case, name, xn, wn, dyn)
        assert normalized_error(g.cpu().numpy(), ref, den) <= TOL[dtype], name


def test_family_preference_rejects_unknown_families(lib):
    assert lib.dwc_testing_prefer_family(7) == -1
    assert lib.dwc_testing_prefer_family(3) == -1
    assert lib.dwc_testing_prefer_family(0) == 0
    assert lib.dwc_testing_tc_row_pairs(3) == -1
    assert lib.dwc_testing_tc_row_pairs(-1) == -1
    assert lib.dwc_testing_tc_row_pairs(0) == 0


def test_tcgen05_call_inside_a_cuda_graph(lib):
    """The tcgen05 path takes stream-ordered scratch (the stacked copy and the Toeplitz runs)
    during the call: captured into a CUDA graph it must record that allocation and its free,
    and every replay must give the eager call's result (here on fresh inputs each replay)."""
    assert lib.dwc_testing_prefer_family(0) >= 0
    case = Case(4, 40, 44, 64, 17, 17, 1, 8, "bf16", "normal", 61)
    x, w = case.x().cuda(), case.w().cuda()
    assert dwc.path("fwd", None, None, None, case.N, case.H, case.W, case.C, case.FH, case.FW,
                    1, case.pad, CODE["bf16"]) == 2
    xs = torch.empty_like(x)
    xs.copy_(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dwc.fwd(xs, w, 1, case.pad)          # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        yg = dwc.fwd(xs, w, 1, case.pad)
    for seed in (62, 63):
        other = Case(**{**case.__dict__, "seed": seed})
        xn = other.x().cuda()
        xs.copy_(xn)
        g.replay()
        torch.cuda.synchronize()
        assert dwc.device_status() == 0
        assert torch.equal(yg, dwc.fwd(xn, w, 1, case.pad))
