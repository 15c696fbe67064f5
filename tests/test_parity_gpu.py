"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element by element,
on identical seeded inputs.  Full tensors at sizes the oracle finishes in seconds (several
tiles, ragged tails in every dimension), sampled outputs at the full workload sizes."""
import numpy as np
import pytest
import torch

import depthwise_convolution_nhwc_gb300 as dwc
import oracle
from depthwise_convolution_nhwc_gb300.inputs import WORKLOADS, Case, sweep_cases
from parity_util import TOL, mare, normalized_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dwc.build()
    dwc.load_library()
    yield
    assert dwc.device_status() == 0, "a kernel reported a timed-out wait"


def run_all(case: Case, passes=("fwd", "bwd_data", "bwd_filter")):
    x, w, dy = case.x(), case.w(), case.dy()
    xd, wd, dyd = x.cuda(), w.cuda(), dy.cuda()
    out = {}
    if "fwd" in passes:
        out["fwd"] = dwc.fwd(xd, wd, case.stride, case.pad)
    if "bwd_data" in passes:
        out["bwd_data"] = dwc.bwd_data(dyd, wd, (case.H, case.W), case.stride, case.pad)
    if "bwd_filter" in passes:
        out["bwd_filter"] = dwc.bwd_filter(xd, dyd, (case.FH, case.FW), case.stride, case.pad)
    torch.cuda.synchronize()
    return x, w, dy, {k: v.cpu().numpy() for k, v in out.items()}


def check_full(case: Case, passes=("fwd", "bwd_data", "bwd_filter")):
    x, w, dy, got = run_all(case, passes)
    s, p = case.stride, case.pad
    x, w, dy = (t.double().numpy() for t in (x, w, dy))
    ax, aw, ady = np.abs(x), np.abs(w), np.abs(dy)
    for name, g in got.items():
        if name == "fwd":
            ref, den = oracle.fwd(x, w, s, p), oracle.fwd(ax, aw, s, p)
        elif name == "bwd_data":
            ref = oracle.bwd_data(dy, w, (case.H, case.W), s, p)
            den = oracle.bwd_data(ady, aw, (case.H, case.W), s, p)
        else:
            ref = oracle.bwd_filter(x, dy, (case.FH, case.FW), s, p)
            den = oracle.bwd_filter(ax, ady, (case.FH, case.FW), s, p)
        assert g.shape == ref.shape, (name, g.shape, ref.shape)
        err = normalized_error(g, ref, den)
        assert err <= TOL[case.dtype], f"{name} {case}: normalized error {err:.3e} (MARE {mare(g, ref):.2e})"


def C_(N, H, W, C, F, s=1, p=None, dtype="f32", seed=7, FW=None):
    FW = F if FW is None else FW
    return Case(N, H, W, C, F, FW, s, (F - 1) // 2 if p is None else p, dtype, "normal", seed)


# Fast-path cases: several column tiles, ragged widths/heights, channel blocks with a tail.
FAST = [
    C_(1, 6, 112, 64, 7),           # filter gradient: shallower lookahead (wide fp32 rows)
    C_(1, 5, 230, 64, 7),           # filter gradient: row cut into column parts
    C_(1, 4, 300, 64, 3),
    C_(1, 5, 223, 64, 13),
    C_(1, 20, 60, 64, 51),          # 51 taps: row kernels (fwd / bwd_data), general gradient
    C_(2, 9, 40, 64, 33, p=14),
    C_(1, 30, 45, 64, 41),
    C_(1, 12, 13, 64, 45, p=22),    # map smaller than the filter, small-map kernels
    C_(2, 17, 19, 64, 3),
    C_(1, 23, 37, 128, 7),
    C_(2, 9, 70, 96, 5),            # two column tiles, channel tail of 32
    # 7x7 channel tails past a multiple of 64 (the forward and backward data run the tail as a
    # second launch on 2 / 4 lane groups)
    C_(2, 17, 29, 96, 7),
    C_(1, 20, 40, 80, 7),
    C_(1, 12, 33, 160, 7),
    C_(2, 13, 53, 96, 7),           # 7x7 filter gradient, rotated layout: padded columns, tail
    C_(3, 9, 56, 192, 7),           # rotated layout, several slices per image
    C_(1, 14, 14, 32, 3, p=1),      # fewer channels than one block
    C_(3, 11, 13, 8, 9),            # 8 channels
    C_(1, 30, 30, 64, 13),
    C_(1, 21, 45, 64, 17),
    C_(1, 40, 33, 64, 31),          # largest filter, ragged
    C_(2, 7, 7, 128, 31),           # filter much larger than the map
    C_(1, 12, 300, 64, 7),          # wide rows: several column tiles
    C_(1, 9, 9, 64, 5, p=0),        # no padding
    C_(1, 9, 9, 64, 5, p=4),        # padding larger than (F-1)/2
    C_(1, 1, 1, 64, 3),             # single pixel
    C_(2, 5, 40, 64, 11),
    # shapes aimed at the 16-bit tensor-core kernel (filters from 9 taps): wide rows (many
    # groups per tile, short bands), no padding, padding beyond (F-1)/2, odd sizes
    C_(1, 20, 200, 64, 11),
    C_(1, 9, 9, 64, 9, p=0),
    C_(1, 9, 9, 64, 9, p=8),
    C_(2, 37, 23, 16, 21),
    C_(1, 3, 70, 8, 27, p=13),
    C_(2, 19, 26, 32, 15),          # smallest filter and row width of the tensor-core rule
    # small maps (at most 16 x 16): both width classes (8, 16), every tap-offset bound
    # (3, 7, 11, 15), channel tails, batches that do not fill the last image group,
    # non-square maps, filter windows over several CTAs of the filter gradient
    C_(3, 16, 16, 40, 13),
    C_(5, 8, 8, 64, 31),
    C_(2, 16, 5, 32, 21),
    C_(2, 12, 16, 64, 23),
    C_(1, 15, 15, 32, 3, p=0),
    C_(9, 6, 6, 16, 5),
    C_(2, 16, 16, 8, 31),
    C_(7, 7, 7, 96, 7),
    C_(8, 8, 8, 96, 31),            # warp per image with the largest window of 8-wide maps
    C_(4, 8, 6, 32, 5),
    C_(2, 16, 16, 24, 9),
    # 7 x 7 maps with 3 to 7 taps and "same" padding (a thread per image and channel pair):
    # a channel tail inside one block of 32 pairs, image slices of the filter gradient with a
    # short last slice, and another padding (not that kernel)
    C_(3, 7, 7, 40, 3),
    C_(2, 7, 7, 64, 5),
    C_(77, 7, 7, 1024, 5),
    C_(2, 7, 7, 64, 5, p=1),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("case", FAST, ids=lambda c: f"n{c.N}_{c.H}x{c.W}_c{c.C}_f{c.FH}_p{c.pad}")
def test_fast_path_full_tensors(case, dtype):
    case = Case(**{**case.__dict__, "dtype": dtype})
    if dtype != "f32" and case.C % 8:
        pytest.skip("16-bit fast path needs C % 8 == 0")
    fam = dwc.path("fwd", None, None, None, case.N, case.H, case.W, case.C, case.FH, case.FW,
                   case.stride, case.pad, {"f32": 0, "bf16": 1, "f16": 2}[dtype])
    assert fam in (1, 3) or (fam in (2, 4) and dtype != "f32")
    check_full(case)


# Stride-2 fast paths of all three passes (3x3, 5x5, 7x7): ragged sizes, odd maps, pads
# 0..F-1, channel tails.
STRIDE2 = [
    C_(2, 17, 19, 64, 3, s=2),
    C_(1, 23, 37, 128, 5, s=2),
    C_(2, 9, 70, 96, 7, s=2),
    C_(3, 11, 13, 8, 3, s=2, p=0),
    C_(1, 12, 300, 64, 3, s=2),       # filter gradient: row cut into column parts
    C_(1, 8, 8, 64, 7, s=2, p=6),
    C_(2, 56, 56, 32, 5, s=2),
    C_(2, 20, 21, 64, 5, s=2, p=1),   # odd padding with a 5x5 filter
    C_(1, 30, 31, 64, 7, s=2, p=2),
    C_(6, 40, 40, 24, 3, s=2),        # many slices, C not a multiple of the channel block
    C_(1, 5, 5, 16, 7, s=2, p=3),     # map smaller than the filter
    C_(2, 21, 27, 144, 3, s=2),       # channel tails on lane groups (16 and 40 channels)
    C_(1, 20, 33, 40, 5, s=2),
    # 9 to 13 taps (backward data on the per-pixel-class kernel)
    C_(2, 30, 34, 64, 9, s=2),
    C_(1, 25, 41, 128, 11, s=2),
    C_(2, 28, 28, 64, 13, s=2),
    C_(1, 9, 11, 64, 13, s=2, p=6),   # map smaller than the filter
    C_(2, 23, 19, 72, 11, s=2, p=3),  # pad below (F-1)/2, C not a multiple of the block
]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("case", STRIDE2, ids=lambda c: f"n{c.N}_{c.H}x{c.W}_c{c.C}_f{c.FH}_p{c.pad}")
def test_stride2_fast_path(case, dtype):
    case = Case(**{**case.__dict__, "dtype": dtype})
    if dtype != "f32" and case.C % 8:
        pytest.skip("16-bit fast path needs C % 8 == 0")
    code = {"f32": 0, "bf16": 1, "f16": 2}[dtype]
    args = (case.N, case.H, case.W, case.C, case.FH, case.FW, case.stride, case.pad, code)
    assert dwc.path("fwd", None, None, None, *args) == 1
    assert dwc.path("bwd_data", None, None, None, *args) == 1
    assert dwc.path("bwd_filter", None, None, None, *args) == 1
    check_full(case)


# General-kernel cases: strides, even/non-square filters, odd channel counts.
GENERAL = [
    C_(2, 9, 11, 5, 3, s=2, p=1),
    C_(1, 12, 10, 6, 4, p=1),
    C_(2, 8, 9, 3, 3, FW=5, p=1),
    C_(1, 10, 10, 7, 5, s=3, p=2),
    C_(1, 6, 6, 16, 33, p=16),
    C_(1, 8, 8, 12, 7, dtype="bf16"),
]


@pytest.mark.parametrize("case", GENERAL, ids=lambda c: f"s{c.stride}_f{c.FH}x{c.FW}_c{c.C}_{c.dtype}")
def test_general_path_full_tensors(case):
    check_full(case)


def test_unaligned_pointers_use_general_path_correctly():
    case = C_(1, 9, 10, 16, 5)
    x, w, dy = case.x(), case.w(), case.dy()
    # offset every tensor by one element inside a larger buffer: element-aligned, not 16-B
    def shifted(t):
        buf = torch.zeros(t.numel() + 1, dtype=t.dtype, device="cuda")
        v = buf[1:].view(t.shape)
        v.copy_(t.cuda())
        return v
    xd, wd, dyd = shifted(x), shifted(w), shifted(dy)
    y = dwc.fwd(xd, wd, 1, case.pad)
    dw = dwc.bwd_filter(xd, dyd, (5, 5), 1, case.pad)
    torch.cuda.synchronize()
    assert normalized_error(y.cpu().numpy(), oracle.fwd(x, w, 1, 2),
                            oracle.fwd(x.abs(), w.abs(), 1, 2)) <= TOL["f32"]
    assert normalized_error(dw.cpu().numpy(), oracle.bwd_filter(x, dy, (5, 5), 1, 2),
                            oracle.bwd_filter(x.abs(), dy.abs(), (5, 5), 1, 2)) <= TOL["f32"]


def test_delta_filter_is_identity_bit_exact():
    for dt in ("f32", "bf16"):
        case = C_(2, 13, 21, 64, 7, dtype=dt)
        x = case.x().cuda()
        w = torch.zeros(7, 7, 64, dtype=x.dtype, device="cuda")
        w[3, 3] = 1
        y = dwc.fwd(x, w, 1, 3)
        assert torch.equal(y, x.float())
        dx = dwc.bwd_data(x, w, (13, 21), 1, 3)
        assert torch.equal(dx, x.float())


@pytest.mark.parametrize("case", [C_(4, 28, 28, 128, 13),
                                  C_(64, 7, 7, 256, 3)],     # 7x7 maps: slices summed in clusters
                         ids=lambda c: f"{c.N}x{c.H}x{c.W}x{c.C}_f{c.FH}")
def test_bwd_filter_is_deterministic(case):
    x, dy = case.x().cuda(), case.dy().cuda()
    f, p = (case.FH, case.FW), case.pad
    a = dwc.bwd_filter(x, dy, f, 1, p).clone()
    for _ in range(3):
        b = dwc.bwd_filter(x, dy, f, 1, p)
        assert torch.equal(a, b)


def test_outputs_do_not_write_outside_their_buffers():
    """Canary bytes around every output buffer stay untouched (bounds check of the stores)."""
    case = C_(2, 11, 19, 96, 7)
    x, w, dy = case.x().cuda(), case.w().cuda(), case.dy().cuda()
    pad = 4096
    for name, shape in (("fwd", (2, 11, 19, 96)), ("bwd_data", (2, 11, 19, 96)), ("bwd_filter", (7, 7, 96))):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * pad,), 1234.5, dtype=torch.float32, device="cuda")
        out = buf[pad:pad + n].view(shape)
        if name == "fwd":
            dwc.fwd(x, w, 1, 3, out=out)
        elif name == "bwd_data":
            dwc.bwd_data(dy, w, (11, 19), 1, 3, out=out)
        else:
            dwc.bwd_filter(x, dy, (7, 7), 1, 3, out=out)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == 1234.5) and torch.all(buf[pad + n:] == 1234.5), name


def test_mismatched_buffers_are_rejected():
    """A caller-supplied buffer of the wrong dtype, shape or layout is refused before any
    launch (the library sees only its pointer: a 16-bit tensor taking fp32 outputs would be
    written past its end)."""
    case = C_(2, 9, 9, 64, 3, dtype="bf16")
    x, w, dy = case.x().cuda(), case.w().cuda(), case.dy().cuda()
    with pytest.raises(ValueError):
        dwc.fwd(x, w, 1, 1, out=torch.empty(x.shape, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        dwc.bwd_data(dy, w, (9, 9), 1, 1, out=torch.empty((2, 9, 9, 32), device="cuda"))
    with pytest.raises(ValueError):
        dwc.bwd_data(dy, w, (9, 9), 1, 1, out=torch.empty((2, 9, 64, 9), device="cuda").transpose(2, 3))
    with pytest.raises(ValueError):
        dwc.bwd_filter(x, dy[:1], (3, 3), 1, 1)
    with pytest.raises(ValueError):
        dwc.bwd_filter(x, dy, (3, 3), 1, 1, out=torch.empty((3, 3, 64), dtype=torch.bfloat16, device="cuda"))
    y = dwc.fwd(x, w, 1, 1, out=torch.empty(x.shape, dtype=torch.bfloat16, device="cuda"),
                out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert y.dtype == torch.bfloat16


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs two visible GPUs")
def test_second_device_after_first():
    """Kernels that opt in to more than 48 KiB of shared memory do so on every device they
    run on (the opt-in is per device): the same calls on GPU 1 after GPU 0 agree bit for bit."""
    case = C_(2, 28, 28, 128, 7)
    res = []
    for d in (0, 1):
        with torch.cuda.device(d):
            x, w, dy = (t.to(f"cuda:{d}") for t in (case.x(), case.w(), case.dy()))
            y = dwc.fwd(x, w, 1, 3)
            dx = dwc.bwd_data(dy, w, (28, 28), 1, 3)
            dw = dwc.bwd_filter(x, dy, (7, 7), 1, 3)
            torch.cuda.synchronize()
            res.append([t.cpu() for t in (y, dx, dw)])
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_empty_batch():
    x = torch.zeros(0, 8, 8, 64, device="cuda")
    w = torch.randn(3, 3, 64, device="cuda")
    assert dwc.fwd(x, w, 1, 1).shape == (0, 8, 8, 64)
    dw = dwc.bwd_filter(x, torch.zeros(0, 8, 8, 64, device="cuda"), (3, 3), 1, 1)
    torch.cuda.synchronize()
    assert torch.all(dw == 0)


def test_empty_batch_every_entry_point():
    """N = 0 through the stride-2, stripe, fused and 16-bit-output paths: empty outputs and a
    zero filter gradient, no launch errors."""
    x = torch.zeros(0, 9, 9, 64, device="cuda", dtype=torch.bfloat16)
    for (F, s) in ((3, 2), (7, 1)):
        w = torch.randn(F, F, 64, device="cuda").bfloat16()
        OH = (9 + 2 * ((F - 1) // 2) - F) // s + 1
        y = dwc.fwd(x, w, s, (F - 1) // 2, out_dtype=torch.bfloat16)
        dx = dwc.bwd_data(torch.zeros(0, OH, OH, 64, device="cuda").bfloat16(), w, (9, 9), s,
                          (F - 1) // 2, out_dtype=torch.bfloat16)
        dw = dwc.bwd_filter(x, torch.zeros(0, OH, OH, 64, device="cuda").bfloat16(), (F, F), s,
                            (F - 1) // 2)
        torch.cuda.synchronize()
        assert y.shape == (0, OH, OH, 64) and dx.shape == (0, 9, 9, 64) and torch.all(dw == 0)
    ws = torch.randn(7, 3, 64, device="cuda").bfloat16()       # stripe filter
    dw = dwc.bwd_filter(x, torch.zeros(0, 5, 9, 64, device="cuda").bfloat16(), (7, 3), 1, 1)
    y = dwc.fwd(x, ws, 1, 1)
    prm = [torch.ones(64, device="cuda") for _ in range(4)]
    yb = dwc.fwd_bn_act(torch.zeros(0, 9, 9, 64, device="cuda"), torch.randn(3, 3, 64, device="cuda"),
                        *prm, 1e-5, "relu", 1, 1)
    torch.cuda.synchronize()
    assert torch.all(dw == 0) and y.shape == (0, 5, 9, 64) and yb.shape == (0, 9, 9, 64)
    assert dwc.device_status() == 0


# ---- full workload sizes: sampled outputs the oracle computes one by one ----------------

def check_sampled(case: Case, passes, n_samples=2048, seed=0):
    x, w, dy, got = run_all(case, passes)
    rng = np.random.default_rng(seed)
    s, p = case.stride, case.pad
    x, w, dy = (t.double().numpy() for t in (x, w, dy))   # exact widening, once
    ax, aw, ady = np.abs(x), np.abs(w), np.abs(dy)
    for name, g in got.items():
        flat = g.ravel()
        idx = rng.integers(0, flat.size, n_samples)
        # always include the corners of the tensor (borders and the ragged tail)
        idx = np.concatenate([idx, [0, flat.size - 1, flat.size // 2]])
        if name == "fwd":
            ref, den = oracle.fwd_at(x, w, idx, s, p), oracle.fwd_at(ax, aw, idx, s, p)
        elif name == "bwd_data":
            ref = oracle.bwd_data_at(dy, w, (case.H, case.W), idx, s, p)
            den = oracle.bwd_data_at(ady, aw, (case.H, case.W), idx, s, p)
        else:
            ref = oracle.bwd_filter_at(x, dy, (case.FH, case.FW), idx, s, p)
            den = oracle.bwd_filter_at(ax, ady, (case.FH, case.FW), idx, s, p)
        err = normalized_error(flat[idx], ref, den)
        assert err <= TOL[case.dtype], f"{name} {case}: normalized error {err:.3e}"


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_workloads_full_size_sampled(name):
    case = WORKLOADS[name]
    passes = ("fwd",) if name.startswith("fwd_") else ("fwd", "bwd_data", "bwd_filter")
    if name == "fwd_f32_n1_14x14_c32_f3":
        check_full(case, passes)
    else:
        check_sampled(case, passes)


def test_sweep_full_size_sampled():
    """Every filter size of the sweep on every stage shape, fp32 and bf16, all passes."""
    for case in sweep_cases():
        check_sampled(case, ("fwd", "bwd_data", "bwd_filter"), n_samples=256, seed=case.seed)


# -- BN + Act + forward DWC (the fusion of §5.2) -----------------------------------------

BNACT = [
    C_(2, 17, 19, 64, 3),
    C_(1, 23, 37, 128, 5),
    C_(2, 9, 70, 96, 7),            # two column tiles, channel tail
    C_(1, 12, 300, 64, 7),          # many column tiles: interior lanes and both borders
    C_(3, 11, 13, 8, 3, p=0),
    C_(1, 9, 9, 64, 5, p=4),        # padding beyond (F-1)/2: whole rows in the padding
    C_(1, 1, 1, 64, 3),
    C_(2, 17, 19, 64, 3, s=2),
    C_(1, 23, 37, 128, 5, s=2),
    C_(1, 30, 31, 64, 7, s=2, p=2),
    C_(1, 8, 8, 64, 7, s=2, p=6),
]
# the general fused kernel: larger filters, stride 3, odd channel counts
BNACT_GENERAL = [C_(1, 12, 13, 64, 9), C_(1, 10, 10, 7, 5, s=3, p=2), C_(2, 9, 11, 5, 3, s=2, p=1)]


def bnact_denominator(xn, wn, prm, eps, stride, pad, idx=None):
    """Error scale of a fused output: the sum over its taps of the magnitudes that form each
    product, (|x| + |mean|) * |scale| + |beta| times |w|.  The BN value carries a rounding
    error of that size before the activation, and the activation (1-Lipschitz) does not
    shrink it: near zero the fp32 and fp64 values may fall on either side of the ReLU."""
    mean, var, gamma, beta = prm
    mag = oracle.bn_act(np.abs(xn), -np.abs(mean), var, np.abs(gamma), np.abs(beta), eps, "none")
    if idx is None:
        return oracle.fwd(mag, np.abs(wn), stride, pad)
    return oracle.fwd_at(mag, np.abs(wn), idx, stride, pad)


def check_bnact(case, act, expect_path=None):
    x, w = case.x(), case.w()
    if act == "relu6":
        x = (x.float() * 4).to(x.dtype)      # some normalised values beyond 6
    mean, var, gamma, beta = case.bn()
    eps = 1e-5
    if expect_path is not None:
        code = {"f32": 0, "bf16": 1, "f16": 2}[case.dtype]
        assert dwc.path("fwd_bn_act", None, None, None, case.N, case.H, case.W, case.C, case.FH,
                        case.FW, case.stride, case.pad, code) == expect_path
    y = dwc.fwd_bn_act(x.cuda(), w.cuda(), mean.cuda(), var.cuda(), gamma.cuda(), beta.cuda(),
                       eps, act, case.stride, case.pad)
    torch.cuda.synchronize()
    xn, wn = x.double().numpy(), w.double().numpy()
    prm = [t.double().numpy() for t in (mean, var, gamma, beta)]
    ref = oracle.fwd_bn_act(xn, wn, *prm, eps, act, case.stride, case.pad)
    den = bnact_denominator(xn, wn, prm, eps, case.stride, case.pad)
    g = y.cpu().numpy()
    assert g.shape == ref.shape
    err = normalized_error(g, ref, den)
    assert err <= TOL[case.dtype], f"fwd_bn_act {act} {case}: normalized error {err:.3e}"


@pytest.mark.parametrize("act", ["none", "relu", "relu6"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("case", BNACT, ids=lambda c: f"n{c.N}_{c.H}x{c.W}_c{c.C}_f{c.FH}_s{c.stride}_p{c.pad}")
def test_fwd_bn_act_fast_path(case, dtype, act):
    case = Case(**{**case.__dict__, "dtype": dtype})
    if dtype != "f32" and case.C % 8:
        pytest.skip("16-bit fast path needs C % 8 == 0")
    check_bnact(case, act, expect_path=1)


@pytest.mark.parametrize("act", ["none", "relu", "relu6"])
@pytest.mark.parametrize("case", BNACT_GENERAL, ids=lambda c: f"f{c.FH}_s{c.stride}_c{c.C}")
def test_fwd_bn_act_general_path(case, act):
    check_bnact(case, act, expect_path=0)


def test_fwd_bn_act_full_workload_sampled():
    """The fused kernel at the 7x7 benchmark shape, checked on sampled outputs."""
    case = WORKLOADS["f32_n64_56x56_c128_f7"]
    x, w = case.x(), case.w()
    mean, var, gamma, beta = case.bn()
    y = dwc.fwd_bn_act(x.cuda(), w.cuda(), mean.cuda(), var.cuda(), gamma.cuda(), beta.cuda(),
                       1e-5, "relu", case.stride, case.pad)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    idx = rng.choice(y.numel(), 4096, replace=False)
    # include the four corners of the first image's first channel block
    OH, OW, C = y.shape[1], y.shape[2], y.shape[3]
    idx = np.concatenate([idx, [0, (OW - 1) * C, (OH - 1) * OW * C, (OH * OW - 1) * C]])
    xn, wn = x.double().numpy(), w.double().numpy()
    prm = [t.double().numpy() for t in (mean, var, gamma, beta)]
    ref = oracle.fwd_bn_act_at(xn, wn, *prm, 1e-5, "relu", idx, case.stride, case.pad)
    den = bnact_denominator(xn, wn, prm, 1e-5, case.stride, case.pad, idx)
    err = normalized_error(y.cpu().numpy().ravel()[idx], ref, den)
    assert err <= TOL["f32"], err


# -- 16-bit outputs (forward and backward data, outputs of the input's own type) ----------

OUT16 = [
    C_(2, 17, 19, 64, 3),           # row kernels
    C_(1, 23, 37, 128, 7),
    C_(1, 20, 60, 64, 17),          # tensor-core kernels (wide rows, 17 taps)
    C_(2, 7, 7, 128, 9),            # small-map kernels
    C_(3, 7, 7, 64, 3),             # 7x7 maps, thread per image and channel pair
    C_(2, 7, 7, 128, 7),
    C_(8, 8, 8, 256, 31),           # warp per image, large window (shared-memory plan)
    C_(2, 17, 19, 64, 3, s=2),      # stride-2 kernels
    C_(1, 23, 37, 128, 7, s=2),
    C_(1, 10, 10, 16, 5, s=3, p=2), # general kernels
    # channel tails on lane groups (16-bit outputs too): C below and above 64
    C_(2, 15, 21, 40, 7),
    C_(1, 19, 23, 88, 7),
    C_(2, 16, 17, 24, 3),
    C_(1, 21, 27, 144, 7, s=2),
    C_(2, 20, 22, 48, 5, s=2),
    # stride 2 with 9 to 13 taps
    C_(1, 25, 29, 64, 11, s=2),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("case", OUT16, ids=lambda c: f"n{c.N}_{c.H}x{c.W}_c{c.C}_f{c.FH}_s{c.stride}")
def test_16bit_outputs(case, dtype):
    case = Case(**{**case.__dict__, "dtype": dtype})
    x, w, dy = case.x(), case.w(), case.dy()
    td = x.dtype
    y = dwc.fwd(x.cuda(), w.cuda(), case.stride, case.pad, out_dtype=td)
    dx = dwc.bwd_data(dy.cuda(), w.cuda(), (case.H, case.W), case.stride, case.pad, out_dtype=td)
    torch.cuda.synchronize()
    assert y.dtype == td and dx.dtype == td
    s, p = case.stride, case.pad
    xn, wn, dyn = (t.double().numpy() for t in (x, w, dy))
    # fp16 outputs below 2**-14 are subnormal: their rounding error is absolute, up to half
    # the spacing 2**-24, on top of the normalised bound (bf16 keeps fp32's exponent range)
    quantum = 2.0 ** -25 if dtype == "f16" else 0.0

    def check(name, got, ref, den):
        got = got.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        bad = np.abs(got - ref) > TOL[dtype] * den + quantum
        assert not bad.any(), f"{name} {case}: {int(bad.sum())} elements beyond the bound"

    check("fwd", y, oracle.fwd(xn, wn, s, p), oracle.fwd(np.abs(xn), np.abs(wn), s, p))
    check("bwd_data", dx, oracle.bwd_data(dyn, wn, (case.H, case.W), s, p),
          oracle.bwd_data(np.abs(dyn), np.abs(wn), (case.H, case.W), s, p))
    # the 16-bit output is the fp32 output rounded once to nearest even
    y32 = dwc.fwd(x.cuda(), w.cuda(), s, p)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), y32.cpu().to(td))



# -- stripe (non-square) filters: row and filter-gradient kernels with the filter height read
# at run time ---------------------------------------------------------------------------------

STRIPES = [
    C_(2, 17, 19, 64, 7, FW=1, p=0),     # 7 x 1
    C_(2, 17, 19, 64, 1, FW=7, p=0),     # 1 x 7
    C_(1, 23, 37, 64, 5, FW=3, p=1),
    C_(1, 23, 37, 64, 3, FW=7, p=1),
    C_(1, 60, 40, 64, 51, FW=5, p=2),    # SLaK-style stripes
    C_(1, 20, 70, 64, 5, FW=51, p=2),    # (16-bit: tensor-core kernel, rows >= 24 wide)
    C_(2, 30, 45, 96, 13, FW=3, p=4),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("case", STRIPES, ids=lambda c: f"n{c.N}_{c.H}x{c.W}_c{c.C}_f{c.FH}x{c.FW}_p{c.pad}")
def test_stripe_filters(case, dtype):
    case = Case(**{**case.__dict__, "dtype": dtype})
    code = {"f32": 0, "bf16": 1, "f16": 2}[dtype]
    args = (case.N, case.H, case.W, case.C, case.FH, case.FW, case.stride, case.pad, code)
    assert dwc.path("fwd", None, None, None, *args) in ((1,) if dtype == "f32" else (1, 2, 4))
    assert dwc.path("bwd_data", None, None, None, *args) in ((1,) if dtype == "f32" else (1, 2, 4))
    assert dwc.path("bwd_filter", None, None, None, *args) == 1
    check_full(case)


# -- seeded random shapes across every dispatch branch ------------------------------------

def random_cases(count=120, seed=20261203):
    """Valid problems drawn at random: maps 1..70 (some up to 300 wide, some small maps),
    channel counts that keep the fast-path layout rule or break it, square odd filters
    3..51, stripes, even filters, strides 1..3, pads 0..F-1, every input dtype."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        dtype = ["f32", "bf16", "f16"][rng.integers(3)]
        s = int(rng.choice([1, 1, 1, 1, 2, 2, 3]))
        kind = rng.integers(5)
        if kind == 0:
            FH = FW = int(rng.choice([3, 5, 7]))
        elif kind == 1:
            FH = FW = int(rng.choice([9, 13, 17, 25, 31, 41, 51]))
        elif kind == 2:
            FH, FW = int(rng.integers(1, 32)), int(rng.choice([1, 3, 5, 7, 9, 15, 21]))
        elif kind == 3:
            FH = FW = int(rng.choice([9, 13, 21, 31]))
        else:
            FH = FW = int(rng.choice([2, 4, 6]))
        pad = int(rng.integers(0, max(FH, FW)))
        if kind == 3:   # small maps
            H, W = int(rng.integers(max(1, FH - 2 * pad), 17)), int(rng.integers(max(1, FW - 2 * pad), 17))
        else:
            H = int(rng.integers(max(1, FH - 2 * pad), 40))
            W = int(rng.choice([rng.integers(max(1, FW - 2 * pad), 70), rng.integers(100, 300)]))
        C = int(rng.choice([8, 16, 24, 64, 96, 128, 136, 5]))
        N = int(rng.integers(1, 3))
        case = Case(N, H, W, C, FH, FW, s, pad, dtype, "normal", int(rng.integers(1 << 20)))
        if case.OH < 1 or case.OW < 1:
            continue
        if N * H * W * C * FH * FW > 60_000_000:   # keep the fp64 oracle within seconds
            continue
        out.append(case)
    return out


@pytest.mark.parametrize("case", random_cases(),
                         ids=lambda c: f"{c.dtype}_n{c.N}_{c.H}x{c.W}_c{c.C}_f{c.FH}x{c.FW}_s{c.stride}_p{c.pad}")
def test_random_shapes_all_passes(case):
    check_full(case)


# -- channel counts that are not a multiple of 64: the tail block on lane groups ----------

TAILS = [C_(2, 13, 37, c, f) for c, f in
         ((8, 3), (16, 5), (24, 7), (32, 3), (40, 5), (72, 7), (80, 3), (96, 5), (136, 7), (144, 3))]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", TAILS, ids=lambda c: f"c{c.C}_f{c.FH}")
def test_channel_tail_lane_groups(case, dtype):
    case = Case(**{**case.__dict__, "dtype": dtype})
    if dtype != "f32" and case.C % 8:
        pytest.skip("16-bit fast path needs C % 8 == 0")
    check_full(case)
