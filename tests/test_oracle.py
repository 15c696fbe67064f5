"""Pins for the fp64 CPU oracle, independent of the oracle's own code.

Each check ties the oracle to something other than itself:

* library routines: ``scipy.signal.correlate2d`` per channel (the textbook 2-D
  cross-correlation; §2.1 / Fig. 1 of "Flash-DWC: Making Depthwise Convolution
  Compute-Efficient on GPUs" reduces DWC to one such correlation per channel), torch CPU
  float64 ``conv2d(groups=C)`` and its autograd gradients (the framework the pages compare
  outputs and gradients against, §6.3.2);
* closed forms: delta filters (Y == X, shifted copies with zero fill), a constant input
  through a constant filter (valid-tap counts at the padding borders), separable filters
  (a row pass then a column pass with ``numpy.correlate``);
* identities: the adjoint relations that define both backward passes (§5.1), the
  finite-difference identity of the filter gradient, the scatter and gather forms of the
  data gradient, linearity, horizontal-flip symmetry;
* mutation checks: plausible mistakes planted in a copy of the oracle's C source (dropped
  tap, wrong pad sign, transposed filter axes, missing rotation, wrong stride) must each
  fail at least one of these pins.
"""
import itertools

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

scipy_signal = pytest.importorskip("scipy.signal")

RNG = np.random.default_rng(20260913)


def rand(*shape):
    return RNG.standard_normal(shape)


def rel_err(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    scale = max(np.abs(b).max(initial=0.0), 1e-300)
    return float(np.abs(a - b).max(initial=0.0) / scale)


def torch_fwd(x, w, s, p):
    xt = torch.from_numpy(x).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w).permute(2, 0, 1).unsqueeze(1)
    y = F.conv2d(xt, wt, stride=s, padding=p, groups=x.shape[3])
    return y.permute(0, 2, 3, 1).contiguous().numpy()


def torch_grads(x, w, dy, s, p):
    xt = torch.from_numpy(x).permute(0, 3, 1, 2).clone().requires_grad_(True)
    wt = torch.from_numpy(w).permute(2, 0, 1).unsqueeze(1).clone().requires_grad_(True)
    y = F.conv2d(xt, wt, stride=s, padding=p, groups=x.shape[3])
    y.backward(torch.from_numpy(dy).permute(0, 3, 1, 2))
    dx = xt.grad.permute(0, 2, 3, 1).contiguous().numpy()
    dw = wt.grad.squeeze(1).permute(1, 2, 0).contiguous().numpy()
    return dx, dw


def scipy_fwd(x, w, s, p):
    N, H, W, C = x.shape
    FH, FW, _ = w.shape
    xp = np.pad(x, ((0, 0), (p, p), (p, p), (0, 0)))
    OH = oracle.out_dim(H, FH, s, p)
    OW = oracle.out_dim(W, FW, s, p)
    y = np.zeros((N, OH, OW, C))
    for n in range(N):
        for c in range(C):
            full = scipy_signal.correlate2d(xp[n, :, :, c], w[:, :, c], mode="valid")
            y[n, :, :, c] = full[::s, ::s][:OH, :OW]
    return y


# (N, H, W, C, FH, FW, stride, pad): odd, even and non-square filters, strides 1-3,
# pads from 0 past F-1, filters larger than the image, single-pixel images.
SHAPES = [
    (1, 5, 5, 1, 3, 3, 1, 1),
    (2, 7, 6, 3, 3, 3, 1, 0),
    (1, 9, 8, 4, 5, 5, 1, 2),
    (2, 6, 9, 2, 3, 5, 1, 1),
    (1, 8, 7, 3, 5, 3, 2, 2),
    (1, 9, 9, 2, 7, 7, 2, 3),
    (2, 5, 7, 3, 4, 2, 1, 1),
    (1, 4, 4, 2, 7, 7, 1, 3),
    (1, 3, 5, 2, 9, 9, 1, 4),
    (1, 1, 1, 3, 3, 3, 1, 1),
    (1, 10, 11, 2, 3, 3, 3, 1),
    (1, 6, 6, 2, 3, 3, 1, 4),
    (1, 7, 9, 5, 1, 1, 1, 0),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_fwd_matches_scipy_correlate2d(shape):
    N, H, W, C, FH, FW, s, p = shape
    x, w = rand(N, H, W, C), rand(FH, FW, C)
    y = oracle.fwd(x, w, s, p)
    assert y.shape == scipy_fwd(x, w, s, p).shape
    assert rel_err(y, scipy_fwd(x, w, s, p)) < 1e-13


@pytest.mark.parametrize("shape", SHAPES)
def test_all_passes_match_torch_fp64(shape):
    N, H, W, C, FH, FW, s, p = shape
    x, w = rand(N, H, W, C), rand(FH, FW, C)
    y_ref = torch_fwd(x, w, s, p)
    y = oracle.fwd(x, w, s, p)
    assert y.shape == y_ref.shape
    assert rel_err(y, y_ref) < 1e-13
    dy = rand(*y.shape)
    dx_ref, dw_ref = torch_grads(x, w, dy, s, p)
    assert rel_err(oracle.bwd_data(dy, w, (H, W), s, p), dx_ref) < 1e-13
    assert rel_err(oracle.bwd_filter(x, dy, (FH, FW), s, p), dw_ref) < 1e-13


@pytest.mark.parametrize("F", [1, 3, 5, 7, 13])
def test_delta_filter_is_identity_bit_exact(F):
    x = rand(2, 9, 11, 5)
    w = np.zeros((F, F, 5))
    w[F // 2, F // 2, :] = 1.0
    y = oracle.fwd(x, w, 1, F // 2)
    assert np.array_equal(y, x)


@pytest.mark.parametrize("a,b", [(0, 0), (2, 1), (1, 3), (3, 3)])
def test_shifted_delta_is_shifted_copy_with_zero_fill(a, b):
    F, p = 4, 1
    N, H, W, C = 1, 6, 7, 3
    x = rand(N, H, W, C)
    w = np.zeros((F, F, C))
    w[a, b, :] = 1.0
    y = oracle.fwd(x, w, 1, p)
    OH, OW = y.shape[1:3]
    for oh, ow in itertools.product(range(OH), range(OW)):
        ih, iw = oh + a - p, ow + b - p
        want = x[0, ih, iw] if (0 <= ih < H and 0 <= iw < W) else np.zeros(C)
        assert np.array_equal(y[0, oh, ow], want)


@pytest.mark.parametrize("H,W,F,s,p", [(7, 9, 3, 1, 1), (8, 8, 5, 1, 2), (6, 7, 7, 1, 3),
                                        (9, 8, 3, 2, 1), (5, 5, 7, 1, 6), (4, 6, 5, 3, 4)])
def test_box_filter_on_constant_input_closed_form(H, W, F, s, p):
    a, b = 0.75, -1.25          # dyadic: every partial sum is exact in fp64
    x = np.full((1, H, W, 2), a)
    w = np.full((F, F, 2), b)
    y = oracle.fwd(x, w, s, p)

    def cnt(o, n_in):           # taps of output o that land inside [0, n_in)
        lo = o * s - p
        return max(0, min(n_in, lo + F) - max(0, lo))

    for oh, ow in itertools.product(range(y.shape[1]), range(y.shape[2])):
        assert np.all(y[0, oh, ow] == a * b * cnt(oh, H) * cnt(ow, W))


def test_separable_filter_row_then_column():
    N, H, W, C, F_, p = 1, 8, 9, 3, 5, 2
    x = rand(N, H, W, C)
    u, v = rand(F_, C), rand(F_, C)
    w = u[:, None, :] * v[None, :, :]
    y = oracle.fwd(x, w, 1, p)
    xp = np.pad(x, ((0, 0), (p, p), (p, p), (0, 0)))
    for c in range(C):
        rows = np.stack([np.correlate(xp[0, i, :, c], v[:, c], mode="valid")
                         for i in range(H + 2 * p)])
        cols = np.stack([np.correlate(rows[:, j], u[:, c], mode="valid")
                         for j in range(rows.shape[1])], axis=1)
        assert rel_err(y[0, :, :, c], cols) < 1e-13


@pytest.mark.parametrize("shape", SHAPES)
def test_adjoint_identities(shape):
    N, H, W, C, FH, FW, s, p = shape
    x, w = rand(N, H, W, C), rand(FH, FW, C)
    y = oracle.fwd(x, w, s, p)
    dy = rand(*y.shape)
    lhs = float(np.sum(dy * y))
    via_dx = float(np.sum(oracle.bwd_data(dy, w, (H, W), s, p) * x))
    via_dw = float(np.sum(oracle.bwd_filter(x, dy, (FH, FW), s, p) * w))
    scale = float(np.sum(np.abs(dy) * oracle.fwd(np.abs(x), np.abs(w), s, p))) + 1e-300
    assert abs(lhs - via_dx) / scale < 1e-13
    assert abs(lhs - via_dw) / scale < 1e-13


@pytest.mark.parametrize("shape", SHAPES[:8])
def test_filter_gradient_finite_difference(shape):
    """dW[fh,fw,c] = <dY, fwd(X, e_{fh,fw,c})>: exact for a linear map."""
    N, H, W, C, FH, FW, s, p = shape
    x = rand(N, H, W, C)
    OH, OW = oracle.out_dim(H, FH, s, p), oracle.out_dim(W, FW, s, p)
    dy = rand(N, OH, OW, C)
    dw = oracle.bwd_filter(x, dy, (FH, FW), s, p)
    for _ in range(6):
        fh, fw, c = RNG.integers(FH), RNG.integers(FW), RNG.integers(C)
        e = np.zeros((FH, FW, C))
        e[fh, fw, c] = 1.0
        probe = float(np.sum(dy * oracle.fwd(x, e, s, p)))
        assert abs(dw[fh, fw, c] - probe) <= 1e-13 * (abs(probe) + 1.0)


@pytest.mark.parametrize("shape", SHAPES)
def test_data_gradient_scatter_equals_gather(shape):
    N, H, W, C, FH, FW, s, p = shape
    w = rand(FH, FW, C)
    OH, OW = oracle.out_dim(H, FH, s, p), oracle.out_dim(W, FW, s, p)
    dy = rand(N, OH, OW, C)
    dx = oracle.bwd_data(dy, w, (H, W), s, p)
    idx = np.arange(dx.size)
    assert rel_err(oracle.bwd_data_at(dy, w, (H, W), idx, s, p), dx.ravel()) < 1e-13


@pytest.mark.parametrize("shape", SHAPES[:6])
def test_sampled_forms_equal_full_tensors(shape):
    N, H, W, C, FH, FW, s, p = shape
    x, w = rand(N, H, W, C), rand(FH, FW, C)
    y = oracle.fwd(x, w, s, p)
    dy = rand(*y.shape)
    iy = RNG.integers(0, y.size, 50)
    assert np.array_equal(oracle.fwd_at(x, w, iy, s, p), y.ravel()[iy])
    dw = oracle.bwd_filter(x, dy, (FH, FW), s, p)
    iw = RNG.integers(0, dw.size, 20)
    assert np.array_equal(oracle.bwd_filter_at(x, dy, (FH, FW), iw, s, p), dw.ravel()[iw])


def test_linearity_and_flip_symmetry():
    N, H, W, C, F_, p = 2, 7, 8, 3, 5, 2
    x1, x2, w1, w2 = rand(N, H, W, C), rand(N, H, W, C), rand(F_, F_, C), rand(F_, F_, C)
    a, b = 0.5, -2.0
    y = oracle.fwd(a * x1 + b * x2, w1, 1, p)
    assert rel_err(y, a * oracle.fwd(x1, w1, 1, p) + b * oracle.fwd(x2, w1, 1, p)) < 1e-13
    y = oracle.fwd(x1, a * w1 + b * w2, 1, p)
    assert rel_err(y, a * oracle.fwd(x1, w1, 1, p) + b * oracle.fwd(x1, w2, 1, p)) < 1e-13
    # flipping the image and the filter left-right flips the output (symmetric padding)
    yf = oracle.fwd(x1[:, :, ::-1], w1[:, ::-1], 1, p)
    assert rel_err(yf, oracle.fwd(x1, w1, 1, p)[:, :, ::-1]) < 1e-13
    # channel permutation equivariance
    perm = RNG.permutation(C)
    assert np.array_equal(oracle.fwd(x1[..., perm], w1[..., perm], 1, p),
                          oracle.fwd(x1, w1, 1, p)[..., perm])


# -- BN + Act + DWC (the fusion of §5.2) ------------------------------------------------

def torch_fwd_bn_act(x, w, mean, var, gamma, beta, eps, act, s, p):
    """Library form: torch's eval-mode batch_norm, relu / relu6 and grouped conv2d in fp64."""
    xt = torch.from_numpy(x).permute(0, 3, 1, 2)
    t = lambda v: torch.from_numpy(np.asarray(v, np.float64))
    z = F.batch_norm(xt, t(mean), t(var), t(gamma), t(beta), training=False, eps=eps)
    z = {"none": lambda v: v, "relu": F.relu, "relu6": F.relu6}[act](z)
    wt = torch.from_numpy(w).permute(2, 0, 1).unsqueeze(1)
    y = F.conv2d(z, wt, stride=s, padding=p, groups=x.shape[3])
    return y.permute(0, 2, 3, 1).contiguous().numpy()


def bn_params(C, spread=1.0):
    return (RNG.uniform(-0.5, 0.5, C), RNG.uniform(0.5, 2.0, C), RNG.uniform(0.5, 1.5, C) * spread,
            RNG.uniform(-0.5, 0.5, C))


@pytest.mark.parametrize("act", ["none", "relu", "relu6"])
@pytest.mark.parametrize("shape", SHAPES[:9])
def test_fwd_bn_act_matches_torch_fp64(shape, act):
    N, H, W, C, FH, FW, s, p = shape
    x, w = rand(N, H, W, C) * 3, rand(FH, FW, C)
    mean, var, gamma, beta = bn_params(C, spread=4.0)   # wide enough that ReLU6 clips
    got = oracle.fwd_bn_act(x, w, mean, var, gamma, beta, 1e-5, act, s, p)
    ref = torch_fwd_bn_act(x, w, mean, var, gamma, beta, 1e-5, act, s, p)
    assert got.shape == ref.shape and rel_err(got, ref) <= 1e-12


@pytest.mark.parametrize("act,beta,z", [("none", -2.0, -2.0), ("relu", -2.0, 0.0), ("relu", 1.5, 1.5),
                                        ("relu6", 7.25, 6.0), ("relu6", -0.5, 0.0), ("none", 0.0, 2.0)])
@pytest.mark.parametrize("H,W,F_,s,p", [(7, 9, 3, 1, 1), (6, 7, 7, 1, 3), (9, 8, 3, 2, 1), (5, 5, 7, 1, 6)])
def test_bn_act_constant_input_pads_with_zero(H, W, F_, s, p, act, beta, z):
    """x == mean + 2 with var + eps == 4 makes the normalised value exactly 1, so the BN gives
    gamma + beta; gamma is 0 except in the last case (gamma 2, beta 0).  A box filter then
    gives z * b * (taps inside the image), which holds only if the padding is zero AFTER the
    activation (padding with act(BN(0)) would add taps at the borders)."""
    C, a, b = 2, 0.75, -1.25
    gamma = 2.0 if z == 2.0 else 0.0
    x = np.full((1, H, W, C), a + 2.0)
    w = np.full((F_, F_, C), b)
    y = oracle.fwd_bn_act(x, w, [a] * C, [3.75] * C, [gamma] * C, [beta] * C, 0.25, act, s, p)

    def cnt(o, n_in):
        lo = o * s - p
        return max(0, min(n_in, lo + F_) - max(0, lo))

    for oh, ow in itertools.product(range(y.shape[1]), range(y.shape[2])):
        assert np.all(y[0, oh, ow] == z * b * cnt(oh, H) * cnt(ow, W))


def test_bn_act_identity_parameters_reduce_to_plain_forward():
    x, w = rand(2, 7, 8, 3), rand(5, 5, 3)
    y = oracle.fwd_bn_act(x, w, [0.0] * 3, [0.75] * 3, [1.0] * 3, [0.0] * 3, 0.25, "none", 1, 2)
    assert np.array_equal(y, oracle.fwd(x, w, 1, 2))


def test_fwd_bn_act_sampled_equals_full():
    x, w = rand(2, 9, 10, 4), rand(3, 3, 4)
    prm = bn_params(4)
    full = oracle.fwd_bn_act(x, w, *prm, 1e-5, "relu", 2, 1)
    idx = RNG.choice(full.size, 40, replace=False)
    assert np.array_equal(oracle.fwd_bn_act_at(x, w, *prm, 1e-5, "relu", idx, 2, 1),
                          full.ravel()[idx])


def _random_shapes(count=40, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < count:
        FH, FW = int(rng.integers(1, 8)), int(rng.integers(1, 8))
        s, p = int(rng.integers(1, 4)), int(rng.integers(0, max(FH, FW)))
        H, W = int(rng.integers(1, 12)), int(rng.integers(1, 12))
        if oracle.out_dim(H, FH, s, p) < 1 or oracle.out_dim(W, FW, s, p) < 1:
            continue
        out.append((int(rng.integers(1, 3)), H, W, int(rng.integers(1, 5)), FH, FW, s, p))
    return out


@pytest.mark.parametrize("shape", _random_shapes())
def test_random_shapes_match_torch_fp64(shape):
    """Seeded random problems (any filter 1..7 x 1..7, strides 1-3, pads 0..F-1): all three
    passes against torch's fp64 grouped conv2d and its autograd gradients."""
    N, H, W, C, FH, FW, s, p = shape
    x, w = rand(N, H, W, C), rand(FH, FW, C)
    y = oracle.fwd(x, w, s, p)
    assert y.shape == torch_fwd(x, w, s, p).shape and rel_err(y, torch_fwd(x, w, s, p)) <= 1e-12
    dy = rand(*y.shape)
    dx_ref, dw_ref = torch_grads(x, w, dy, s, p)
    assert rel_err(oracle.bwd_data(dy, w, (H, W), s, p), dx_ref) <= 1e-12
    assert rel_err(oracle.bwd_filter(x, dy, (FH, FW), s, p), dw_ref) <= 1e-12


def test_out_dim_and_empty_outputs():
    assert oracle.out_dim(56, 7, 1, 3) == 56
    assert oracle.out_dim(56, 31, 1, 15) == 56
    assert oracle.out_dim(14, 3, 2, 1) == 7
    assert oracle.out_dim(3, 7, 1, 1) == 0
    x, w = rand(1, 3, 3, 2), rand(7, 7, 2)
    assert oracle.fwd(x, w, 1, 1).shape == (1, 0, 0, 2)


# -- mutation checks: plant a mistake in a copy of the C source (on the CPU) ---------------

MUTANTS = {
    "dropped_last_tap": ("for (int fw = 0; fw < FW; ++fw) {\n            int iw = ow * s + fw - p;",
                         "for (int fw = 0; fw < FW - 1; ++fw) {\n            int iw = ow * s + fw - p;"),
    "pad_sign": ("int ih = oh * s + fh - p;\n        if (ih < 0 || ih >= H) continue;\n        for (int fw = 0; fw < FW; ++fw) {\n            int iw = ow * s + fw - p;",
                 "int ih = oh * s + fh + p;\n        if (ih < 0 || ih >= H) continue;\n        for (int fw = 0; fw < FW; ++fw) {\n            int iw = ow * s + fw - p;"),
    "filter_axes_transposed": ("acc += x[nhwc(n, ih, iw, c, H, W, C)] * w[hwc(fh, fw, c, FW, C)];\n        }\n    }\n    return acc;",
                               "acc += x[nhwc(n, ih, iw, c, H, W, C)] * w[hwc(fw, fh, c, FW, C)];\n        }\n    }\n    return acc;"),
    "bwd_data_unrotated": ("dx[nhwc(n, ih, iw, c, H, W, C)] += g * w[hwc(fh, fw, c, FW, C)];",
                           "dx[nhwc(n, ih, iw, c, H, W, C)] += g * w[hwc(FH - 1 - fh, FW - 1 - fw, c, FW, C)];"),
    "bwd_filter_stride_ignored": ("int ih = oh * s + fh - p;\n            if (ih < 0 || ih >= H) continue;\n            for (int ow = 0; ow < OW; ++ow) {",
                                  "int ih = oh + fh - p;\n            if (ih < 0 || ih >= H) continue;\n            for (int ow = 0; ow < OW; ++ow) {"),
    "bn_act_relu_dropped": ("if (act >= 1 && v < 0.0) v = 0.0;", "if (act >= 3 && v < 0.0) v = 0.0;"),
    "bn_sqrt_dropped": ("- mean[c]) / sqrt(var[c] + eps) * gamma[c] + beta[c];",
                        "- mean[c]) / (var[c] + eps) * gamma[c] + beta[c];"),
    "bn_relu6_unclipped": ("if (act == 2 && v > 6.0) v = 6.0;", "if (act == 2 && v > 7.0) v = 7.0;"),
    "fwd_channel_mixed": ("acc += x[nhwc(n, ih, iw, c, H, W, C)] * w[hwc(fh, fw, c, FW, C)];\n        }\n    }\n    return acc;",
                          "acc += x[nhwc(n, ih, iw, c, H, W, C)] * w[hwc(fh, fw, 0, FW, C)];\n        }\n    }\n    return acc;"),
}


def _pins_pass(o: "oracle.Oracle") -> bool:
    """Run the library and identity pins against one oracle build; True if all hold."""
    for shape in SHAPES[:9]:
        N, H, W, C, FH, FW, s, p = shape
        x, w = rand(N, H, W, C), rand(FH, FW, C)
        y = o.fwd(x, w, s, p)
        if y.shape != scipy_fwd(x, w, s, p).shape or rel_err(y, scipy_fwd(x, w, s, p)) > 1e-12:
            return False
        dy = rand(*y.shape)
        dx_ref, dw_ref = torch_grads(x, w, dy, s, p)
        if rel_err(o.bwd_data(dy, w, (H, W), s, p), dx_ref) > 1e-12:
            return False
        if rel_err(o.bwd_filter(x, dy, (FH, FW), s, p), dw_ref) > 1e-12:
            return False
        mean, var, gamma, beta = bn_params(C, spread=4.0)
        for act in ("none", "relu", "relu6"):
            xs = x * 3
            if rel_err(o.fwd_bn_act(xs, w, mean, var, gamma, beta, 1e-5, act, s, p),
                       torch_fwd_bn_act(xs, w, mean, var, gamma, beta, 1e-5, act, s, p)) > 1e-12:
                return False
    return True


def test_unmodified_source_passes_pins():
    assert _pins_pass(oracle.get())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    old, new = MUTANTS[name]
    src = oracle.source()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    variant = oracle.load_source_variant(src.replace(old, new, 1), name)
    assert not _pins_pass(variant), f"planted mistake {name} was not caught by the pins"
