"""Seeded synthetic inputs for depthwise 2-D convolution.

This module only draws random tensors; it holds none of the convolution's arithmetic.  Both
the CUDA path and the fp64 oracle are fed from here, so that they see identical values.

Recipe (the workloads of "Flash-DWC: Making Depthwise Convolution Compute-Efficient on
GPUs", §6.1.1 and §6.3.2, which use random synthetic tensors, no dataset):

* tensors are drawn in fp32 on the CPU from ``torch.Generator().manual_seed(seed')`` with
  ``seed' = 1000 * seed + role`` (role: x=1, w=2, dy=3), so every tensor of a case has its
  own reproducible stream;
* ``dist="uniform"`` draws U(-1, 1); ``dist="normal"`` draws N(0, 1) for activations and
  gradients and N(0, 1/(FH*FW)) for filters (fan-in scaling of the filter);
* 16-bit cases round the fp32 draw to bf16/fp16 with round-to-nearest-even
  (``Tensor.to``); the oracle then consumes exactly the rounded values.

Layouts are channels last: x and dy are N x H x W x C (dy has the output spatial size) and
the filter is FH x FW x C.

Batch-normalisation parameters for the fused BN + Act + DWC (role 4, fp32, C values each):
mean ~ U(-0.5, 0.5), var ~ U(0.25, 2), gamma ~ U(0.5, 1.5) and beta ~ U(-0.5, 0.5), so that
a ReLU clips a sizeable share of the normalised values; the fused forward input x stays
N(0, 1), scaled by 4 for ReLU6 cases so that some values clip at 6.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

ROLE_X, ROLE_W, ROLE_DY, ROLE_BN = 1, 2, 3, 4

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def out_dim(n_in: int, f: int, stride: int, pad: int) -> int:
    """Output extent floor((n_in + 2*pad - f)/stride) + 1 (0 if the filter does not fit)."""
    num = n_in + 2 * pad - f
    return 0 if num < 0 else num // stride + 1


def draw(shape, *, seed: int, role: int, dist: str = "normal", std: float = 1.0,
         dtype: str = "f32") -> torch.Tensor:
    """One seeded CPU tensor of ``shape`` in ``dtype`` ("f32", "bf16" or "f16")."""
    g = torch.Generator().manual_seed(1000 * int(seed) + int(role))
    if dist == "uniform":
        t = torch.rand(tuple(shape), generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "normal":
        t = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
        if std != 1.0:
            t = t * std
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return t.to(DTYPES[dtype]).contiguous()


@dataclass(frozen=True)
class Case:
    """One DWC problem: shapes, stride/pad, dtype, distribution and seed."""
    N: int
    H: int
    W: int
    C: int
    FH: int
    FW: int
    stride: int = 1
    pad: int = 0
    dtype: str = "f32"
    dist: str = "normal"
    seed: int = 0
    name: str = field(default="", compare=False)

    @property
    def OH(self) -> int:
        return out_dim(self.H, self.FH, self.stride, self.pad)

    @property
    def OW(self) -> int:
        return out_dim(self.W, self.FW, self.stride, self.pad)

    def x(self) -> torch.Tensor:
        return draw((self.N, self.H, self.W, self.C), seed=self.seed, role=ROLE_X,
                    dist=self.dist, dtype=self.dtype)

    def w(self) -> torch.Tensor:
        std = 1.0 if self.dist == "uniform" else (self.FH * self.FW) ** -0.5
        return draw((self.FH, self.FW, self.C), seed=self.seed, role=ROLE_W,
                    dist=self.dist, std=std, dtype=self.dtype)

    def dy(self) -> torch.Tensor:
        return draw((self.N, self.OH, self.OW, self.C), seed=self.seed, role=ROLE_DY,
                    dist=self.dist, dtype=self.dtype)

    def bn(self):
        """Batch statistics and affine parameters (mean, var, gamma, beta) of the fused
        BN + Act + DWC: C fp32 values each."""
        g = torch.Generator().manual_seed(1000 * int(self.seed) + ROLE_BN)
        u = torch.rand((4, self.C), generator=g, dtype=torch.float32)
        mean = u[0] - 0.5
        var = 0.25 + 1.75 * u[1]
        gamma = 0.5 + u[2]
        beta = u[3] - 0.5
        return tuple(t.contiguous() for t in (mean, var, gamma, beta))

    def elem_bytes(self) -> int:
        return torch.tensor([], dtype=DTYPES[self.dtype]).element_size()


# The benchmark workloads, named by what they are.
_WORKLOADS = {
    # latency / correctness case: U(-1,1), seed 0
    "fwd_f32_n1_14x14_c32_f3": Case(1, 14, 14, 32, 3, 3, 1, 1, "f32", "uniform", 0),
    # ConvNeXt-stage shape, 7x7 filter
    "f32_n64_56x56_c128_f7": Case(64, 56, 56, 128, 7, 7, 1, 3, "f32", "normal", 1),
    # large-kernel shape, 31x31 filter, bf16 inputs, fp32 accumulate/output
    "bf16_n32_56x56_c128_f31": Case(32, 56, 56, 128, 31, 31, 1, 15, "bf16", "normal", 2),
    # backward shape, 13x13 filter, fp32 and bf16
    "f32_n64_28x28_c256_f13": Case(64, 28, 28, 256, 13, 13, 1, 6, "f32", "normal", 3),
    "bf16_n64_28x28_c256_f13": Case(64, 28, 28, 256, 13, 13, 1, 6, "bf16", "normal", 3),
    # wide maps (the early stages of 224-pixel networks), 7x7 filter
    "f32_n64_112x112_c64_f7": Case(64, 112, 112, 64, 7, 7, 1, 3, "f32", "normal", 4),
    "f32_n16_224x224_c32_f7": Case(16, 224, 224, 32, 7, 7, 1, 3, "f32", "normal", 5),
    # last stage of 224-pixel networks (7x7 maps), 3x3 and 7x7 filters
    "f32_n64_7x7_c1024_f3": Case(64, 7, 7, 1024, 3, 3, 1, 1, "f32", "normal", 6),
    "f32_n64_7x7_c1024_f7": Case(64, 7, 7, 1024, 7, 7, 1, 3, "f32", "normal", 7),
}
WORKLOADS = {k: replace(v, name=k) for k, v in _WORKLOADS.items()}

SWEEP_FILTERS = (3, 5, 7, 9, 13, 17, 21, 27, 31)
SWEEP_SHAPES = ((64, 56, 56, 128), (64, 28, 28, 256), (64, 14, 14, 512), (64, 7, 7, 1024))


def sweep_cases(dtypes=("f32", "bf16")):
    """Filter sweep: every filter size over the four stage shapes, pad=(F-1)/2, stride 1."""
    out = []
    k = 100
    for dt in dtypes:
        for (N, H, W, C) in SWEEP_SHAPES:
            for F in SWEEP_FILTERS:
                k += 1
                out.append(Case(N, H, W, C, F, F, 1, (F - 1) // 2, dt, "normal", k,
                                name=f"sweep_{dt}_n{N}_{H}x{W}_c{C}_f{F}"))
    return out


LARGE_FILTERS = (41, 51)


def large_filter_cases(dtypes=("f32", "bf16")):
    """Filters beyond the sweep (41 and 51 taps, the largest the pages evaluate) over the
    four stage shapes, pad=(F-1)/2, stride 1."""
    out = []
    k = 500
    for dt in dtypes:
        for (N, H, W, C) in SWEEP_SHAPES:
            for F in LARGE_FILTERS:
                k += 1
                out.append(Case(N, H, W, C, F, F, 1, (F - 1) // 2, dt, "normal", k,
                                name=f"large_{dt}_n{N}_{H}x{W}_c{C}_f{F}"))
    return out


# Down-sampling layers of mobile networks (stride 2): N x H x W x C of the layer input and
# the filter size, pad (F-1)/2.
STRIDE2_SHAPES = ((64, 112, 112, 96, 3), (64, 56, 56, 144, 3), (64, 28, 28, 192, 3),
                  (64, 14, 14, 576, 3), (64, 56, 56, 128, 5), (64, 28, 28, 256, 5),
                  (64, 56, 56, 144, 7), (64, 28, 28, 256, 7),
                  # the down-sampling layers of large-kernel networks
                  (64, 56, 56, 128, 9), (64, 56, 56, 128, 11), (64, 56, 56, 128, 13),
                  (32, 112, 112, 96, 9))


def stride2_cases(dtypes=("f32", "bf16")):
    """Stride-2 sweep: the down-sampling shapes above, pad=(F-1)/2."""
    out = []
    k = 300
    for dt in dtypes:
        for (N, H, W, C, F) in STRIDE2_SHAPES:
            k += 1
            out.append(Case(N, H, W, C, F, F, 2, (F - 1) // 2, dt, "normal", k,
                            name=f"s2_{dt}_n{N}_{H}x{W}_c{C}_f{F}"))
    return out

