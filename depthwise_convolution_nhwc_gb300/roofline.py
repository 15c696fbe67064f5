"""Work and traffic accounting for the roofline (host logic, no GPU).

Units ("Flash-DWC: Making Depthwise Convolution Compute-Efficient on GPUs", §2.2 and the
cuBLAS matching of §6.1.1, which count 2*N*OH*OW*C*FH*FW FLOPs per pass):

* nominal FLOPs  = 2 * N * OH * OW * C * FH * FW, the same for all three passes;
* valid FLOPs    = 2 * (multiply-adds whose input tap lies inside the image), the work a
                   kernel that never multiplies padding must do (also the same for the three
                   passes: each is a re-indexing of the same set of products);
* compulsory bytes: every input read once in its dtype and every fp32 output written once
                   (fwd: X, W -> Y; bwd_data: dY, W -> dX; bwd_filter: X, dY -> dW).

Peaks: HBM bandwidth and bf16 tensor throughput are the measured values of the machine's
peak file; the fp32 multiply-add peak is measured in the benchmark's own run (the packed
fp32x2 FMA microbenchmark of the library, all SMs) and passed in; without a measurement it
falls back to the unit counts (SMs x 128 fp32 lanes x 2 FLOP x maximum SM clock).
"""
from __future__ import annotations

import json
import os

from .inputs import Case

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

GB300_SMS = 152
FP32_LANES_PER_SM = 128
GB300_MAX_SM_MHZ = 2070.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def nominal_flops(c: Case) -> int:
    return 2 * c.N * c.OH * c.OW * c.C * c.FH * c.FW


def _tap_count(n_out: int, n_in: int, f: int, s: int, p: int) -> int:
    tot = 0
    for o in range(n_out):
        lo = o * s - p
        tot += max(0, min(n_in, lo + f) - max(0, lo))
    return tot


def valid_flops(c: Case) -> int:
    return 2 * c.N * c.C * _tap_count(c.OH, c.H, c.FH, c.stride, c.pad) * \
        _tap_count(c.OW, c.W, c.FW, c.stride, c.pad)


def compulsory_bytes(c: Case, which: str) -> int:
    e = c.elem_bytes()
    nx = c.N * c.H * c.W * c.C
    ny = c.N * c.OH * c.OW * c.C
    nw = c.FH * c.FW * c.C
    if which == "fwd":
        return e * (nx + nw) + 4 * ny
    if which == "fwd_bn_act":   # plus the four per-channel BN vectors
        return e * (nx + nw) + 4 * ny + 16 * c.C
    if which == "bwd_data":
        return e * (ny + nw) + 4 * nx
    if which == "bwd_filter":
        return e * (nx + ny) + 4 * nw
    raise ValueError(which)


def derived_fp32_tflops(sm_count: int = GB300_SMS, sm_mhz: float = GB300_MAX_SM_MHZ) -> float:
    """fp32 multiply-add peak from the unit counts: SMs x 128 lanes x 2 FLOP x clock."""
    return sm_count * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


def load_peaks(path: str | None = None, fp32_tflops: float | None = None,
               sm_count: int | None = None) -> dict:
    """Measured peaks if the peak file exists, else the stated fallbacks.  `fp32_tflops`: the
    fp32 multiply-add peak measured in this run (else derived from `sm_count` SMs, default
    152, at the maximum clock)."""
    path = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    if fp32_tflops:
        fp32, fp32_src = float(fp32_tflops), "measured"
    else:
        fp32, fp32_src = derived_fp32_tflops(sm_count or GB300_SMS), "derived"
    try:
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "fp32_tflops": fp32, "fp32_source": fp32_src, "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "bf16_tflops_sustained": 1700.0, "fp32_tflops": fp32, "fp32_source": fp32_src,
                "source": "fallback"}


def roofline_time_s(c: Case, which: str, peaks: dict, tensor: bool = False) -> tuple[float, str]:
    """Lower bound on one pass's time and the resource that sets it: "hbm", "alu" (fp32
    FFMA peak, CUDA-core kernels) or "tensor" (measured 16-bit tensor peak, for the
    tensor-core kernels)."""
    t_mem = compulsory_bytes(c, which) / (peaks["hbm_gbs"] * 1e9)
    if tensor:
        t_cmp, kind = valid_flops(c) / (peaks["bf16_tflops"] * 1e12), "tensor"
    else:
        t_cmp, kind = valid_flops(c) / (peaks["fp32_tflops"] * 1e12), "alu"
    return (t_mem, "hbm") if t_mem >= t_cmp else (t_cmp, kind)
