"""bench.py prints one JSON line with the keys the benchmark contract names.  The reference
arm (the fp64 oracle on the host cores) runs on CPU; the CUDA arm needs a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args, timeout=600):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


BASE_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e")


def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--steps", "1", "--warmup", "1",
                  "--workload", "fwd_f32_n1_14x14_c32_f3", "--passes", "fwd")
    for k in BASE_KEYS:
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"].startswith("f32 N=1 14x14 C=32 3x3")


@pytest.mark.gpu
def test_cuda_arm_line():
    d = run_bench("--steps", "5", "--warmup", "3", "--e2e-steps", "2", "--no-cpu-baseline",
                  "--per-filter-steps", "1")
    for k in BASE_KEYS + ("roofline", "gpu_launches", "clocks", "per_pass"):
        assert k in d, k
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    r = d["roofline"]
    assert r["bound"] in ("hbm", "alu", "tensor") and 0 < r["frac"] < 2 and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["value"] < d["value"]  # the copies are inside the end-to-end region
    assert d["gpu_launches"] == 5 * 4  # fwd, bwd_data, filter gradient + slice sum
    assert set(d["per_pass"]) == {"fwd", "bwd_data", "bwd_filter"}
    assert e["link"]["h2d_gbs"] > 0 and e["link"]["d2h_gbs"] > 0
    # the alu roofline denominator is the fp32x2 rate measured in the same run
    alu = d["alu_peaks"]["tflops"]
    assert set(alu) == {"ffma", "ffma2", "hfma2", "bf16x2"} and all(v > 0 for v in alu.values())
    from depthwise_convolution_nhwc_gb300.inputs import SWEEP_FILTERS
    pts = d["per_filter"]["points"]
    assert {(p["dtype"], p["F"]) for p in pts} == {(dt, F) for dt in ("f32", "bf16")
                                                   for F in SWEEP_FILTERS}
    for p in pts:
        for name in ("fwd", "bwd_data", "bwd_filter"):
            assert p[name]["us"] > 0 and 0 < p[name]["frac"] < 2
