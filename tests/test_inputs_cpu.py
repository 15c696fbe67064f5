"""Host-side checks of the seeded input generators and the benchmark's workload lists (no GPU):
every case is a valid problem, draws are reproducible, and the batch-norm parameters fall in
the ranges their recipe states."""
import os
import subprocess
import sys

import torch

from depthwise_convolution_nhwc_gb300.inputs import (LARGE_FILTERS, STRIDE2_SHAPES, WORKLOADS,
                                                     Case, large_filter_cases, out_dim,
                                                     stride2_cases, sweep_cases)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_every_listed_case_is_a_valid_problem():
    cases = list(WORKLOADS.values()) + sweep_cases() + stride2_cases() + large_filter_cases()
    names = [c.name for c in cases]
    assert len(names) == len(set(names)), "workload names must be unique"
    for c in cases:
        assert c.OH >= 1 and c.OW >= 1, c
        assert c.OH == out_dim(c.H, c.FH, c.stride, c.pad)


def test_stride2_and_large_filter_sets():
    s2 = stride2_cases(("f32",))
    assert [(c.N, c.H, c.W, c.C, c.FH) for c in s2] == list(STRIDE2_SHAPES)
    assert all(c.stride == 2 and c.pad == (c.FH - 1) // 2 for c in s2)
    big = large_filter_cases(("f32", "bf16"))
    assert sorted({c.FH for c in big}) == list(LARGE_FILTERS)
    assert len(big) == 2 * 4 * len(LARGE_FILTERS)


def test_draws_are_reproducible_and_distinct_per_role():
    c = Case(2, 5, 6, 8, 3, 3, 1, 1, "bf16", "normal", 42)
    assert torch.equal(c.x(), c.x()) and torch.equal(c.w(), c.w())
    assert c.x().dtype == torch.bfloat16
    assert not torch.equal(c.x().float()[0, 0, 0, :], c.dy().float()[0, 0, 0, :])


def test_batch_norm_parameters_follow_the_recipe():
    c = Case(1, 4, 4, 512, 3, 3, 1, 1, "f32", "normal", 7)
    mean, var, gamma, beta = c.bn()
    assert all(t.shape == (512,) and t.dtype == torch.float32 for t in (mean, var, gamma, beta))
    assert mean.abs().max() <= 0.5 and beta.abs().max() <= 0.5
    assert var.min() >= 0.25 and var.max() <= 2.0
    assert gamma.min() >= 0.5 and gamma.max() <= 1.5
    again = c.bn()
    assert all(torch.equal(a, b) for a, b in zip((mean, var, gamma, beta), again))


def test_bench_knows_every_named_workload():
    """bench.py resolves every named case (the reference arm's lookup, no GPU needed)."""
    code = ("import bench, sys; from depthwise_convolution_nhwc_gb300.inputs import *; "
            "names = list(WORKLOADS) + [c.name for c in sweep_cases() + stride2_cases() + "
            "large_filter_cases()]; [bench.get_case(n) for n in names]; print(len(names))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0, out.stderr[-2000:]
    assert int(out.stdout.strip().splitlines()[-1]) > 100
