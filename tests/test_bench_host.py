"""Host logic of bench.py that needs no GPU: the per-pass DRAM accounting read from an ncu
raw-page CSV (the `roofline.traffic` figure of the benchmark line)."""
import csv
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def write_raw(path, launches):
    """An ncu raw-page CSV: header row, units row, one row per launch (name, read, write)."""
    with open(path, "w", newline="") as f:
        w = csv.writer(f)
        w.writerow(["ID", "Kernel Name", "dram__bytes_read.sum", "dram__bytes_write.sum"])
        w.writerow(["", "", "Mbyte", "Kbyte"])
        for i, (name, rd, wr) in enumerate(launches):
            w.writerow([i, name, rd, wr])


def test_cuda_core_step(bench, tmp_path):
    raw = tmp_path / "raw.csv"
    write_raw(raw, [
        ("void dwc::rows_kernel<float, 7, 7, 2, 8, 3, 0, dwc::Pair64, 1, (int)-1, float, 1>(CUtensorMap_st, CUtensorMap_st, dwc::RowsArgs)", 100.0, 50.0),
        ("void dwc::rows_kernel<float, 7, 7, 2, 8, 3, 1, dwc::Pair64, 1, (int)-1, float, 1>(CUtensorMap_st, CUtensorMap_st, dwc::RowsArgs)", 101.0, 51.0),
        ("void dwc::fgrad_kernel<float, 7, 7, dwc::FgradTile<7, 7, 0, 0, 0, 0, 1, 0, 0, 1>, 1>(CUtensorMap_st, CUtensorMap_st, dwc::FgradArgs)", 218.0, 90.0),
        ("dwc::reduce_slices4_kernel(const float4 *, int, unsigned long, float4 *)", 2.0, 25.0),
    ])
    per = bench.traffic_per_pass(str(raw))
    assert per["fwd"] == pytest.approx(100e6 + 50e3)
    assert per["bwd_data"] == pytest.approx(101e6 + 51e3)
    assert per["bwd_filter"] == pytest.approx(220e6 + 115e3)   # kernel + slice sum


def test_tcgen05_step(bench, tmp_path):
    """Each tcgen05 main kernel belongs to the pass of the preparation launched before it;
    the gradient's stacking kernel counts with its pass."""
    raw = tmp_path / "raw.csv"
    write_raw(raw, [
        ("void dwc::tc_prep_kernel<__nv_bfloat16, 0>(dwc::TcPrepArgs)", 10.0, 20.0),
        ("void dwc::tc_rows_kernel<__nv_bfloat16, float, 4, 1>(dwc::TcArgs)", 30.0, 40.0),
        ("void dwc::tc_prep_kernel<__nv_bfloat16, 1>(dwc::TcPrepArgs)", 11.0, 21.0),
        ("void dwc::tc_rows_kernel<__nv_bfloat16, float, 4, 1>(dwc::TcArgs)", 31.0, 41.0),
        ("void dwc::tc_stack_pm_kernel<__nv_bfloat16>(dwc::TcStackArgs, dwc::TcStackArgs, uint4 *, int)", 5.0, 6.0),
        ("void dwc::tc_fgrad_kernel<__nv_bfloat16, 0>(dwc::TcFgArgs)", 7.0, 8.0),
    ])
    per = bench.traffic_per_pass(str(raw))
    assert per["fwd"] == pytest.approx(40e6 + 60e3)
    assert per["bwd_data"] == pytest.approx(42e6 + 62e3)
    assert per["bwd_filter"] == pytest.approx(12e6 + 14e3)


def test_small_map_rows_by_launch_order(bench, tmp_path):
    """The 7x7-map and small-map row kernels take the rotation as an argument: the first
    launch of the step is the forward pass, the second the backward data."""
    raw = tmp_path / "raw.csv"
    write_raw(raw, [
        ("void dwc::tiny_rows_kernel<float, 3, float>(dwc::TinyArgs)", 1.0, 0.0),
        ("void dwc::tiny_rows_kernel<float, 3, float>(dwc::TinyArgs)", 2.0, 0.0),
        ("void dwc::tiny_fgrad_cluster_kernel<float, 3>(CUtensorMap_st, CUtensorMap_st, dwc::TinyFgcArgs)", 3.0, 0.0),
    ])
    per = bench.traffic_per_pass(str(raw))
    assert (per["fwd"], per["bwd_data"], per["bwd_filter"]) == pytest.approx((1e6, 2e6, 3e6))
    # a run of the forward pass alone books every row launch to it
    per = bench.traffic_per_pass(str(raw), passes=("fwd",))
    assert per["fwd"] == pytest.approx(3e6)
