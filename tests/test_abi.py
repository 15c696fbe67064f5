"""C ABI checks that need no GPU: the library loads, exports every symbol include/*.h
declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import glob
import os
import re

import pytest

import depthwise_convolution_nhwc_gb300 as dwc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(dwc.LIB_PATH):
        dwc.build()
    return dwc.load_library()


def declared_functions():
    names = set()
    for header in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(header).read(), flags=re.S)
        names.update(re.findall(r"\b(dwc_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(dwc.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_refuses_missing_path(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        dwc.load_library(str(tmp_path / "nope.so"))


def test_status_strings_and_version(lib):
    assert lib.dwc_version() >= 100
    for code in range(7):
        assert lib.dwc_status_string(code)
    assert lib.dwc_status_string(99) == b"unknown status"


GOOD = dict(N=1, H=8, W=8, C=16, FH=3, FW=3, stride=1, pad=1, dtype=0)
FAKE = 0x10000  # never dereferenced: every case below fails validation first


def call_fwd(lib, x=FAKE, w=FAKE, y=FAKE, **kw):
    a = dict(GOOD, **kw)
    return lib.dwc_fwd(x, w, y, a["N"], a["H"], a["W"], a["C"], a["FH"], a["FW"], a["stride"],
                       a["pad"], a["dtype"], None)


@pytest.mark.parametrize("kw", [dict(dtype=7), dict(N=-1), dict(C=-2), dict(H=0), dict(W=0),
                                dict(FH=0), dict(FW=0), dict(stride=0), dict(pad=-1),
                                dict(H=2, W=2, FH=7, FW=7, pad=1)])
def test_invalid_arguments_rejected_on_host(lib, kw):
    assert call_fwd(lib, **kw) == 1
    a = dict(GOOD, **kw)
    assert lib.dwc_bwd_data(FAKE, FAKE, FAKE, a["N"], a["H"], a["W"], a["C"], a["FH"], a["FW"],
                            a["stride"], a["pad"], a["dtype"], None) == 1
    assert lib.dwc_bwd_filter(FAKE, FAKE, FAKE, a["N"], a["H"], a["W"], a["C"], a["FH"], a["FW"],
                              a["stride"], a["pad"], a["dtype"], FAKE, 1 << 20, None) == 1
    assert lib.dwc_bwd_filter_workspace_size(a["N"], a["H"], a["W"], a["C"], a["FH"], a["FW"],
                                             a["stride"], a["pad"], a["dtype"]) == 0
    assert lib.dwc_path(0, None, None, None, a["N"], a["H"], a["W"], a["C"], a["FH"], a["FW"],
                        a["stride"], a["pad"], a["dtype"]) == -1


def test_null_pointers_rejected(lib):
    assert call_fwd(lib, x=None) == 1
    assert call_fwd(lib, w=None) == 1
    assert call_fwd(lib, y=None) == 1


def test_misaligned_pointers_rejected(lib):
    assert call_fwd(lib, x=FAKE + 2) == 3          # fp32 needs 4-byte alignment
    assert call_fwd(lib, y=FAKE + 1) == 3
    assert call_fwd(lib, x=FAKE + 1, dtype=1) == 3  # bf16 needs 2-byte alignment


def call_fwd_bn_act(lib, x=FAKE, mean=FAKE, var=FAKE, gamma=FAKE, beta=FAKE, eps=1e-5, act=1,
                    w=FAKE, y=FAKE, **kw):
    a = dict(GOOD, **kw)
    return lib.dwc_fwd_bn_act(x, mean, var, gamma, beta, eps, act, w, y, a["N"], a["H"], a["W"],
                              a["C"], a["FH"], a["FW"], a["stride"], a["pad"], a["dtype"], None)


def test_fused_bn_act_arguments_rejected_on_host(lib):
    for kw in (dict(mean=None), dict(var=None), dict(gamma=None), dict(beta=None), dict(x=None),
               dict(act=3), dict(act=-1), dict(eps=-1.0), dict(eps=float("nan")),
               dict(eps=float("inf")), dict(stride=0), dict(dtype=7)):
        assert call_fwd_bn_act(lib, **kw) == 1, kw
    assert call_fwd_bn_act(lib, gamma=FAKE + 2) == 3    # BN parameters are fp32
    assert call_fwd_bn_act(lib, x=FAKE + 2) == 3


def test_fused_bn_act_path_selection(lib):
    p = lambda **kw: lib.dwc_path(3, None, None, None, *[dict(GOOD, **kw)[k] for k in
                                  ("N", "H", "W", "C", "FH", "FW", "stride", "pad", "dtype")])
    assert p() == 1 and p(FH=5, FW=5, pad=2) == 1 and p(FH=7, FW=7, pad=3, stride=2) == 1
    assert p(FH=9, FW=9, pad=4, H=20, W=20) == 0      # larger filters: general fused kernel
    assert p(stride=3) == 0 and p(C=6) == 0 and p(FH=3, FW=5) == 0
    assert p(C=8, dtype=1) == 1 and p(C=12, dtype=1) == 0


def test_output_dtype_validated_on_host(lib):
    a = dict(GOOD, C=16)
    args = [a[k] for k in ("N", "H", "W", "C", "FH", "FW", "stride", "pad")]
    for fn in (lib.dwc_fwd_ex, lib.dwc_bwd_data_ex):
        assert fn(FAKE, FAKE, FAKE, *args, 0, 1, None) == 1      # fp32 inputs, bf16 output
        assert fn(FAKE, FAKE, FAKE, *args, 1, 2, None) == 1      # bf16 inputs, fp16 output
        assert fn(FAKE, FAKE, FAKE, *args, 2, 1, None) == 1
        assert fn(FAKE, FAKE, FAKE, *args, 1, 7, None) == 1      # unknown output type
        assert fn(FAKE, FAKE, FAKE + 1, *args, 1, 1, None) == 3  # 16-bit output, odd address
        assert fn(FAKE, FAKE, None, *args, 1, 1, None) == 1


def test_size_limits(lib):
    assert call_fwd(lib, N=1 << 20, H=1 << 12, W=1 << 12, C=1 << 10) == 2


def test_workspace_rejected_when_small(lib):
    a = GOOD
    code = lib.dwc_bwd_filter(FAKE, FAKE, FAKE, a["N"], a["H"], a["W"], a["C"], a["FH"], a["FW"],
                              a["stride"], a["pad"], a["dtype"], None, 0, None)
    assert code == 4


def test_path_selection_host_logic(lib):
    p = lambda pass_, **kw: lib.dwc_path(pass_, None, None, None, *[dict(GOOD, **kw)[k] for k in
                                          ("N", "H", "W", "C", "FH", "FW", "stride", "pad", "dtype")])
    # small maps (at most 16 x 16): small-map kernels for the filters they serve best
    f5 = dict(FH=5, FW=5, pad=2)
    assert p(0) == 1 and p(2) == 1                          # 8x8, 3x3: row kernels
    assert p(0, **f5) == 3 and p(1, **f5) == 3 and p(2, **f5) == 3
    big_map = dict(H=40, W=40)
    assert p(0, **big_map) == 1 and p(1, **big_map) == 1 and p(2, **big_map) == 1
    f13 = dict(FH=13, FW=13, pad=6)
    assert p(0, H=16, W=16, **f13) == 3 and p(0, H=17, W=16, **f13) == 1
    assert p(0, H=16, W=17, **f13) == 1
    assert p(1, H=16, W=16, FH=13, FW=13, pad=0) == 3      # dy is 4 x 4, dx 16 x 16
    f9 = dict(H=16, W=16, FH=9, FW=9, pad=4)
    assert p(0, **f9) == 1 and p(2, **f9) == 3             # 16 wide, 9 taps: gradient only
    # stride 2: fast paths of all three passes for 3x3, 5x5, 7x7
    assert p(0, stride=2) == 1 and p(0, stride=2, FH=5, FW=5, pad=2) == 1
    assert p(1, stride=2) == 1 and p(2, stride=2) == 1
    assert p(1, stride=2, FH=7, FW=7, pad=3) == 1 and p(2, stride=2, FH=7, FW=7, pad=3) == 1
    # filter gradient: a row too wide for one 256-column TMA box is cut into column parts
    assert p(2, stride=2, W=300) == 1 and p(1, stride=2, W=300) == 1
    assert p(2, W=300) == 1 and p(2, W=224, FH=31, FW=31, pad=15) == 1
    # stride 2 with 9..13 taps: every pass on the fast kernels
    s2_9 = dict(stride=2, FH=9, FW=9, pad=4, H=40, W=40)
    assert p(0, **s2_9) == 1 and p(2, **s2_9) == 1 and p(1, **s2_9) == 1
    assert p(0, stride=2, FH=13, FW=13, pad=6, H=40, W=40) == 1
    assert p(0, stride=2, FH=15, FW=15, pad=7, H=40, W=40) == 0 and p(0, stride=3) == 0
    assert p(0, stride=2, C=6) == 0
    assert p(0, FH=4, FW=4) == 0               # even filter
    # stripe (non-square) filters: row and filter-gradient kernels for odd widths 1..51
    assert p(0, FH=3, FW=5) == 1 and p(1, FH=3, FW=5) == 1 and p(2, FH=3, FW=5) == 1
    assert p(2, FH=51, FW=5, pad=2, H=60, W=60) == 1 and p(2, FH=5, FW=51, pad=2, H=60, W=60) == 1
    assert p(0, FH=51, FW=5, pad=2, H=60, W=60) == 1 and p(0, FH=1, FW=7, pad=0) == 1
    assert p(0, FH=5, FW=4) == 0               # even width
    assert p(0, FH=5, FW=53, pad=26, H=60, W=60) == 0
    assert p(0, C=6) == 0                      # fp32 rows must be 16-byte multiples
    assert p(0, C=8, dtype=1, **f5) == 3 and p(0, C=8, dtype=1, **big_map) == 1
    assert p(0, C=12, dtype=1) == 0            # bf16 needs C % 8 == 0
    # 33..51 taps: row kernels, filter gradient in tap chunks
    f33 = dict(FH=33, FW=33, pad=16, H=40, W=40)
    assert p(0, **f33) == 1 and p(1, **f33) == 1 and p(2, **f33) == 1
    assert p(2, FH=51, FW=51, pad=25, H=60, W=60) == 1
    assert p(0, FH=51, FW=51, pad=25, H=60, W=60) == 1
    assert p(0, FH=53, FW=53, pad=26, H=60, W=60) == 0
    # 16-bit inputs: tensor-core kernels for large filters on wide rows
    big = dict(H=56, W=56, C=64, FH=31, FW=31, pad=15)
    assert p(0, **big, dtype=1) == 2 and p(1, **big, dtype=2) == 2 and p(2, **big, dtype=1) == 2
    assert p(0, **big) == 1 and p(2, **big) == 1          # fp32 stays on CUDA cores
    # 16-bit filter gradients: tcgen05 from 13 taps on rows of 44+ outputs (wide tiles) or of
    # 17 to 32 outputs (narrow tiles, up to 33 taps), else the warp-level MMA kernel
    # (family 4) for large filters
    assert p(2, **dict(big, FH=13, FW=13, pad=6), dtype=1) == 2
    assert p(2, **dict(big, FH=11, FW=11, pad=5), dtype=1) == 1
    assert p(2, **dict(big, W=28), dtype=1) == 2
    assert p(2, **dict(big, W=40), dtype=1) == 4
    assert p(0, **dict(big, FH=7, FW=7, pad=3), dtype=1) == 1
    # tcgen05 from 9 taps on rows of 28+ outputs, from 17 taps on 17- to 27-wide rows
    assert p(0, **dict(big, W=28, FH=9, FW=9, pad=4), dtype=1) == 2
    assert p(0, **dict(big, W=27, FH=9, FW=9, pad=4), dtype=1) == 1
    assert p(0, **dict(big, W=17), dtype=1) == 2
    assert p(0, **dict(big, W=16), dtype=1) == 1          # narrow rows: row-streaming kernel
    # 14 x 14 maps: tcgen05 from 13 taps on large batches of channel planes
    l14 = dict(N=64, H=14, W=14, C=512, dtype=1)
    assert p(0, **l14, FH=13, FW=13, pad=6) == 2 and p(1, **l14, FH=31, FW=31, pad=15) == 2
    assert p(0, **l14, FH=9, FW=9, pad=4) != 2
    # small maps stay on the small-map kernel (14 x 14 with few planes, and 7 x 7)
    m14 = dict(H=14, W=14, C=64, dtype=1)
    assert p(0, **m14, FH=31, FW=31, pad=15) == 3 and p(1, **m14, FH=31, FW=31, pad=15) == 3
    assert p(0, **m14, FH=13, FW=13, pad=6) == 3
    assert p(0, H=7, W=7, C=64, dtype=1, FH=31, FW=31, pad=15) == 3
    # an unaligned (but element-aligned) pointer falls back to the general kernels
    assert lib.dwc_path(0, FAKE + 4, None, None, 1, 8, 8, 16, 3, 3, 1, 1, 0) == 0


def test_kernel_launch_counts(lib):
    n = lambda pass_, **kw: lib.dwc_kernel_launches(pass_, *[dict(GOOD, **kw)[k] for k in
                                                    ("N", "H", "W", "C", "FH", "FW", "stride", "pad", "dtype")])
    f7 = dict(N=64, H=56, W=56, C=128, FH=7, FW=7, pad=3)
    assert n(0, **f7) == 1 and n(1, **f7) == 1 and n(2, **f7) == 2
    assert n(0, **dict(f7, C=96)) == 2                     # lane-group tail: a second launch
    assert n(3, **f7) == 2 and n(3, **dict(f7, dtype=1)) == 3   # BN + Act 7x7: apply (+ widen w) + forward
    assert n(3, **dict(f7, H=14, W=14)) == 1                # narrow rows: the fused kernel
    assert n(0, **dict(f7, C=32)) == 1                     # the tail is the only launch
    big = dict(N=32, H=56, W=56, C=128, FH=31, FW=31, pad=15, dtype=1)
    assert n(0, **big) == 2 and n(1, **big) == 2          # tcgen05: preparation + main
    assert n(2, **big) == 2                               # tcgen05 gradient: copies + main
    assert n(2, **dict(big, dtype=0)) == 2                # fp32: kernel + slice sum
    m7 = dict(N=64, H=7, W=7, C=1024, FH=3, FW=3, pad=1)
    assert n(2, **m7) == 1                               # 7x7 maps, 3 taps: clusters sum
    assert n(2, **dict(m7, FH=7, FW=7, pad=3)) == 2       # 7 taps: kernel + slice sum
    assert n(2, **dict(m7, C=1026)) == 2                 # rows not 16-byte multiples: two launches
    assert n(0, **dict(big, N=0)) == 0
    assert n(0, FH=4, FW=4, **{k: v for k, v in GOOD.items() if k not in ("FH", "FW")}) == 1
    assert n(0, stride=0) == -1


def test_wait_limit_setting_round_trips(lib):
    prev = lib.dwc_set_wait_limit_ns(5_000_000)
    try:
        assert lib.dwc_set_wait_limit_ns(7_000_000) == 5_000_000
    finally:
        assert lib.dwc_set_wait_limit_ns(prev) == 7_000_000


@pytest.mark.parametrize("args", [(4, 1, 1), (-1, 1, 1), (0, 0, 1), (0, 1, 0)])
def test_fma_probe_rejects_bad_arguments(lib, args):
    kind, blocks, iters = args
    assert lib.dwc_fma_rate_probe(kind, blocks, iters, FAKE, None) == 1
    assert lib.dwc_fma_rate_probe(0, 1, 1, None, None) == 1
