"""fp64 CPU oracle for depthwise 2-D convolution (DWC).

TEST INFRASTRUCTURE ONLY.  This package is the correctness reference the CUDA library is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it.  It shares no code with the CUDA library and the library never
calls it.

The arithmetic lives in ``dwc_oracle.c`` (plain C, fp64, loop-by-loop definition of the
forward pass and both backward passes, following "Flash-DWC: Making Depthwise Convolution
Compute-Efficient on GPUs", §2.1 / Fig. 1, §2.3 and §5.1, and of the BN + Act that §5.2
fuses in front of the forward pass).  This module only compiles it
with the host C compiler and marshals numpy arrays through ``ctypes``.

Layouts (channels last, §2.3): x, y, dx, dy are N x H x W x C; the filter is FH x FW x C.
Every input is converted to float64 before the call (exact for fp32, bf16 and fp16 values),
and every result is float64.

Pins: this oracle is checked in ``tests/test_oracle.py`` against library routines
(scipy.signal.correlate2d per channel, torch CPU float64 conv2d with groups=C and its
autograd gradients), closed forms (delta filter, box filter with padding borders, separable
filters), the adjoint identities between the three passes, the finite-difference identity
for the filter gradient and the agreement of its scatter and gather backward-data forms.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dwc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libdwc_oracle.so")

_lock = threading.Lock()


def _compile(src: str, out: str) -> str:
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("oracle: no C compiler found (gcc/cc)")
    tmp = out + f".tmp{os.getpid()}"
    # -ffp-contract=off keeps every multiply and add a separate fp64 rounding, as written.
    tail = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    try:
        subprocess.run([cc, "-fopenmp"] + tail, check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run([cc] + tail, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``dwc_oracle.c`` into ``oracle/_build/libdwc_oracle.so`` (OpenMP if available)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        return _compile(_SRC, _LIB_PATH)


def _f64(a) -> np.ndarray:
    """Contiguous float64 copy/view of a numpy array or CPU torch tensor (exact widening)."""
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _idx(flat_idx) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(flat_idx, dtype=np.int64).ravel())


class Oracle:
    """ctypes front end of one compiled copy of the oracle's C source."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        i = ctypes.c_int
        shape = [i] * 8
        lib.dwc_oracle_out_dim.argtypes = [i, i, i, i]
        lib.dwc_oracle_out_dim.restype = i
        lib.dwc_oracle_max_threads.restype = i
        lib.dwc_oracle_set_threads.argtypes = [i]
        for name in ("dwc_oracle_fwd", "dwc_oracle_bwd_data", "dwc_oracle_bwd_filter"):
            getattr(lib, name).argtypes = [dp, dp, dp] + shape
            getattr(lib, name).restype = None
        for name in ("dwc_oracle_fwd_at", "dwc_oracle_bwd_data_at", "dwc_oracle_bwd_filter_at"):
            getattr(lib, name).argtypes = [dp, dp, ip, ctypes.c_long, dp] + shape
            getattr(lib, name).restype = None
        lib.dwc_oracle_bn_act.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double, i, dp,
                                          ctypes.c_long, i]
        lib.dwc_oracle_bn_act.restype = None
        self.lib = lib
        self.path = lib_path

    def out_dim(self, n_in: int, f: int, stride: int, pad: int) -> int:
        """floor((n_in + 2*pad - f) / stride) + 1, or 0 when the filter does not fit."""
        return int(self.lib.dwc_oracle_out_dim(n_in, f, stride, pad))

    def max_threads(self) -> int:
        return int(self.lib.dwc_oracle_max_threads())

    def set_threads(self, n: int) -> None:
        self.lib.dwc_oracle_set_threads(int(n))

    @staticmethod
    def _dims(x_shape, w_shape):
        N, H, W, C = (int(v) for v in x_shape)
        FH, FW, C2 = (int(v) for v in w_shape)
        if C2 != C:
            raise ValueError(f"channel mismatch: input C={C}, filter C={C2}")
        return N, H, W, C, FH, FW

    def fwd(self, x, w, stride: int = 1, pad: int = 0) -> np.ndarray:
        """Y = DWC(X, W): y[n,oh,ow,c] = sum_{fh,fw} x[n,oh*s+fh-p,ow*s+fw-p,c]*w[fh,fw,c]."""
        x, w = _f64(x), _f64(w)
        N, H, W, C, FH, FW = self._dims(x.shape, w.shape)
        OH, OW = self.out_dim(H, FH, stride, pad), self.out_dim(W, FW, stride, pad)
        y = np.zeros((N, OH, OW, C), dtype=np.float64)
        if y.size:
            self.lib.dwc_oracle_fwd(_ptr(x), _ptr(w), _ptr(y), N, H, W, C, FH, FW, stride, pad)
        return y

    def bwd_data(self, dy, w, in_hw, stride: int = 1, pad: int = 0) -> np.ndarray:
        """dX, the adjoint of ``fwd`` in X, for a forward input of spatial size in_hw=(H, W)."""
        dy, w = _f64(dy), _f64(w)
        N, OH, OW, C = (int(v) for v in dy.shape)
        FH, FW, _ = (int(v) for v in w.shape)
        H, W = (int(v) for v in in_hw)
        if (self.out_dim(H, FH, stride, pad), self.out_dim(W, FW, stride, pad)) != (OH, OW):
            raise ValueError("dy spatial size does not match the forward output of in_hw")
        dx = np.zeros((N, H, W, C), dtype=np.float64)
        if dx.size:
            self.lib.dwc_oracle_bwd_data(_ptr(dy), _ptr(w), _ptr(dx), N, H, W, C, FH, FW,
                                         stride, pad)
        return dx

    def bwd_filter(self, x, dy, f_hw, stride: int = 1, pad: int = 0) -> np.ndarray:
        """dW[fh,fw,c] = sum_{n,oh,ow} x[n,oh*s+fh-p,ow*s+fw-p,c] * dy[n,oh,ow,c]."""
        x, dy = _f64(x), _f64(dy)
        N, H, W, C = (int(v) for v in x.shape)
        FH, FW = (int(v) for v in f_hw)
        if tuple(dy.shape) != (N, self.out_dim(H, FH, stride, pad),
                               self.out_dim(W, FW, stride, pad), C):
            raise ValueError("dy shape does not match the forward output")
        dw = np.zeros((FH, FW, C), dtype=np.float64)
        if dw.size:
            self.lib.dwc_oracle_bwd_filter(_ptr(x), _ptr(dy), _ptr(dw), N, H, W, C, FH, FW,
                                           stride, pad)
        return dw

    def fwd_at(self, x, w, flat_idx, stride: int = 1, pad: int = 0) -> np.ndarray:
        """Forward outputs at flat indices of the N x OH x OW x C output, one by one."""
        x, w = _f64(x), _f64(w)
        N, H, W, C, FH, FW = self._dims(x.shape, w.shape)
        idx = _idx(flat_idx)
        out = np.zeros(idx.size, dtype=np.float64)
        self.lib.dwc_oracle_fwd_at(_ptr(x), _ptr(w), _iptr(idx), idx.size, _ptr(out),
                                   N, H, W, C, FH, FW, stride, pad)
        return out

    def bwd_data_at(self, dy, w, in_hw, flat_idx, stride: int = 1, pad: int = 0) -> np.ndarray:
        """Backward-data elements at flat indices of the N x H x W x C gradient (gather form)."""
        dy, w = _f64(dy), _f64(w)
        N, OH, OW, C = (int(v) for v in dy.shape)
        FH, FW, _ = (int(v) for v in w.shape)
        H, W = (int(v) for v in in_hw)
        idx = _idx(flat_idx)
        out = np.zeros(idx.size, dtype=np.float64)
        self.lib.dwc_oracle_bwd_data_at(_ptr(dy), _ptr(w), _iptr(idx), idx.size, _ptr(out),
                                        N, H, W, C, FH, FW, stride, pad)
        return out

    def bwd_filter_at(self, x, dy, f_hw, flat_idx, stride: int = 1, pad: int = 0) -> np.ndarray:
        """Filter-gradient elements at flat indices of the FH x FW x C gradient."""
        x, dy = _f64(x), _f64(dy)
        N, H, W, C = (int(v) for v in x.shape)
        FH, FW = (int(v) for v in f_hw)
        idx = _idx(flat_idx)
        out = np.zeros(idx.size, dtype=np.float64)
        self.lib.dwc_oracle_bwd_filter_at(_ptr(x), _ptr(dy), _iptr(idx), idx.size, _ptr(out),
                                          N, H, W, C, FH, FW, stride, pad)
        return out

    ACTS = {"none": 0, "relu": 1, "relu6": 2}

    def bn_act(self, x, mean, var, gamma, beta, eps: float, act: str) -> np.ndarray:
        """z = act((x - mean) / sqrt(var + eps) * gamma + beta) per channel (last axis), the
        BN + Act that precede a fused forward DWC; act is "none", "relu" or "relu6"."""
        x = _f64(x)
        C = int(x.shape[-1])
        prm = [_f64(v).ravel() for v in (mean, var, gamma, beta)]
        if any(v.size != C for v in prm):
            raise ValueError("BN parameters need one value per channel")
        z = np.zeros_like(x)
        if z.size:
            self.lib.dwc_oracle_bn_act(_ptr(x), *(_ptr(v) for v in prm), float(eps),
                                       self.ACTS[act], _ptr(z), z.size // C, C)
        return z

    def fwd_bn_act(self, x, w, mean, var, gamma, beta, eps: float, act: str,
                   stride: int = 1, pad: int = 0) -> np.ndarray:
        """Y = DWC(act(BN(X)), W), in the pages' order: BN, then Act, then the DWC, whose zero
        padding applies to act(BN(X))."""
        return self.fwd(self.bn_act(x, mean, var, gamma, beta, eps, act), w, stride, pad)

    def fwd_bn_act_at(self, x, w, mean, var, gamma, beta, eps: float, act: str, flat_idx,
                      stride: int = 1, pad: int = 0) -> np.ndarray:
        """Fused forward outputs at flat indices of the N x OH x OW x C output."""
        return self.fwd_at(self.bn_act(x, mean, var, gamma, beta, eps, act), w, flat_idx,
                           stride, pad)


_default = None


def get() -> Oracle:
    """The oracle compiled from ``dwc_oracle.c`` (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def load_source_variant(c_source: str, tag: str) -> Oracle:
    """Compile a modified copy of the oracle's C source (tests plant mistakes this way to
    show that the pins catch them) and return its front end."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    src = os.path.join(_BUILD_DIR, f"variant_{tag}.c")
    with open(src, "w") as f:
        f.write(c_source)
    return Oracle(_compile(src, os.path.join(_BUILD_DIR, f"libvariant_{tag}.so")))


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def out_dim(n_in, f, stride, pad):
    return get().out_dim(n_in, f, stride, pad)


def max_threads():
    return get().max_threads()


def set_threads(n):
    get().set_threads(n)


def fwd(x, w, stride=1, pad=0):
    return get().fwd(x, w, stride, pad)


def bwd_data(dy, w, in_hw, stride=1, pad=0):
    return get().bwd_data(dy, w, in_hw, stride, pad)


def bwd_filter(x, dy, f_hw, stride=1, pad=0):
    return get().bwd_filter(x, dy, f_hw, stride, pad)


def fwd_at(x, w, flat_idx, stride=1, pad=0):
    return get().fwd_at(x, w, flat_idx, stride, pad)


def bwd_data_at(dy, w, in_hw, flat_idx, stride=1, pad=0):
    return get().bwd_data_at(dy, w, in_hw, flat_idx, stride, pad)


def bwd_filter_at(x, dy, f_hw, flat_idx, stride=1, pad=0):
    return get().bwd_filter_at(x, dy, f_hw, flat_idx, stride, pad)


def bn_act(x, mean, var, gamma, beta, eps, act):
    return get().bn_act(x, mean, var, gamma, beta, eps, act)


def fwd_bn_act(x, w, mean, var, gamma, beta, eps, act, stride=1, pad=0):
    return get().fwd_bn_act(x, w, mean, var, gamma, beta, eps, act, stride, pad)


def fwd_bn_act_at(x, w, mean, var, gamma, beta, eps, act, flat_idx, stride=1, pad=0):
    return get().fwd_bn_act_at(x, w, mean, var, gamma, beta, eps, act, flat_idx, stride, pad)


__all__ = ["Oracle", "get", "load_source_variant", "source", "build", "out_dim", "max_threads", "set_threads", "fwd", "bwd_data", "bwd_filter",
           "fwd_at", "bwd_data_at", "bwd_filter_at", "bn_act", "fwd_bn_act", "fwd_bn_act_at"]
