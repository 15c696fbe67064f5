"""GB300 depthwise 2-D convolution (DWC), channels last, forward + both backward passes.

Thin ctypes binding over the C ABI in ``include/dwc.h`` (``libdwc_gb300.so``, built from
``csrc/`` for sm_103a).  The binding only marshals arguments: it checks tensor shapes,
allocates outputs and workspaces with PyTorch (used for device memory and streams only) and
calls ``dwc_fwd`` / ``dwc_fwd_bn_act`` / ``dwc_bwd_data`` / ``dwc_bwd_filter`` on the current
CUDA stream.  Every
step of the computation runs in the library's CUDA kernels; there is no CPU fallback, and a
missing library is an error.

Layouts ("Flash-DWC: Making Depthwise Convolution Compute-Efficient on GPUs", §2.3):
``x``/``dx`` are N x H x W x C, ``y``/``dy`` are N x OH x OW x C, ``w``/``dw`` are
FH x FW x C, all contiguous.  Inputs are fp32, bf16 or fp16 (one dtype per call); outputs
are always fp32.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .inputs import out_dim

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdwc_gb300.so")

DWC_F32, DWC_BF16, DWC_F16 = 0, 1, 2
ACTS = {"none": 0, "relu": 1, "relu6": 2}   # dwc_act_t
STATUS = {0: "DWC_OK", 1: "DWC_ERR_INVALID_ARG", 2: "DWC_ERR_UNSUPPORTED",
          3: "DWC_ERR_ALIGNMENT", 4: "DWC_ERR_WORKSPACE", 5: "DWC_ERR_CUDA",
          6: "DWC_ERR_TIMEOUT"}

# Every symbol include/*.h declares (checked by the tests).
EXPORTS = ("dwc_fwd", "dwc_fwd_ex", "dwc_fwd_bn_act", "dwc_bwd_data", "dwc_bwd_data_ex",
           "dwc_bwd_filter_workspace_size", "dwc_bwd_filter", "dwc_bwd_filter_noalloc",
           "dwc_device_status", "dwc_set_wait_limit_ns", "dwc_fma_rate_probe",
           "dwc_status_string", "dwc_version", "dwc_path", "dwc_kernel_launches",
           "dwc_testing_stall_next_row_launch", "dwc_testing_prefer_family",
           "dwc_testing_tc_row_pairs")
FMA_KINDS = {"ffma": 0, "ffma2": 1, "hfma2": 2, "bf16x2": 3}  # dwc_fma_rate_probe kinds

_lock = threading.Lock()
_lib = None


class DwcError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({status_string(code)})")


def build(verbose: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(verbose=verbose)


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libdwc_gb300.so and declare the C signatures.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it with depthwise_convolution_nhwc_gb300.build() "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(p)
        i, vp, sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        shape = [i] * 8
        lib.dwc_fwd.argtypes = [vp, vp, vp] + shape + [i, vp]
        lib.dwc_fwd.restype = i
        lib.dwc_fwd_bn_act.argtypes = [vp, vp, vp, vp, vp, ctypes.c_float, i, vp, vp] + shape + [i, vp]
        lib.dwc_fwd_bn_act.restype = i
        lib.dwc_fwd_ex.argtypes = [vp, vp, vp] + shape + [i, i, vp]
        lib.dwc_fwd_ex.restype = i
        lib.dwc_bwd_data_ex.argtypes = [vp, vp, vp] + shape + [i, i, vp]
        lib.dwc_bwd_data_ex.restype = i
        lib.dwc_bwd_data.argtypes = [vp, vp, vp] + shape + [i, vp]
        lib.dwc_bwd_data.restype = i
        lib.dwc_bwd_filter_workspace_size.argtypes = shape + [i]
        lib.dwc_bwd_filter_workspace_size.restype = sz
        lib.dwc_bwd_filter.argtypes = [vp, vp, vp] + shape + [i, vp, sz, vp]
        lib.dwc_bwd_filter.restype = i
        lib.dwc_bwd_filter_noalloc.argtypes = [vp, vp, vp] + shape + [i, vp]
        lib.dwc_bwd_filter_noalloc.restype = i
        lib.dwc_device_status.argtypes = [vp]
        lib.dwc_device_status.restype = i
        lib.dwc_status_string.argtypes = [i]
        lib.dwc_status_string.restype = ctypes.c_char_p
        lib.dwc_version.argtypes = []
        lib.dwc_version.restype = i
        lib.dwc_path.argtypes = [i, vp, vp, vp] + shape + [i]
        lib.dwc_path.restype = i
        lib.dwc_kernel_launches.argtypes = [i] + shape + [i]
        lib.dwc_kernel_launches.restype = i
        lib.dwc_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        lib.dwc_set_wait_limit_ns.restype = ctypes.c_ulonglong
        lib.dwc_fma_rate_probe.argtypes = [i, i, i, vp, vp]
        lib.dwc_fma_rate_probe.restype = i
        lib.dwc_testing_stall_next_row_launch.argtypes = []
        lib.dwc_testing_stall_next_row_launch.restype = None
        lib.dwc_testing_prefer_family.argtypes = [i]
        lib.dwc_testing_prefer_family.restype = i
        lib.dwc_testing_tc_row_pairs.argtypes = [i]
        lib.dwc_testing_tc_row_pairs.restype = i
        if path is None:
            _lib = lib
        return lib


def status_string(code: int) -> str:
    return load_library().dwc_status_string(int(code)).decode()


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return DWC_F32
    if t.dtype == torch.bfloat16:
        return DWC_BF16
    if t.dtype == torch.float16:
        return DWC_F16
    raise TypeError(f"unsupported dtype {t.dtype} (fp32, bf16 or fp16)")


def _stream_ptr(stream) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _check_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device (no CPU fallback)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous (channels-last dims N,H,W,C)")


def _check_buffer(t, shape, dtype, device, what):
    """A caller-supplied tensor must be exactly what the kernels read or write: the library
    sees only its pointer."""
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != device:
        raise ValueError(f"{what} must be a {tuple(shape)} {dtype} tensor on {device} "
                         f"(got {tuple(t.shape)} {t.dtype} on {t.device})")
    _check_cuda(t)


def _call(fn: str, *args):
    code = getattr(load_library(), fn)(*args)
    if code != 0:
        raise DwcError(fn, code)


def fwd(x, w, stride: int = 1, pad: int = 0, out=None, stream=None, out_dtype=None):
    """Y[n,oh,ow,c] = sum_{fh,fw} X[n,oh*s+fh-p,ow*s+fw-p,c] * W[fh,fw,c].  Output fp32, or
    out_dtype = the 16-bit input's own dtype (fp32 result rounded once at the store)."""
    torch = _torch()
    _check_cuda(x, w)
    N, H, W, C = x.shape
    FH, FW, C2 = w.shape
    if C2 != C or w.dtype != x.dtype:
        raise ValueError("filter must be FH x FW x C with the input's dtype")
    od = torch.float32 if out_dtype is None else out_dtype
    OH, OW = out_dim(H, FH, stride, pad), out_dim(W, FW, stride, pad)
    if out is None:
        out = torch.empty((N, max(OH, 0), max(OW, 0), C), device=x.device, dtype=od)
    else:
        _check_buffer(out, (N, max(OH, 0), max(OW, 0), C), od, x.device, "out")
    if od == torch.float32:
        _call("dwc_fwd", x.data_ptr(), w.data_ptr(), out.data_ptr(), N, H, W, C, FH, FW, stride,
              pad, _dtype_code(x), _stream_ptr(stream))
    else:
        _call("dwc_fwd_ex", x.data_ptr(), w.data_ptr(), out.data_ptr(), N, H, W, C, FH, FW, stride,
              pad, _dtype_code(x), _dtype_code(torch.empty(0, dtype=od)), _stream_ptr(stream))
    return out


def fwd_bn_act(x, w, mean, var, gamma, beta, eps: float = 1e-5, act: str = "relu",
               stride: int = 1, pad: int = 0, out=None, stream=None):
    """Y = DWC(act(BN(X)), W) in one pass: BN(X) = (X - mean) / sqrt(var + eps) * gamma + beta
    per channel, act "none" / "relu" / "relu6"; the DWC zero-pads act(BN(X)).  mean, var,
    gamma, beta: C fp32 values each on the device (fp32 output)."""
    torch = _torch()
    _check_cuda(x, w, mean, var, gamma, beta)
    N, H, W, C = x.shape
    FH, FW, C2 = w.shape
    if C2 != C or w.dtype != x.dtype:
        raise ValueError("filter must be FH x FW x C with the input's dtype")
    for t in (mean, var, gamma, beta):
        if t.dtype != torch.float32 or t.numel() != C:
            raise ValueError("BN parameters must be C fp32 values each")
    OH, OW = out_dim(H, FH, stride, pad), out_dim(W, FW, stride, pad)
    if out is None:
        out = torch.empty((N, max(OH, 0), max(OW, 0), C), device=x.device, dtype=torch.float32)
    else:
        _check_buffer(out, (N, max(OH, 0), max(OW, 0), C), torch.float32, x.device, "out")
    _call("dwc_fwd_bn_act", x.data_ptr(), mean.data_ptr(), var.data_ptr(), gamma.data_ptr(),
          beta.data_ptr(), float(eps), ACTS[act], w.data_ptr(), out.data_ptr(), N, H, W, C, FH,
          FW, stride, pad, _dtype_code(x), _stream_ptr(stream))
    return out


def bwd_data(dy, w, in_hw, stride: int = 1, pad: int = 0, out=None, stream=None, out_dtype=None):
    """dX = adjoint of ``fwd`` in X for a forward input of spatial size in_hw.  Output fp32, or
    out_dtype = the 16-bit input's own dtype."""
    torch = _torch()
    _check_cuda(dy, w)
    N, OH, OW, C = dy.shape
    FH, FW, _ = w.shape
    H, W = (int(v) for v in in_hw)
    if (out_dim(H, FH, stride, pad), out_dim(W, FW, stride, pad)) != (OH, OW):
        raise ValueError("dy spatial size does not match the forward output of in_hw")
    if w.dtype != dy.dtype:
        raise ValueError("filter must have dy's dtype")
    od = torch.float32 if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((N, H, W, C), device=dy.device, dtype=od)
    else:
        _check_buffer(out, (N, H, W, C), od, dy.device, "out")
    if od == torch.float32:
        _call("dwc_bwd_data", dy.data_ptr(), w.data_ptr(), out.data_ptr(), N, H, W, C, FH, FW,
              stride, pad, _dtype_code(dy), _stream_ptr(stream))
    else:
        _call("dwc_bwd_data_ex", dy.data_ptr(), w.data_ptr(), out.data_ptr(), N, H, W, C, FH, FW,
              stride, pad, _dtype_code(dy), _dtype_code(torch.empty(0, dtype=od)),
              _stream_ptr(stream))
    return out


def bwd_filter_workspace_size(x_shape, f_hw, stride: int = 1, pad: int = 0, dtype=None) -> int:
    torch = _torch()
    N, H, W, C = (int(v) for v in x_shape)
    FH, FW = (int(v) for v in f_hw)
    code = _dtype_code(torch.empty(0, dtype=dtype or torch.float32))
    return int(load_library().dwc_bwd_filter_workspace_size(N, H, W, C, FH, FW, stride, pad, code))


_ws_cache = {}


def workspace(nbytes: int, device):
    """A cached device buffer of at least nbytes (allocated by PyTorch, reused across calls
    on the same device and stream order)."""
    torch = _torch()
    key = str(device)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def bwd_filter(x, dy, f_hw, stride: int = 1, pad: int = 0, out=None, ws=None, stream=None):
    """dW[fh,fw,c] = sum_{n,oh,ow} X[n,oh*s+fh-p,ow*s+fw-p,c] * dY[n,oh,ow,c]  (fp32 output)."""
    torch = _torch()
    _check_cuda(x, dy)
    N, H, W, C = x.shape
    FH, FW = (int(v) for v in f_hw)
    OH, OW = out_dim(H, FH, stride, pad), out_dim(W, FW, stride, pad)
    _check_buffer(dy, (N, max(OH, 0), max(OW, 0), C), x.dtype, x.device, "dy")
    if out is None:
        out = torch.empty((FH, FW, C), device=x.device, dtype=torch.float32)
    else:
        _check_buffer(out, (FH, FW, C), torch.float32, x.device, "out")
    nbytes = load_library().dwc_bwd_filter_workspace_size(N, H, W, C, FH, FW, stride, pad,
                                                          _dtype_code(x))
    if ws is None:
        ws = workspace(nbytes, x.device)
    _call("dwc_bwd_filter", x.data_ptr(), dy.data_ptr(), out.data_ptr(), N, H, W, C, FH, FW,
          stride, pad, _dtype_code(x), ws.data_ptr(), ws.numel() * ws.element_size(),
          _stream_ptr(stream))
    return out


def device_status(stream=None) -> int:
    """Synchronise the stream and read/clear the kernels' status word (0 = DWC_OK)."""
    return int(load_library().dwc_device_status(_stream_ptr(stream)))


def set_wait_limit_ns(ns: int) -> int:
    """Limit of every wait inside kernels launched from now on (0: the 2 s default); returns
    the previous setting."""
    return int(load_library().dwc_set_wait_limit_ns(int(ns)))


def fma_rate_probe(kind: str, blocks: int, iters: int, out, stream=None) -> None:
    """Launch the CUDA-core multiply-add rate microbenchmark (``kind`` in FMA_KINDS) on the
    stream; ``out`` is a float32 device tensor of at least blocks * 256 elements."""
    _check_cuda(out)
    if out.numel() < blocks * 256:
        raise ValueError("out needs blocks * 256 floats")
    _call("dwc_fma_rate_probe", FMA_KINDS[kind], int(blocks), int(iters), out.data_ptr(),
          _stream_ptr(stream))


def path(pass_: str, a, b, out, N, H, W, C, FH, FW, stride, pad, dtype_code) -> int:
    """Kernel family of a call: 4 warp-level MMA and 2 tcgen05 tensor-core kernels (16-bit
    inputs), 3 small-map kernels (maps up to 16x16), 1 fast CUDA-core kernels, 0 general
    kernels, -1 invalid."""
    p = {"fwd": 0, "bwd_data": 1, "bwd_filter": 2, "fwd_bn_act": 3}[pass_]
    return int(load_library().dwc_path(p, a, b, out, N, H, W, C, FH, FW, stride, pad,
                                       dtype_code))


def kernel_launches(pass_: str, N, H, W, C, FH, FW, stride, pad, dtype_code) -> int:
    """Kernel launches of this library that a call makes (aligned tensors), -1 invalid."""
    p = {"fwd": 0, "bwd_data": 1, "bwd_filter": 2, "fwd_bn_act": 3}[pass_]
    return int(load_library().dwc_kernel_launches(p, N, H, W, C, FH, FW, stride, pad, dtype_code))


__all__ = ["build", "load_library", "fwd", "fwd_bn_act", "bwd_data", "bwd_filter",
           "bwd_filter_workspace_size", "device_status", "set_wait_limit_ns", "fma_rate_probe",
           "path", "kernel_launches", "status_string", "DwcError", "EXPORTS", "FMA_KINDS",
           "LIB_PATH"]
