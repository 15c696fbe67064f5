"""Build the CUDA library ``libdwc_gb300.so`` in-tree with nvcc, for sm_103a only.

Every ``csrc/*.cu`` file is compiled to an object in parallel, then linked into a shared
library next to this file.  Rebuilds only what changed (sources or headers newer than the
object).  No CPU fallback exists: importing the binding without this library fails loudly.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libdwc_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdwc_gb300.so")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(obj: str, src: str, hdr_mtime: float) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return t < os.path.getmtime(src) or t < hdr_mtime


def build(verbose: bool = False, jobs: int | None = None, extra_flags=None) -> str:
    """Compile and link the library; returns its path."""
    nvcc = nvcc_path()
    os.makedirs(OBJ_DIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_mtime = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    objs = [os.path.join(OBJ_DIR, os.path.basename(s)[:-3] + ".o") for s in srcs]
    flags = NVCC_FLAGS + list(extra_flags or [])
    if verbose:
        flags = flags + ["-Xptxas", "-v"]

    todo = [(s, o) for s, o in zip(srcs, objs) if _stale(o, s, hdr_mtime)]

    def compile_one(so):
        s, o = so
        cmd = [nvcc] + ARCH + flags + ["-c", s, "-o", o + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(s)}:\n{r.stderr[-6000:]}")
        os.replace(o + ".tmp", o)
        return s, r.stderr

    jobs = jobs or min(len(todo), os.cpu_count() or 4) or 1
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        for s, log in ex.map(compile_one, todo):
            if verbose and log:
                sys.stderr.write(f"== {os.path.basename(s)}\n{log}")

    if todo or not os.path.exists(LIB_PATH):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-6000:]}")
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
