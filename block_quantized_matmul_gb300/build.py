"""Build libqmm.so in-tree: every csrc/*.cu compiled for sm_103a in parallel, then linked.

Usage: python -m block_quantized_matmul_gb300.build [--debug]   (or build() from Python).
The library lands next to this file; object files go to csrc/_build/ (git-ignored).
--debug (or QMM_DEBUG=1 in the environment) builds libqmm_debug.so instead, with -DQMM_DEBUG: every
kernel checks its tile, block and ring-slot indices, skips an access that fails and records it for
qmm_device_status (QMM_ERR_BOUNDS).  The release library is not touched.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ_DIR = os.path.join(CSRC, "_build")
LIB = os.path.join(HERE, "libqmm.so")
LIB_DEBUG = os.path.join(HERE, "libqmm_debug.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(HERE, "..", "include", "qmm.h")]


def _debug_default() -> bool:
    return os.environ.get("QMM_DEBUG") == "1"


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(OBJ_DIR + ("_debug" if debug else ""), os.path.basename(src)[:-3] + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, *(["-DQMM_DEBUG"] if debug else []), "-c", src, "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        sys.stderr.write(res.stdout + res.stderr)
    return obj


def up_to_date(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps() if os.path.exists(p))


def build(force: bool = False, verbose: bool = False, debug: bool | None = None) -> str:
    """Compile and link libqmm.so (or, with debug, libqmm_debug.so) for sm_103a; returns its path."""
    debug = _debug_default() if debug is None else debug
    lib = LIB_DEBUG if debug else LIB
    if not force and up_to_date(debug):
        return lib
    os.makedirs(OBJ_DIR + ("_debug" if debug else ""), exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fPIC", "-lcudart",
           "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug=True if "--debug" in sys.argv else None))
