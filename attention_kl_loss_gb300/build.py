"""Build the in-tree shared library ``_lib/libstreamkl.so`` with nvcc.

Every translation unit is compiled for sm_103a only (GB300), in parallel, then
linked with the static CUDA runtime. Nothing is installed outside the tree.

``build(debug=True)`` builds ``_lib/libstreamkl_debug.so`` from the same
sources with STREAMKL_DEVICE_CHECKS defined: the kernels then check the
operands of every TMA copy, TMEM access and mbarrier against their layout
and report a failed check as STREAMKL_ERR_DEVICE_CHECK in the caller's
status word instead of issuing the access.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB_NAME = "libstreamkl.so"
DEBUG_LIB_NAME = "libstreamkl_debug.so"
SOURCES = ["api.cu", "fwd.cu", "bwd.cu", "bwd_sep.cu", "bwd_short.cu", "bwd_fused.cu", "bwd_fused128.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", f"-I{os.path.join(ROOT, 'include')}"]


def nvcc() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin on PATH)")


def lib_path(debug: bool = False) -> str:
    return os.path.join(OUT_DIR, DEBUG_LIB_NAME if debug else LIB_NAME)


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False,
          debug: bool = False) -> str:
    """Compile (if stale) and return the library path (the debug build with
    device-side range checks when ``debug``)."""
    os.makedirs(OUT_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "streamkl.h"))
    objs = []
    jobs = []
    tag = "_debug" if debug else ""
    extra = ["-DSTREAMKL_DEVICE_CHECKS"] if debug else []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, src.replace(".cu", f"{tag}.o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", s, "-o", o]
            if ptxas_info:
                cmd += ["-Xptxas", "-v"]
            jobs.append(cmd)

    def run(cmd):
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p

    with cf.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        for cmd, p in ex.map(run, jobs):
            if verbose or ptxas_info or p.returncode != 0:
                sys.stderr.write(p.stdout + p.stderr)
            if p.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    lib = lib_path(debug)
    if force or _stale(lib, objs):
        cmd = [nvcc(), *ARCH, "-shared", "-o", lib, *objs]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            sys.stderr.write(p.stdout + p.stderr)
            raise RuntimeError(f"link failed: {' '.join(cmd)}")
    return lib


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv, force="-f" in sys.argv,
                debug="--debug" in sys.argv))
