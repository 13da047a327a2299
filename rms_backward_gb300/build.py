"""Builds the C-ABI shared library ``libmhcpb.so`` in-tree with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked
with the static CUDA runtime (no dependency on a libcudart found at run time).
Output: ``rms_backward_gb300/_build/libmhcpb.so``.  Incremental: a unit is
rebuilt only when it, or a header it may include, is newer than its object.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmhcpb.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              f"-I{INCLUDE}", f"-I{CSRC}"] + ARCH


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmhcpb.so")


def _newest_header() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def build(verbose: bool = False, extra_flags=None, out_dir=None) -> str:
    """Compile and link; returns the library path.  ``extra_flags`` (extra nvcc
    defines for instrumented copies) require ``out_dir`` so that the product
    library in ``_build/`` is never replaced by an instrumented one."""
    if extra_flags and not out_dir:
        raise ValueError("extra_flags need a separate out_dir")
    nvcc = _nvcc()
    bdir = out_dir or BUILD
    lib = os.path.join(bdir, "libmhcpb.so")
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_t = _newest_header()
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_t) \
                and not extra_flags:
            return obj, None
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            return obj, f"$ {' '.join(cmd)}\n{res.stdout}\n{res.stderr}"
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr, file=sys.stderr)
        return obj, None

    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    errs = [e for _, e in results if e]
    if errs:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errs))
    objs = [o for o, _ in results]
    if not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        tmp = lib + ".tmp"
        cmd = [nvcc, "-shared", "--cudart", "static", *ARCH, "-o", tmp, *objs,
               "-ldl", "-lrt", "-lpthread"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n$ {' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))
