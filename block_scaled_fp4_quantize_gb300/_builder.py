"""Build the CUDA library ``libfp4q.so`` in-tree for sm_103a (GB300).

Each translation unit is compiled in parallel with nvcc, then linked into a
shared object with the CUDA runtime linked statically, so the library needs
nothing but the driver at run time.  ``fast_math=True`` builds a second copy
with ``-use_fast_math`` (the numerics are written to give identical bits).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
SOURCES = ["fp4q_api.cu", "k_tile.cu", "k_ct.cu", "k_ctb.cu", "k_ctb_grouped.cu", "k_ctb_rht.cu", "k_ctl.cu", "k_row.cu", "k_aux.cu", "k_mxfp4.cu", "k_mxfp8.cu", "fp4q_host.cu", "fp4q_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfp4q")


def lib_path(fast_math: bool = False) -> str:
    return os.path.join(BUILD, "libfp4q_fastmath.so" if fast_math else "libfp4q.so")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(fast_math: bool = False, force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    out = lib_path(fast_math)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "fp4q.h"))
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    if not force and not _stale(out, srcs + headers + [os.path.abspath(__file__)]):
        return out
    tag = "fm" if fast_math else "std"
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if fast_math:
        flags.append("-use_fast_math")
    if verbose:
        flags += ["-Xptxas", "-v"]
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".%s.o" % tag))
        r = subprocess.run([cc] + flags + ["-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            print(log)
    tmp = out + ".tmp%d" % os.getpid()
    r = subprocess.run([cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys

    print(build(fast_math="--fast-math" in sys.argv, force="--force" in sys.argv, verbose="-v" in sys.argv))
