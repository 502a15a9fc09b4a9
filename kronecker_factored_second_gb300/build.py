"""In-tree build of libokls.so (sm_103a) with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library next to this file.  Used by ``__graft_entry__.build()`` and by the
Python binding when the library is missing and a build is requested.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libokls.so")
SOURCES = ["okls_api.cu", "okls_gemm.cu", "okls_elementwise.cu", "okls_ns_small.cu",
           "okls_soap.cu", "okls_clean.cu", "okls_clean_large.cu",
           "okls_soap_large.cu", "okls_eig.cu", "okls_bjacobi.cu", "okls_tc3.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(debug: bool = False) -> list[str]:
    f = ARCH + ["-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
                "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    f += ["-O0", "-G"] if debug else ["-O3"]
    return f


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout)
        raise RuntimeError("command failed: " + " ".join(cmd))
    if r.stdout.strip():
        sys.stderr.write(r.stdout)


def build_library(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every source for sm_103a and link libokls.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def one(src: str) -> str:
        obj = os.path.join(BUILD, src + ".o")
        cmd = [cc, "-c", os.path.join(CSRC, src), "-o", obj] + _flags() + extra
        if verbose:
            print(" ".join(cmd))
        _run(cmd)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(one, SOURCES))
    tmp = LIB + ".tmp"
    _run([cc, "-shared", "-o", tmp] + objs + ARCH + ["--cudart", "static", "-Xcompiler", "-fPIC"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(verbose=True, ptxas_info="-v" in sys.argv))
