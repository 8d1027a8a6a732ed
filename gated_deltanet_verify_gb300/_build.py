"""Build the in-tree CUDA library ``libgdn_verify.so`` for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library (CUDA runtime linked statically, so the library only needs the
driver; no other CUDA library is linked).  Rebuilds only what changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdn_verify.so")
# the checked variant: every global access of the verify-family and rollback kernels bounds-checked
CHECKED_BUILD = os.path.join(PKG, "_build_checked")
CHECKED_LIB = os.path.join(PKG, "libgdn_verify_checked.so")

SOURCES = ["gdn_api.cu", "verify.cu", "rollback.cu", "prefill.cu", "proj.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn_verify.so")


def _headers() -> List[str]:
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs


def _stale(target: str, deps: List[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _machine_marker(build_dir: str, lib: str) -> str:
    """Objects from another host architecture (e.g. an x86 build copied to an
    aarch64 machine) are discarded rather than linked."""
    m = os.path.join(build_dir, "MACHINE")
    here = platform.machine()
    prev = open(m).read().strip() if os.path.exists(m) else None
    if prev != here:
        for f in os.listdir(build_dir):
            if f.endswith(".o"):
                os.remove(os.path.join(build_dir, f))
        if os.path.exists(lib):
            os.remove(lib)
        with open(m, "w") as fh:
            fh.write(here + "\n")
    return here


def build(verbose: bool = False, extra_flags: List[str] = (), checked: bool = False) -> str:
    """Build libgdn_verify.so, or with ``checked`` the bounds-checked variant
    libgdn_verify_checked.so (-DGDN_CHECKED=1, its own object directory)."""
    BUILD = CHECKED_BUILD if checked else globals()["BUILD"]
    LIB = CHECKED_LIB if checked else globals()["LIB"]
    if checked:
        extra_flags = [*extra_flags, "-DGDN_CHECKED=1"]
    os.makedirs(BUILD, exist_ok=True)
    _machine_marker(BUILD, LIB)
    cc = nvcc()
    hdrs = _headers()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if _stale(o, [s] + hdrs):
            jobs.append([cc, *ARCH, *FLAGS, *extra_flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            print(" ".join(cmd))
            print(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {cmd[-3]}")
        return r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        list(ex.map(run, jobs))
    if jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        run([cc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv))
