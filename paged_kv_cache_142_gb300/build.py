"""Build libpa_gb300.so in-tree with nvcc for sm_103a.

Every translation unit under ``csrc/`` is compiled in parallel to
``_build/*.o``; the objects are linked into ``libpa_gb300.so`` next to this
file (CUDA runtime linked statically, so the library loads on a host with no
GPU).  A rebuild happens when the library is missing, older than any source
or header, or was built for another machine architecture.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB_NAME = "libpa_gb300.so"
LIB = os.path.join(PKG, LIB_NAME)
STAMP = os.path.join(BUILD, "stamp.txt")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpa_gb300.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _inputs():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                               + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stamp_text() -> str:
    return f"{platform.machine()} {' '.join(NVCC_FLAGS)}"


def is_stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return True
    with open(STAMP) as f:
        if f.read().strip() != _stamp_text():
            return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _inputs())


def _compile(src: str, verbose_ptxas: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [_nvcc()] + NVCC_FLAGS + ["-c", src, "-o", obj]
    if verbose_ptxas and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, quiet: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile the library if needed; return its path."""
    if not force and not is_stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    logs = []
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        futs = [ex.submit(_compile, s, verbose_ptxas) for s in srcs]
        objs = []
        for f in futs:
            obj, log = f.result()
            objs.append(obj)
            if log.strip():
                logs.append(log)
    tmp = LIB + ".tmp"
    cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(_stamp_text())
    if not quiet:
        for log in logs:
            sys.stderr.write(log)
        sys.stderr.write(f"built {LIB}\n")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
