"""Builds libcas.so in-tree with nvcc for sm_103a (GB300).

Each .cu file is compiled in parallel to an object in ``_build/`` and linked
into ``bit_level_weight_gb300/libcas.so``. A rebuild happens only when a
source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libcas.so")
# The CAS_DEBUG variant: device code also records inconsistent encoded data
# (superblock indices that decrease or run past their section) in a flag read
# by cas_device_status. Same C ABI; built on request only.
OUT_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libcas_debug.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "cas.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _compile(src: str, extra: list[str], out: str = OUT) -> str:
    obj = os.path.join(out, os.path.basename(src) + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, extra: list[str] | None = None, verbose: bool = False, debug: bool = False) -> str:
    """Compile every kernel for sm_103a and link libcas.so (debug: the
    CAS_DEBUG variant libcas_debug.so); returns its path."""
    lib, out = (LIB_DEBUG, OUT_DEBUG) if debug else (LIB, OUT)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out, exist_ok=True)
    extra = list(extra or []) + (["-DCAS_DEBUG"] if debug else [])
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, out), srcs))
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(f"built {lib}")
    return lib


if __name__ == "__main__":
    import sys
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None)
