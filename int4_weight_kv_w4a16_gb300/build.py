"""Build libfutr.so from csrc/*.cu for sm_103a (nvcc, no cmake).

Each translation unit is compiled in parallel into ``_build/`` and linked into
``libfutr.so`` next to this file.  The build is skipped when the library is
newer than every source and header.

``build(debug=True)`` (or ``python -m int4_weight_kv_w4a16_gb300.build
--debug``) makes the debug variant ``libfutr_debug.so`` from the same sources
with ``-DFUTR_DEBUG``: device bounds checks before the global accesses of the
split records, the projection outputs, the weight-unit and KV-tile copies (a
failed check reports FUTR_ERR_BOUNDS and skips the access).  ``futr.lib()``
loads it when the environment has FUTR_DEBUG=1.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libfutr.so")
LIB_DEBUG = os.path.join(PKG, "libfutr_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfutr.so")
    return path


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _inputs():
    hdr = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdr += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sources() + hdr + [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _compile(src: str, extra, out_dir: str = BUILD) -> str:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Compile and link libfutr.so (debug: libfutr_debug.so); returns its path."""
    lib = LIB_DEBUG if debug else LIB
    if not force and up_to_date(lib):
        return lib
    out_dir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(out_dir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    if debug:
        extra += ["-DFUTR_DEBUG"]
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, out_dir), sources()))
    tmp = lib + ".tmp"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
