"""Build libq4k.so in-tree for GB300 (sm_103a) with nvcc.

Each ``csrc/*.cu`` file is compiled on its own (in parallel) with
``-gencode arch=compute_103a,code=sm_103a``; the objects are linked into
``q4_weight_matmul_gb300/libq4k.so`` (CUDA runtime linked statically).
A build is skipped when the library is newer than every source file.

    python -m q4_weight_matmul_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libq4k.so")
PEAKS_SRC = os.path.join(CSRC, "peaks", "peaks.cu")
PEAKS_LIB = os.path.join(PKG, "libq4k_peaks.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
          "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libq4k.so")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale() -> bool:
    if not os.path.exists(LIB_PATH) or not os.path.exists(PEAKS_LIB):
        return True
    t = min(os.path.getmtime(LIB_PATH), os.path.getmtime(PEAKS_LIB))
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) \
        + glob.glob(os.path.join(INCLUDE, "*.h")) + [PEAKS_SRC, os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
    if src == PEAKS_SRC:
        obj = os.path.join(BUILD_DIR, "peaks_probe.o")
    cmd = [nvcc(), *ARCH, *CFLAGS, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA source and link libq4k.so (and the benchmark's
    tensor-rate probe, libq4k_peaks.so); return the library's path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = sources() + [PEAKS_SRC]
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), srcs))
    for path, members in ((LIB_PATH, objs[:-1]), (PEAKS_LIB, objs[-1:])):
        tmp = path + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *members]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(path)} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
