"""Builds ``libzeroshard.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel), then one
nvcc link produces the shared library next to this file.  No cmake, no torch
extension machinery: the library is a plain C-ABI shared object.
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
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libzeroshard.so")
# the debug build: the same sources with the kernels' index checks compiled in
CHECKED_BUILD_DIR = os.path.join(PKG, "_build_checked")
CHECKED_LIB_PATH = os.path.join(PKG, "libzeroshard_checked.so")

SOURCES = ["shard_step.cu", "clip.cu", "sgd.cu", "adam8.cu", "layout.cu", "cpu_step.cpp", "diag.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -ffp-contract=off keeps host arithmetic (step coefficients, the CPU step) free
# of fused multiply-adds, matching the device code's explicit _rn operations;
# -fno-math-errno lets the host compiler vectorise sqrtf (results unchanged).
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-O3,-fPIC,-fvisibility=hidden,-ffp-contract=off,-fno-math-errno",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib_path: str) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "zero_shard.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compile every source and link ``libzeroshard.so`` (``checked``: the
    debug build ``libzeroshard_checked.so``, with the kernels' index checks);
    returns its path."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    build_dir = CHECKED_BUILD_DIR if checked else BUILD_DIR
    if checked:
        extra_flags = (*extra_flags, "-DZS_CHECKED=1")
    if not force and not _stale(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    exe = nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [exe, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, "-shared", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


def build_all(force: bool = False) -> tuple:
    """Both libraries, compiled side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        a = ex.submit(build, force)
        b = ex.submit(build, force, False, (), True)
        return a.result(), b.result()


def host_vectorization_report() -> str:
    """The host compiler's report on the loops of the host-core step
    (csrc/cpu_step.cpp) it vectorized, compiled with the library's own flags
    plus -fopt-info-vec-optimized; one line per vectorized loop."""
    import tempfile
    with tempfile.TemporaryDirectory() as d:
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-Xcompiler", "-fopt-info-vec-optimized", "-c",
               os.path.join(CSRC, "cpu_step.cpp"), "-o", os.path.join(d, "cpu_step.o")]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed:\n{r.stdout}\n{r.stderr}")
    lines = [ln for ln in (r.stdout + r.stderr).splitlines() if "cpu_step.cpp" in ln and "vectorized" in ln]
    return "\n".join(sorted(set(lines), key=lambda ln: int(ln.split(":")[1]) if ln.split(":")[1].isdigit() else 0))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv))
