"""Build libst24.so (the CUDA library behind include/st24.h) for sm_103a.

Each translation unit under csrc/ is compiled by its own nvcc process (in
parallel), then linked into one shared library with the CUDA runtime linked
statically, so loading the library needs no CUDA driver until a call is made.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libst24.so")
# The failure-detection self-test (linked into the library, declared in st24_selftest.h).
SELFTEST_SRC = os.path.join(CSRC, "selftest", "st24_selftest.cu")
# The tensor-pipe ceiling probe bench.py's roofline uses (not part of the C ABI).
PEAK_SRC = os.path.join(CSRC, "peak", "peak_mma_sp.cu")
PEAK_LIB = os.path.join(OUT, "libst24_peak.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu"))) + [SELFTEST_SRC]
    deps = srcs + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)]
    return srcs, deps


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    srcs, deps = _inputs()
    peak_deps = [PEAK_SRC, os.path.abspath(__file__)]
    if not force and not _stale(LIB, deps) and not _stale(PEAK_LIB, peak_deps):
        return LIB
    os.makedirs(OUT, exist_ok=True)
    nvcc = _nvcc()
    flags = FLAGS + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(OUT, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(len(srcs) + 1, os.cpu_count() or 4)) as ex:
        peak_obj = ex.submit(compile_one, PEAK_SRC)
        objs = list(ex.map(compile_one, srcs))
        peak_obj = peak_obj.result()
    for lib, parts in ((LIB, objs), (PEAK_LIB, [peak_obj])):
        tmp = lib + ".tmp.%d" % os.getpid()
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *parts]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
