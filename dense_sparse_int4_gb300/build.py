"""Build the sm_103a shared libraries in-tree with nvcc.

Each CUDA translation unit compiles in parallel; the objects link into
``dense_sparse_int4_gb300/_build/libmq.so`` with the CUDA runtime linked
statically, so the library loads without a GPU driver (CPU-only hosts can
still inspect its exported symbols).  The rate microbenchmarks that the
roofline peaks come from (``csrc/peaks.cu``) build into their own
``_build/libmq_peaks.so``, apart from the product library.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmq.so")
PEAKS_LIB = os.path.join(BUILD, "libmq_peaks.so")
PEAKS_SOURCE = "peaks.cu"
SOURCES = ["abi.cu", "status.cu", "quantize.cu", "select.cu", "pack.cu", "gemm.cu", "image_gemm.cu", "zipper.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(verbose_ptxas: bool):
    f = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "-I", os.path.join(ROOT, "include")]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src, os.path.join(CSRC, "mq_internal.cuh"), os.path.join(ROOT, "include", "mq.h"), __file__]
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    todo = []
    objs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, s.replace(".cu", ".o"))
        objs.append(obj)
        if force or verbose_ptxas or _stale(obj, src):
            todo.append([cc, *_flags(verbose_ptxas), "-c", src, "-o", obj])

    peaks_src = os.path.join(CSRC, PEAKS_SOURCE)
    if force or _stale(PEAKS_LIB, peaks_src):
        tmp_peaks = PEAKS_LIB + f".tmp{os.getpid()}"
        todo.append([cc, *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-o", tmp_peaks, peaks_src,
                     "-cudart", "static"])
    else:
        tmp_peaks = None

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, todo):
                if verbose_ptxas or r.returncode != 0:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if tmp_peaks:
        os.replace(tmp_peaks, PEAKS_LIB)
        todo = [c for c in todo if tmp_peaks not in c]
    if todo or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
