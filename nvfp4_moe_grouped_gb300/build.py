"""Builds the CUDA library (libnvfp4_moe.so) in-tree for sm_103a.

Each translation unit is compiled in parallel with nvcc, then linked into one
shared object with the CUDA runtime linked statically, so the library's only
dependency at load time is the driver.  Used by ``__graft_entry__.build()`` and,
when the library is missing or stale, by the Python binding.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libnvfp4_moe.so")
# cuBLASLt's block-scaled FP4 GEMM as a timing reference for the dense GEMM (benchmark only)
REF_SRC = os.path.join(HERE, "reference_gemm", "cublaslt_fp4.cu")
REF_LIB = os.path.join(BUILD, "libnvfp4_cublaslt.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in _deps())


def _compile(src: str, verbose_ptxas: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas:
        print(res.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    if not force and not is_stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas), srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    build_reference()
    return LIB


def build_reference() -> str | None:
    """The cuBLASLt timing reference, a separate library (it links cuBLASLt dynamically; the layer's library
    depends on the driver only).  A failure here is reported, not raised: nothing but the benchmark's dense-GEMM
    comparison uses it."""
    os.makedirs(BUILD, exist_ok=True)
    tmp = REF_LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-shared", REF_SRC, "-o", tmp, "-lcublasLt"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        print(f"note: the cuBLASLt reference library did not build:\n{res.stderr[-2000:]}")
        return None
    os.replace(tmp, REF_LIB)
    return REF_LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose_ptxas="-v" in sys.argv))
