"""Build libdrs.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

The translation units compile in parallel with nvcc and link into
``vocab_row_sampling_gb300/_build/libdrs.so`` (CUDA runtime linked
statically). Nothing is installed into site-packages.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
REPO_DIR = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(REPO_DIR, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libdrs.so")

SOURCES = ["capi.cu", "row_stats.cu", "row_split.cu", "row_cluster.cu", "topk.cu", "stash.cu", "philox_gumbel.cu", "scale.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# No fast-math: IEEE division, denormals kept (the probabilities can be
# fp32 subnormals that are still representable in bf16).
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "--ftz=false", "--prec-div=true", "--prec-sqrt=true",
              "--fmad=true", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdrs")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "drs.h"))
    return files, headers


def _stale(files, headers) -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in files + headers + [__file__])


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile libdrs.so if it is missing or older than its sources."""
    files, headers = _inputs()
    if not force and not _stale(files, headers):
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src).replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *flags, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {src}")
        return obj

    with ThreadPoolExecutor(max_workers=len(files)) as ex:
        objs = list(ex.map(compile_one, files))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("nvcc link of libdrs.so failed")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
