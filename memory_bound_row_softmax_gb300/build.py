"""Build the C-ABI library ``_build/libmbrs_softmax.so`` for sm_103a.

Each translation unit of ``csrc/`` is compiled by nvcc in parallel, then the
objects are linked into one shared library with the CUDA runtime linked
dynamically (the process shares one runtime with PyTorch: same current
device, same streams).  Run ``python -m memory_bound_row_softmax_gb300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmbrs_softmax.so")
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["abi.cu", "k_warp.cu", "k_warp_whole.cu", "k_cta.cu", "k_cta_whole.cu", "k_cluster.cu", "k_grid.cu", "k_pattern_copy.cu",
           "k_noalloc.cu", "k_masked_warp.cu", "k_masked_warp_whole.cu", "k_masked.cu", "k_masked_whole.cu",
           "k_packed.cu", "k_attention.cu", "attention_abi.cu"]
HEADERS = ["common.cuh", "kernels.cuh", "launch.h", "warp_launch.cuh", "cta_launch.cuh", "attention.cuh",
           "attention_launch.h"]
PUBLIC_HEADERS = ["mbrs_softmax.h", "mbrs_attention.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.exists(os.path.join(home, "bin", "nvcc")):
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


# The files only the attention forward compiles from; the softmax kernels
# and their ABI do not depend on them.
ATTENTION_ONLY = ["k_attention.cu", "attention_abi.cu", "attention.cuh", "attention_launch.h", "mbrs_attention.h"]


def sources_digest() -> str:
    """sha256 over the row-softmax kernel sources and the ABI they are called
    through (identifies the build that profiles/traffic.json was captured
    from; the attention-only files are left out, so that a change there does
    not retire the softmax kernels' traffic records)."""
    import hashlib
    h = hashlib.sha256()
    for f in sorted(SOURCES + HEADERS):
        if f in ATTENTION_ONLY:
            continue
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    for f in PUBLIC_HEADERS:
        if f in ATTENTION_ONLY:
            continue
        with open(os.path.join(INCLUDE, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files += [os.path.join(INCLUDE, f) for f in PUBLIC_HEADERS]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link; returns the library path.  Skips work when up to date."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    home = cuda_home()
    nvcc = os.path.join(home, "bin", "nvcc")
    os.makedirs(BUILD, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr}")
        if verbose and res.stderr:
            sys.stderr.write(res.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    lib64 = os.path.join(home, "lib64")
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs, "-Xlinker", f"-rpath,{lib64}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
