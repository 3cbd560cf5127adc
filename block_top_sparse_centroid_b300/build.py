"""Build libkin.so (the C-ABI CUDA library) in-tree for sm_103a with nvcc.

Usage:  python -m block_top_sparse_centroid_b300.build [--force] [--verbose] [--variant NAME]

Variants are test builds of the same sources with other compile-time limits, written next
to the library as libkin_<name>.so: "shortwait" gives every bounded wait of the kernels
4096 tries instead of about four million, so that a test can make a wait run out quickly.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libkin.so")
VARIANTS = {"shortwait": ["-DKIN_MAX_WAIT_TRIES=4096u"]}

SOURCES = ["centroid.cu", "score_select.cu", "attention.cu", "decode_fused.cu", "token_topk.cu",
           "kin_api.cu", "noalloc.cu"]
HEADERS = ["kin_common.cuh", "attn_common.cuh", "kin_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkin")


def lib_path(variant: str = "") -> str:
    return LIB if not variant else os.path.join(PKG, f"libkin_{variant}.so")


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "kin.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, variant: str = "") -> str:
    """Compile every source into libkin.so (or a test variant) next to this file; returns
    its path."""
    lib = lib_path(variant)
    if not force and not _stale(lib):
        return lib
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "--shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
           *VARIANTS.get(variant, []), "-o", lib + ".tmp"]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    cmd += [os.path.join(CSRC, f) for f in SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed building {os.path.basename(lib)}")
    os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    var = sys.argv[sys.argv.index("--variant") + 1] if "--variant" in sys.argv else ""
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv, variant=var))
