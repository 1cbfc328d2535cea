"""Build the sm_103a CUDA library in-tree:
speculative_decoding_verification_61_gb300/_build/libspecverify.so

Five translation units (chain verify, tree verify, vocab-sharded verify, the adaptive-k
controller, the allocation-free verify), one
-gencode (sm_103a), static CUDA runtime, so the shared object loads with
plain ctypes and needs no GPU at load time.
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
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libspecverify.so")
SOURCES = [os.path.join(CSRC, n)
           for n in ("spec_verify.cu", "tree_verify.cu", "shard_verify.cu", "adapt_k.cu", "noalloc.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, n) for n in ("device_utils.cuh", "verify_common.cuh", "host_common.h")] + [
    os.path.join(INCLUDE, "spec_verify.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA library cannot be built")


def build_cmd(out: str = LIB, extra=()) -> list[str]:
    return [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
            "-Xptxas", "-warn-spills", f"-I{INCLUDE}", f"-I{CSRC}", *extra, "-o", out, *SOURCES]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB + ".tmp"
    cmd = build_cmd(tmp, ["-Xptxas", "-v"] if verbose else [])
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
