"""Build libexattn.so in-tree with nvcc for sm_103a (no torch extension machinery)."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libexattn.so")
SOURCES = [os.path.join(CSRC, "fa_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("fa_fwd_kernel.cuh", "fa_quant.cuh", "fa_bwd_kernel.cuh", "sm103_ptx.cuh")] + [
    os.path.join(ROOT, "include", "exact_attention.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-shared"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libexattn.so")


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library (skipped when it is newer than every source) and return its path."""
    if not force and up_to_date():
        return LIB_PATH
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc(), *NVCC_FLAGS, "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
