"""Build the CUDA library in-tree: attention_online_softmax_gb300/_lib/libattn_gb300.so.

One translation unit, compiled for sm_103a only:
    nvcc -gencode arch=compute_103a,code=sm_103a -lineinfo -O3 -shared ...
Run ``python -m attention_online_softmax_gb300.build`` (add ``-v`` for the
ptxas register / shared-memory report).
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
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libattn_gb300.so")
SOURCES = [os.path.join(CSRC, "attn_api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "prefill_fwd.cuh", "decode.cuh", "bwd.cuh", "bwd_wide.cuh", "bwd_api.cuh", "probe.cuh")] + [
    os.path.join(INCLUDE, "attn.h")]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in DEPS if os.path.exists(p))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not needs_build():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = f"{LIB}.{os.getpid()}.tmp"
    cmd = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
           "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
           f"-I{INCLUDE}", f"-I{CSRC}", "-o", tmp] + SOURCES
    if verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("nvcc failed to build libattn_gb300.so")
    if verbose:
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose="-v" in sys.argv)
    print(LIB)
