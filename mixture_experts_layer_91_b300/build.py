"""Compile the CUDA library in-tree for sm_103a.

    python -m mixture_experts_layer_91_b300.build [--ptxas-log PATH]

Produces mixture_experts_layer_91_b300/lib/libmoe_b300.so from csrc/moe_b300.cu
(one translation unit). nvcc cross-compiles; no GPU is needed.
"""

from __future__ import annotations

import argparse
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIB_DIR, "libmoe_b300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh")))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    hdr = os.path.join(os.path.dirname(PKG), "include", "moe_b300.h")
    return all(os.path.getmtime(s) <= t for s in sources() + [hdr, __file__])


def build(force: bool = False, ptxas_log: str | None = None) -> str:
    if not force and up_to_date() and ptxas_log is None:
        return LIB
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-Xptxas", "-v", "-o", tmp, os.path.join(CSRC, "moe_b300.cu")]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stderr[-4000:]}")
    if ptxas_log:
        with open(ptxas_log, "w") as f:
            f.write(" ".join(cmd) + "\n" + res.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-log")
    a = ap.parse_args()
    print(build(force=True, ptxas_log=a.ptxas_log))
