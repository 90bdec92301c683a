"""Build the generator's host (C) and device (CUDA, sm_103a) shared libraries in-tree."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SO = os.path.join(HERE, "libsynth_host.so")
DEV_SO = os.path.join(HERE, "libsynth_dev.so")


def _stale(out: str, srcs: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in srcs)


def build_host(force: bool = False) -> str:
    src = os.path.join(HERE, "csrc", "synth_host.c")
    if force or _stale(HOST_SO, [src]):
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", HOST_SO, src])
    return HOST_SO


def build_device(force: bool = False) -> str:
    src = os.path.join(HERE, "csrc", "synth_gen.cu")
    if force or _stale(DEV_SO, [src]):
        subprocess.check_call([
            "nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo",
            "-Xcompiler", "-fPIC", "-shared", "-o", DEV_SO, src,
        ])
    return DEV_SO


if __name__ == "__main__":
    build_host(force="--force" in sys.argv)
    build_device(force="--force" in sys.argv)
