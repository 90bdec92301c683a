"""Build libhybrid.so (the CUDA library behind include/hybrid.h) in-tree for sm_103a.

Each translation unit compiles in parallel with nvcc; objects go to _build/
next to this file and the shared library to libhybrid.so in this package.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
SO = os.path.join(HERE, "libhybrid.so")
SOURCES = ["gemv.cu", "bgemv.cu", "gdn.cu", "attn.cu", "attn_pair.cu", "gemm.cu", "prefill.cu", "moe_prefill.cu", "engine.cu", "noalloc.cu"]
HEADERS = ["common.cuh", "kernels.h", "gemv_dev.cuh", "attn_dev.cuh", "attn_kernel.cuh", "gdn_dev.cuh", "tc05.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "--extended-lambda"]


def _extra_flags() -> list[str]:
    """Additional nvcc flags from HY_NVCC_EXTRA (e.g. tuning macros); a change
    of them rebuilds every object."""
    return os.environ.get("HY_NVCC_EXTRA", "").split()


def _deps() -> list[str]:
    return [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "hybrid.h")]


def _stale(out: str, srcs: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in srcs)


def _compile(src: str) -> str:
    obj = os.path.join(OUT, os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    if _stale(obj, [path] + _deps()):
        cmd = ["nvcc", *ARCH, *FLAGS, *_extra_flags(), "-I", os.path.join(ROOT, "include"), "-c", path, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    stamp = os.path.join(OUT, "flags.txt")
    flags = " ".join(_extra_flags())
    if not os.path.exists(stamp) or open(stamp).read() != flags:
        force = True
        with open(stamp, "w") as f:
            f.write(flags)
    if force:
        for s in SOURCES:
            o = os.path.join(OUT, os.path.splitext(s)[0] + ".o")
            if os.path.exists(o):
                os.remove(o)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    if _stale(SO, objs):
        subprocess.check_call(["nvcc", *ARCH, "-shared", "-o", SO, *objs, "-lcudart"])
    return SO


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
