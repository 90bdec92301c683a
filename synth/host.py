"""ctypes binding of the host (C) generator copy; same outputs as synth.gen."""
from __future__ import annotations

import ctypes

import numpy as np

from . import build, gen

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build.build_host())
        u64, f32, u32 = ctypes.c_uint64, ctypes.c_float, ctypes.c_uint32
        vp = ctypes.c_void_p
        _lib.synh_fill_normal_bf16.argtypes = [vp, u64, u64, u64, f32, u64]
        _lib.synh_fill_q4_packed.argtypes = [vp, u64, u64, u64]
        _lib.synh_fill_q4_scales.argtypes = [vp, u64, u64, u64, f32]
        _lib.synh_fill_uniform_ids.argtypes = [vp, u64, u64, u64, u32, u64]
        for f in (_lib.synh_fill_normal_bf16, _lib.synh_fill_q4_packed, _lib.synh_fill_q4_scales,
                  _lib.synh_fill_uniform_ids):
            f.restype = None
    return _lib


def normal_bf16(seed: int, tid: int, n: int, std: float = 0.02, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    lib().synh_fill_normal_bf16(out.ctypes.data, n, seed, tid, float(gen.normal_scale_f32(std)), start)
    return out


def q4_packed(seed: int, tid: int, nbytes: int) -> np.ndarray:
    out = np.empty(nbytes, dtype=np.uint8)
    lib().synh_fill_q4_packed(out.ctypes.data, nbytes, seed, tid)
    return out


def q4_scales(seed: int, tid: int, nblocks: int, s0: float = gen.Q4_S0) -> np.ndarray:
    out = np.empty(nblocks, dtype=np.uint16)
    lib().synh_fill_q4_scales(out.ctypes.data, nblocks, seed, tid + gen.Q4_SCALE_TID_OFFSET,
                              float(gen.q4_scale_mult_f32(s0)))
    return out


def uniform_ids(seed: int, tid: int, n: int, upper: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    lib().synh_fill_uniform_ids(out.ctypes.data, n, seed, tid, upper, start)
    return out
