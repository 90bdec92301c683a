"""ctypes binding of the CUDA generator copy; fills torch CUDA tensors in place
with the same bits as synth.gen / synth.host."""
from __future__ import annotations

import ctypes

from . import build, gen

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build.build_device())
        u64, f32, u32, vp = ctypes.c_uint64, ctypes.c_float, ctypes.c_uint32, ctypes.c_void_p
        _lib.synd_fill_normal_bf16.argtypes = [vp, u64, u64, u64, f32, u64, vp]
        _lib.synd_fill_q4_packed.argtypes = [vp, u64, u64, u64, vp]
        _lib.synd_fill_q4_scales.argtypes = [vp, u64, u64, u64, f32, vp]
        _lib.synd_fill_uniform_ids.argtypes = [vp, u64, u64, u64, u32, u64, vp]
        _lib.synd_fill_f32.argtypes = [vp, u64, f32, vp]
        for f in (_lib.synd_fill_normal_bf16, _lib.synd_fill_q4_packed, _lib.synd_fill_q4_scales,
                  _lib.synd_fill_uniform_ids, _lib.synd_fill_f32):
            f.restype = ctypes.c_int
    return _lib


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(rc: int) -> None:
    if rc != 0:
        raise RuntimeError(f"synth device fill failed: cuda error {rc}")


def fill_normal_bf16(t, seed: int, tid: int, std: float = 0.02, start: int = 0) -> None:
    _check(lib().synd_fill_normal_bf16(t.data_ptr(), t.numel(), seed, tid, float(gen.normal_scale_f32(std)),
                                       start, _stream()))


def fill_q4_packed(t, seed: int, tid: int) -> None:
    _check(lib().synd_fill_q4_packed(t.data_ptr(), t.numel(), seed, tid, _stream()))


def fill_q4_scales(t, seed: int, tid: int, s0: float = gen.Q4_S0) -> None:
    _check(lib().synd_fill_q4_scales(t.data_ptr(), t.numel(), seed, tid + gen.Q4_SCALE_TID_OFFSET,
                                     float(gen.q4_scale_mult_f32(s0)), _stream()))


def fill_uniform_ids(t, seed: int, tid: int, upper: int, start: int = 0) -> None:
    _check(lib().synd_fill_uniform_ids(t.data_ptr(), t.numel(), seed, tid, upper, start, _stream()))


def fill_f32(t, value: float) -> None:
    _check(lib().synd_fill_f32(t.data_ptr(), t.numel(), float(value), _stream()))
