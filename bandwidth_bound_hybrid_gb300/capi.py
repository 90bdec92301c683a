"""ctypes binding of libhybrid.so (include/hybrid.h), same names as the C ABI.

Argument marshalling only: every step of the decode path runs in the CUDA
library.  Loading fails loudly when the library has not been built; there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(HERE, "libhybrid.so")

HY_OK = 0
HY_ERR_ARG = 1
HY_ERR_CAPACITY = 2
HY_ERR_CUDA = 3
HY_ERR_DEVICE_GUARD = 4
HY_ERR_UNSUPPORTED = 5
HY_ERR_NOMEM = 6

HY_GUARD_WAIT_TIMEOUT = 1
HY_GUARD_BAD_INDEX = 2
HY_GUARD_BAD_POSITION = 4

HY_FLAG_DEBUG = 1
HY_FLAG_NO_GRAPH = 2
HY_FLAG_NO_PDL = 4
HY_FLAG_TOKEN_PREFILL = 16

HY_NOALLOC_SCRATCH_BYTES = 1 << 20

i32, u32, u64, f32, vp, sz = ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
P = ctypes.POINTER


class hy_config(ctypes.Structure):
    _fields_ = [("n_layers", i32), ("hidden", i32), ("vocab", i32), ("ffn", i32), ("gdn_heads", i32),
                ("gdn_dk", i32), ("gdn_dv", i32), ("conv_k", i32), ("attn_q_heads", i32), ("attn_kv_heads", i32),
                ("head_dim", i32), ("attn_layer_mask", u64), ("n_experts", i32), ("top_k", i32),
                ("expert_ffn", i32), ("shared_ffn", i32), ("rms_eps", f32), ("rope_theta", f32),
                ("weight_format", i32), ("attn_splits", i32), ("flags", u32), ("kv_format", i32)]


class hy_tensor(ctypes.Structure):
    _fields_ = [("w", vp), ("scales", vp)]


class hy_layer_weights(ctypes.Structure):
    _fields_ = [("norm1", vp), ("w_in", hy_tensor), ("conv_w", vp), ("w_o", hy_tensor), ("norm2", vp),
                ("w_gate", hy_tensor), ("w_up", hy_tensor), ("w_down", hy_tensor), ("router", vp),
                ("exp_gate", hy_tensor), ("exp_up", hy_tensor), ("exp_down", hy_tensor),
                ("sh_gate", hy_tensor), ("sh_up", hy_tensor), ("sh_down", hy_tensor)]


class hy_weights(ctypes.Structure):
    _fields_ = [("embed", vp), ("final_norm", vp), ("lm_head", hy_tensor), ("layers", P(hy_layer_weights))]


# name -> (restype, argtypes), exactly the functions declared in include/hybrid.h
SIGNATURES = {
    "hy_last_error": (ctypes.c_char_p, []),
    "hy_model_create": (ctypes.c_int, [P(hy_config), P(hy_weights), P(vp)]),
    "hy_model_free": (None, [vp]),
    "hy_cache_alloc": (ctypes.c_int, [vp, i32, P(i32), P(vp)]),
    "hy_cache_free": (None, [vp]),
    "hy_cache_alloc_paged": (ctypes.c_int, [vp, i32, P(i32), i32, i32, P(vp)]),
    "hy_cache_free_pages": (i32, [vp]),
    "hy_seq_reset": (ctypes.c_int, [vp, i32, vp]),
    "hy_seq_len": (i32, [vp, i32]),
    "hy_seq_capacity": (i32, [vp, i32]),
    "hy_step_kernels": (i32, [vp]),
    "hy_step_splits": (i32, [vp, i32]),
    "hy_experts_read": (ctypes.c_int, [vp, vp, vp]),
    "hy_seq_fill_synthetic": (ctypes.c_int, [vp, i32, i32, u64, vp]),
    "hy_prefill": (ctypes.c_int, [vp, vp, i32, vp, i32, vp, vp]),
    "hy_decode_step": (ctypes.c_int, [vp, vp, P(i32), i32, vp, vp, vp, vp]),
    "hy_decode_step_host": (ctypes.c_int, [vp, vp, P(i32), i32, vp, vp, vp, vp]),
    "hy_check_device": (ctypes.c_int, [vp, vp, P(u32)]),
    "hy_debug_hidden": (ctypes.c_int, [vp, i32, vp, vp]),
    "hy_debug_router": (ctypes.c_int, [vp, i32, vp, vp, vp]),
    "hy_op_check_device": (ctypes.c_int, [vp, P(u32)]),
    "hy_op_gemv": (ctypes.c_int, [vp, i32, i32, vp, vp, f32, vp, i32, vp]),
    "hy_op_gemv_swiglu": (ctypes.c_int, [vp, vp, i32, i32, vp, vp, f32, vp, vp]),
    "hy_op_gemv_batch": (ctypes.c_int, [P(hy_tensor), P(hy_tensor), i32, i32, i32, i32, vp, i32, vp, f32, vp, i32, i32,
                                        vp]),
    "hy_op_gemm_workspace": (sz, [i32, i32]),
    "hy_op_gemm": (ctypes.c_int, [vp, i32, i32, i32, vp, i32, vp, f32, vp, i32, i32, vp, vp]),
    "hy_op_gemm_swiglu": (ctypes.c_int, [vp, vp, i32, i32, i32, vp, i32, vp, f32, vp, vp, i32, vp, vp]),
    "hy_op_moe_gateup": (ctypes.c_int, [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, f32, vp, vp, vp, vp]),
    "hy_op_moe_down": (ctypes.c_int, [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]),
    "hy_op_argmax_workspace": (sz, []),
    "hy_op_gemv_argmax": (ctypes.c_int, [vp, i32, i32, vp, vp, f32, vp, vp, vp, vp]),
    "hy_op_gdn_step": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp]),
    "hy_op_rope_table": (ctypes.c_int, [vp, i32, i32, f32, vp]),
    "hy_op_attention_workspace": (sz, [i32, i32, i32, i32]),
    "hy_op_attention": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, vp, vp, i32, vp, vp, vp]),
    "hy_op_attention_noalloc": (ctypes.c_int, [vp, vp, vp, i32, i32, i32, i32, vp, vp, i32, vp, vp]),
    "hy_op_attention_i8": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, i32, vp, vp, vp]),
}

_lib = None


def lib():
    """Load libhybrid.so (raises if it has not been built: no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(SO):
            raise RuntimeError(f"{SO} is missing: build it with bandwidth_bound_hybrid_gb300.build.build()")
        L = ctypes.CDLL(SO)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class HybridError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = lib().hy_last_error().decode(errors="replace")
        super().__init__(f"{where} failed with code {code}: {msg}")
        self.code = code


def check(code: int, where: str) -> None:
    if code != HY_OK:
        raise HybridError(code, where)


def __getattr__(name):
    if name in SIGNATURES:
        return getattr(lib(), name)
    raise AttributeError(name)
