"""The C-ABI library loads and exports every function include/hybrid.h
declares; the Python binding covers exactly those names (CPU only: no
compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hybrid.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(hy_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def built_lib():
    from bandwidth_bound_hybrid_gb300 import build
    return ctypes.CDLL(build.build())


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("hy_model_create", "hy_model_free", "hy_cache_alloc", "hy_cache_free", "hy_prefill",
              "hy_decode_step", "hy_decode_step_host", "hy_seq_len", "hy_seq_reset", "hy_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(built_lib):
    missing = [n for n in declared_functions() if not hasattr(built_lib, n)]
    assert not missing, missing


def test_binding_signatures_match_header(built_lib):
    from bandwidth_bound_hybrid_gb300 import capi
    assert sorted(capi.SIGNATURES) == declared_functions()


def test_last_error_is_empty_string_before_any_call(built_lib):
    built_lib.hy_last_error.restype = ctypes.c_char_p
    assert built_lib.hy_last_error() == b""


def test_null_arguments_are_rejected_without_a_gpu(built_lib):
    from bandwidth_bound_hybrid_gb300 import capi
    L = capi.lib()
    out = ctypes.c_void_p()
    assert L.hy_model_create(None, None, ctypes.byref(out)) == capi.HY_ERR_ARG
    assert b"null" in L.hy_last_error()
    assert L.hy_seq_len(None, 0) == -1
    assert L.hy_decode_step(None, None, None, 1, None, None, None, None) == capi.HY_ERR_ARG


def test_new_entry_points_reject_bad_arguments_without_a_gpu(built_lib):
    """Argument checks come before any device call."""
    from bandwidth_bound_hybrid_gb300 import capi
    L = capi.lib()
    total = ctypes.c_uint64(7)
    assert L.hy_experts_read(None, None, ctypes.byref(total)) == capi.HY_ERR_ARG
    assert L.hy_seq_fill_synthetic(None, 0, 16, 1, None) == capi.HY_ERR_ARG
    assert L.hy_step_kernels(None) == 0
    w = capi.hy_tensor(None, None)
    # no weights, batch 0 and 9, a bad format: all refused before a launch
    args = lambda wt, fmt, batch: (ctypes.byref(wt), None, fmt, 16, 256, batch, None, 256, None, 1e-6, None, 16, 0,
                                   None)
    assert L.hy_op_gemv_batch(*args(w, 0, 1)) == capi.HY_ERR_ARG
    assert L.hy_op_gemv_batch(None, None, 0, 16, 256, 1, None, 256, None, 1e-6, None, 16, 0, None) == capi.HY_ERR_ARG
    for batch in (0, 9):
        assert L.hy_op_gemv_batch(*args(w, 0, batch)) == capi.HY_ERR_ARG
    assert L.hy_op_gemv_batch(*args(w, 2, 1)) == capi.HY_ERR_ARG
    assert b"batched" in L.hy_last_error()


def test_config_limits_are_checked_before_any_device_call(built_lib):
    """hy_model_create checks the config before it looks at weights or the
    device: a config past a documented limit gets its error code, one at the
    limit passes on to the weight checks (here: an empty weight table)."""
    import dataclasses

    from bandwidth_bound_hybrid_gb300 import capi
    from bandwidth_bound_hybrid_gb300.model import make_config
    from synth import workloads
    L = capi.lib()
    moe = dataclasses.replace(workloads.MOE35B, n_layers=4, attn_layers=(3,))

    def create(shape, **over):
        cfg = make_config(shape)
        for k, v in over.items():
            setattr(cfg, k, v)
        out = ctypes.c_void_p()
        rc = L.hy_model_create(ctypes.byref(cfg), ctypes.byref(capi.hy_weights()), ctypes.byref(out))
        assert not out.value
        return rc, L.hy_last_error().decode()

    at_limit = (capi.HY_ERR_ARG, "weights.layers is null")
    assert create(moe, n_experts=511) == at_limit
    assert create(moe, n_experts=512)[0] == capi.HY_ERR_UNSUPPORTED
    assert create(moe, top_k=16) == at_limit
    assert create(moe, top_k=17)[0] == capi.HY_ERR_ARG
    assert create(moe, shared_ffn=1024)[0] == capi.HY_ERR_UNSUPPORTED
    dense = workloads.DENSE4B
    assert create(dense) == at_limit
    assert create(dense, n_layers=65)[0] == capi.HY_ERR_ARG
    assert create(dense, head_dim=96)[0] == capi.HY_ERR_UNSUPPORTED
    assert create(dense, attn_kv_heads=1)[0] == capi.HY_ERR_UNSUPPORTED  # 16 q heads per kv head
    assert create(dense, gdn_dk=32)[0] == capi.HY_ERR_UNSUPPORTED
    q4 = dataclasses.replace(dense, weight_format=1)
    assert create(q4) == at_limit
    assert create(q4, hidden=2560 + 128)[0] == capi.HY_ERR_UNSUPPORTED
