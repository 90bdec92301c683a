"""Refusals just past the documented limits, through the C ABI: the call
returns its error code and launches nothing (the output buffer keeps its
sentinel, the sequences keep their lengths, the guard word stays clear).

Every buffer is sized for the full requested shape, so that even a launch
the library should have refused would stay inside its buffers.
"""
import ctypes
import dataclasses

import numpy as np
import pytest

from synth import workloads
from tests.gpu_util import to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L(gpu):
    from bandwidth_bound_hybrid_gb300 import build, capi
    build.build()
    return capi.lib()


# (weight format, with an up matrix, columns): the first column count past each
# shared-memory limit of include/hybrid.h, and column counts off the strip width
PAST_LIMITS = [(0, False, 5888), (0, True, 4736), (1, False, 11520), (1, True, 8960), (0, False, 5856), (1, False, 384)]


@pytest.mark.parametrize("fmt,swiglu,C", PAST_LIMITS)
def test_batched_gemv_refuses_past_its_limits(L, fmt, swiglu, C):
    import torch

    from bandwidth_bound_hybrid_gb300 import capi
    R, B = 16, 8
    keep = []

    def tensor():
        if fmt == 0:
            w = torch.zeros((R, C), dtype=torch.bfloat16, device="cuda")
            keep.append(w)
            return capi.hy_tensor(w.data_ptr(), None)
        qs = torch.zeros((R, C // 2), dtype=torch.uint8, device="cuda")
        sc = torch.zeros((R, C // 32), dtype=torch.int16, device="cuda")
        keep.extend([qs, sc])
        return capi.hy_tensor(qs.data_ptr(), sc.data_ptr())

    tw = tensor()
    tu = tensor() if swiglu else None
    x = torch.ones((B, C), dtype=torch.float32, device="cuda")
    y = torch.full((B, R), 7.0, dtype=torch.float32, device="cuda")
    rc = L.hy_op_gemv_batch(ctypes.byref(tw), ctypes.byref(tu) if swiglu else None, fmt, R, C, B, x.data_ptr(), C,
                            None, 1e-6, y.data_ptr(), R, 0, torch.cuda.current_stream().cuda_stream)
    assert rc == capi.HY_ERR_UNSUPPORTED, L.hy_last_error()
    torch.cuda.synchronize()
    assert np.all(to_np(y) == 7.0)


def test_batched_moe_step_refuses_more_than_64_picks(L):
    """Five sequences at top_k 16 would need 80 routed slots in one batched
    step; the call is refused before any launch and every sequence keeps its
    state."""
    import torch

    from bandwidth_bound_hybrid_gb300 import capi
    from bandwidth_bound_hybrid_gb300.model import HybridModel
    shape = dataclasses.replace(workloads.TINY, name="tiny-moe-k16", vocab=512, ffn=0, n_experts=32, top_k=16,
                                expert_ffn=64, shared_ffn=64)
    model = HybridModel(shape, workloads.device_weights(shape), [8] * 5)
    toks = torch.from_numpy(workloads.host.uniform_ids(3, workloads.PROMPT_TID, 5, shape.vocab)).cuda()
    ids = torch.full((5,), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.HybridError) as err:
        model.decode_batch(list(range(5)), toks, ids)
    assert err.value.code == capi.HY_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert [model.seq_len(s) for s in range(5)] == [0] * 5
    assert np.all(to_np(ids) == -1)
    assert model.check_device() == 0
    model.close()
