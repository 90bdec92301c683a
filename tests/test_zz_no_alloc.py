"""hy_op_attention_noalloc, the attention entry point for callers that cannot
allocate device memory (a host framework owning the whole memory budget, a
latency path where an allocation is not allowed, a plug-in restricted to its
host's allocator): its scratch is a fixed array inside the library instead of
a caller workspace.

Checked through the C ABI against hy_op_attention on the same inputs, on two
calls in a row with different shapes (the second call finds the first call's
leftovers in the shared array); against the oracle element by element; its
device-side refusal of a full cache, read back with hy_op_check_device; and
the size limit.  This file is named to
be collected after the other parity files (only the full-size ones follow),
so that a run stopping at its first failure has run them before it.
"""
import numpy as np
import pytest

from synth import gen
from tests.gpu_util import assert_elementwise, bf16_tensor, rel_l2, to_np

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-5  # the attention parity tolerance of the op tests


@pytest.fixture(scope="module")
def L(gpu):
    from bandwidth_bound_hybrid_gb300 import build, capi
    build.build()
    return capi.lib()


def _inputs(rng, nq, nkv, hd, cap, T):
    import torch
    Kc = gen.f32_to_bf16_bits(rng.standard_normal((nkv, cap, hd)).astype(np.float32))
    Vc = gen.f32_to_bf16_bits(rng.standard_normal((nkv, cap, hd)).astype(np.float32))
    y = torch.from_numpy(rng.standard_normal((nq + 2 * nkv) * hd).astype(np.float32)).cuda()
    ln = torch.tensor([T], dtype=torch.int32, device="cuda")
    return Kc, Vc, y, ln


def test_noalloc_matches_workspace_attention_on_consecutive_calls(L):
    import torch
    st = torch.cuda.current_stream().cuda_stream
    # (nq, nkv, hd, T, nsplit): the dense and MoE attention shapes, automatic and fixed splits
    calls = [(16, 4, 128, 4095, 0), (16, 2, 256, 1500, 7)]
    for i, (nq, nkv, hd, T, nsplit) in enumerate(calls):
        rng = np.random.default_rng(100 + i)
        cap = T + 9
        Kc, Vc, y, ln = _inputs(rng, nq, nkv, hd, cap, T)
        table = torch.empty((cap, hd // 2, 2), dtype=torch.float32, device="cuda")
        assert L.hy_op_rope_table(table.data_ptr(), cap, hd, 1e4, st) == 0
        outs, caches = [], []
        for noalloc in (False, True):
            K, V = bf16_tensor(Kc), bf16_tensor(Vc)
            o = torch.full((nq * hd,), 3.0, dtype=torch.float32, device="cuda")
            if noalloc:
                rc = L.hy_op_attention_noalloc(y.data_ptr(), K.data_ptr(), V.data_ptr(), cap, nq, nkv, hd,
                                               ln.data_ptr(), table.data_ptr(), nsplit, o.data_ptr(), st)
            else:
                ws = torch.zeros(L.hy_op_attention_workspace(nq, nkv, hd, nsplit), dtype=torch.uint8, device="cuda")
                rc = L.hy_op_attention(y.data_ptr(), K.data_ptr(), V.data_ptr(), cap, nq, nkv, hd, ln.data_ptr(),
                                       table.data_ptr(), nsplit, o.data_ptr(), ws.data_ptr(), st)
            assert rc == 0, L.hy_last_error()
            torch.cuda.synchronize()
            outs.append(to_np(o).copy())
            caches.append((to_np(K.view(torch.int16)).copy(), to_np(V.view(torch.int16)).copy()))
        ref, got = outs
        assert np.all(np.isfinite(got))
        assert rel_l2(got, ref) <= ATTN_TOL, f"call {i}: rel-L2 {rel_l2(got, ref):.3g}"
        for a, b in zip(caches[0], caches[1]):  # the same new K/V row appended, nothing else touched
            np.testing.assert_array_equal(a, b)


def test_noalloc_rejects_scratch_beyond_its_fixed_size(L):
    import torch

    from bandwidth_bound_hybrid_gb300 import capi
    st = torch.cuda.current_stream().cuda_stream
    nq, nkv, hd, nsplit, cap, T = 64, 8, 256, 32, 40, 30
    assert L.hy_op_attention_workspace(nq, nkv, hd, nsplit) > capi.HY_NOALLOC_SCRATCH_BYTES
    rng = np.random.default_rng(7)
    Kc, Vc, y, ln = _inputs(rng, nq, nkv, hd, cap, T)
    K, V = bf16_tensor(Kc), bf16_tensor(Vc)
    table = torch.zeros((cap, hd // 2, 2), dtype=torch.float32, device="cuda")
    o = torch.full((nq * hd,), 3.0, dtype=torch.float32, device="cuda")
    rc = L.hy_op_attention_noalloc(y.data_ptr(), K.data_ptr(), V.data_ptr(), cap, nq, nkv, hd, ln.data_ptr(),
                                   table.data_ptr(), nsplit, o.data_ptr(), st)
    assert rc == capi.HY_ERR_UNSUPPORTED
    assert b"exceeds" in L.hy_last_error()
    torch.cuda.synchronize()
    assert torch.all(o == 3.0)  # nothing was launched
    np.testing.assert_array_equal(to_np(K.view(torch.int16)).view(np.uint16), Kc)


def test_noalloc_against_the_oracle_elementwise(L):
    """The same call checked against the oracle itself, each output element
    within its bound, with a negative split count (automatic, as for
    hy_op_attention)."""
    import torch

    from tests.test_gpu_ops import attention_reference
    st = torch.cuda.current_stream().cuda_stream
    nq, nkv, hd, T = 16, 2, 256, 2303
    cap = T + 5
    rng = np.random.default_rng(31)
    Kc = gen.f32_to_bf16_bits(rng.uniform(-1, 1, (nkv, cap, hd)).astype(np.float32))
    Vc = gen.f32_to_bf16_bits(rng.uniform(-1, 1, (nkv, cap, hd)).astype(np.float32))
    y = rng.standard_normal((nq + 2 * nkv) * hd).astype(np.float32)
    K, V, yd = bf16_tensor(Kc), bf16_tensor(Vc), torch.from_numpy(y).cuda()
    ln = torch.tensor([T], dtype=torch.int32, device="cuda")
    table = torch.empty((cap, hd // 2, 2), dtype=torch.float32, device="cuda")
    assert L.hy_op_rope_table(table.data_ptr(), cap, hd, 1e4, st) == 0
    o = torch.full((nq * hd,), 3.0, dtype=torch.float32, device="cuda")
    assert L.hy_op_attention_noalloc(yd.data_ptr(), K.data_ptr(), V.data_ptr(), cap, nq, nkv, hd, ln.data_ptr(),
                                     table.data_ptr(), -1, o.data_ptr(), st) == 0, L.hy_last_error()
    torch.cuda.synchronize()
    ref, _, _, tol = attention_reference(y, Kc, Vc, nq, nkv, hd, T, 0)
    assert_elementwise(to_np(o).reshape(nq, hd), ref, tol, "no-allocation attention")


def test_noalloc_full_cache_is_refused_on_the_device_and_reported(L):
    """A position at the capacity: the kernel leaves the output and the cache
    alone and sets the position guard, which hy_op_check_device reports once
    (then clears); the next valid call reports nothing."""
    import ctypes

    import torch

    from bandwidth_bound_hybrid_gb300 import capi
    st = torch.cuda.current_stream().cuda_stream
    nq, nkv, hd, cap = 4, 2, 64, 32
    rng = np.random.default_rng(5)
    Kc, Vc, y, _ = _inputs(rng, nq, nkv, hd, cap, 0)
    K, V = bf16_tensor(Kc), bf16_tensor(Vc)
    table = torch.empty((cap, hd // 2, 2), dtype=torch.float32, device="cuda")
    assert L.hy_op_rope_table(table.data_ptr(), cap, hd, 1e4, st) == 0
    bits = ctypes.c_uint32(0)
    L.hy_op_check_device(st, ctypes.byref(bits))  # start from a clear word
    for T, want in ((cap, capi.HY_GUARD_BAD_POSITION), (cap - 1, 0)):
        ln = torch.tensor([T], dtype=torch.int32, device="cuda")
        o = torch.full((nq * hd,), 3.0, dtype=torch.float32, device="cuda")
        assert L.hy_op_attention_noalloc(y.data_ptr(), K.data_ptr(), V.data_ptr(), cap, nq, nkv, hd, ln.data_ptr(),
                                         table.data_ptr(), 0, o.data_ptr(), st) == 0
        rc = L.hy_op_check_device(st, ctypes.byref(bits))
        assert bits.value == want
        assert rc == (capi.HY_ERR_DEVICE_GUARD if want else capi.HY_OK)
        if want:
            assert torch.all(o == 3.0)
            np.testing.assert_array_equal(to_np(K.view(torch.int16)).view(np.uint16), Kc)
            assert L.hy_op_check_device(st, ctypes.byref(bits)) == capi.HY_OK and bits.value == 0  # cleared
        else:
            assert np.all(np.isfinite(to_np(o)))
