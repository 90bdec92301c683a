"""hy_op_attention_noalloc, the attention entry point for callers that cannot
allocate device memory (a host framework owning the whole memory budget, a
latency path where an allocation is not allowed, a plug-in restricted to its
host's allocator): its scratch is a fixed array inside the library instead of
a caller workspace.

Checked through the C ABI against hy_op_attention on the same inputs, on two
calls in a row with different shapes (the second call finds the first call's
leftovers in the shared array), plus the size limit.  This file is named to
be collected after the other parity files (only the full-size ones follow),
so that a run stopping at its first failure has run them before it.
"""
import numpy as np
import pytest

from synth import gen
from tests.gpu_util import bf16_tensor, rel_l2, to_np

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
