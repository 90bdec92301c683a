"""Parity of the batched (up to 8 token vectors) tensor-core GEMV, called
through the C ABI, against the FP64 oracle, for bf16 and 4-bit block weights.

Tolerance: the kernel represents the (normalised) token vector in the MMA
operand type (for bf16 weights as two bf16 parts hi + lo, relative error
2^-16; FP16 for 4-bit weights, 2^-11), dequantises 4-bit weights exactly and
accumulates in FP32, so each output is within (u_operand + gamma_n + 16 u32) *
sum|w * xhat| of the exact dot product of the exact weights with the exact
xhat."""
import ctypes

import numpy as np
import pytest

from oracle import oracle as orc
from synth import gen
from tests.gpu_util import bf16_tensor, gamma, to_np

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def L(gpu):
    from bandwidth_bound_hybrid_gb300 import build, capi
    build.build()
    return capi.lib()


def _torch():
    import torch
    return torch


def q4_weights(seed, tid, R, C):
    qs = gen.q4_packed(seed, tid, R * C // 2).reshape(R, C // 2)
    sc = gen.q4_scales(seed, tid, R * C // 32, gen.Q4_S0).reshape(R, C // 32)
    return qs, sc


def dev_tensor(w, fmt):
    """hy_tensor over device copies (kept alive by the returned list)."""
    from bandwidth_bound_hybrid_gb300 import capi
    torch = _torch()
    if fmt == 0:
        d = bf16_tensor(w)
        return capi.hy_tensor(d.data_ptr(), None), [d]
    qs = torch.from_numpy(np.ascontiguousarray(w[0])).cuda()
    sc = torch.from_numpy(np.ascontiguousarray(w[1]).view(np.int16)).cuda()
    return capi.hy_tensor(qs.data_ptr(), sc.data_ptr()), [qs, sc]


def widen(w, fmt):
    if fmt == 0:
        return gen.bf16_bits_to_f32(w).astype(np.float64)
    R = w[0].shape[0]
    return np.stack([orc.mat_row(w, r) for r in range(R)])


def run(L, fmt, R, C, B, norm, accumulate=False, swiglu=False, seed=0):
    torch = _torch()
    rng = np.random.default_rng(seed + R * 31 + C + B)
    if fmt == 0:
        W = gen.f32_to_bf16_bits((rng.standard_normal((R, C)) * 0.02).astype(np.float32))
        Wu = gen.f32_to_bf16_bits((rng.standard_normal((R, C)) * 0.02).astype(np.float32)) if swiglu else None
    else:
        W = q4_weights(seed, 11, R, C)
        Wu = q4_weights(seed, 12, R, C) if swiglu else None
    x = rng.standard_normal((B, C)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, C).astype(np.float32)
    y0 = rng.standard_normal((B, R)).astype(np.float32)
    tw, keep = dev_tensor(W, fmt)
    tu, keep2 = dev_tensor(Wu, fmt) if swiglu else (None, [])
    xd, gd = torch.from_numpy(x).cuda(), torch.from_numpy(g).cuda()
    y = torch.from_numpy(y0.copy()).cuda()
    rc = L.hy_op_gemv_batch(ctypes.byref(tw), ctypes.byref(tu) if swiglu else None, fmt, R, C, B, xd.data_ptr(), C,
                            gd.data_ptr() if norm else None, 1e-6, y.data_ptr(), R, int(accumulate),
                            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, L.hy_last_error()
    torch.cuda.synchronize()
    got = to_np(y)
    uop = 2.0 ** -16 if fmt == 0 else 2.0 ** -11
    Wd = widen(W, fmt)
    for b in range(B):
        xh = orc.rmsnorm(x[b], g, 1e-6) if norm else x[b].astype(np.float64)
        a = Wd @ xh
        sa = np.abs(Wd) @ np.abs(xh)
        rel = uop + gamma(C + 64) + 16 * U32
        if swiglu:
            Wud = widen(Wu, fmt)
            u = Wud @ xh
            su = np.abs(Wud) @ np.abs(xh)
            ref = np.array([orc.lib().orc_silu(float(v)) for v in a]) * u
            tol = 1.1 * rel * sa * np.abs(u) + rel * su * np.abs(a) + 64 * U32 * (np.abs(ref) + 1e-30)
        else:
            ref = a + (y0[b].astype(np.float64) if accumulate else 0.0)
            tol = rel * sa + 16 * U32 * (np.abs(ref) + 1e-30)
        err = np.abs(got[b] - ref)
        bad = np.nonzero(err > tol)[0]
        assert bad.size == 0, f"token {b}: {bad.size} of {R} outside the bound, worst {err[bad].max():.3g}"
    del keep, keep2


@pytest.mark.parametrize("R,C,B", [(16, 256, 1), (37, 512, 3), (300, 2048, 8), (2560, 2048, 5), (5, 1536, 2)])
@pytest.mark.parametrize("norm", [False, True])
def test_batch_gemv_bf16(L, R, C, B, norm):
    run(L, 0, R, C, B, norm)


def test_batch_gemv_rejects_rows_too_wide_for_a_stage(L):
    """bf16 rows wider than two 16-row tiles allow in shared memory are
    refused before any launch (the engine then runs such a matrix per token)."""
    from bandwidth_bound_hybrid_gb300 import capi
    torch = _torch()
    W = torch.zeros((16, 9216), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((2, 9216), device="cuda")
    y = torch.full((2, 16), 3.0, device="cuda")
    tw = capi.hy_tensor(W.data_ptr(), None)
    rc = L.hy_op_gemv_batch(ctypes.byref(tw), None, 0, 16, 9216, 2, x.data_ptr(), 9216, None, 1e-6, y.data_ptr(), 16,
                            0, torch.cuda.current_stream().cuda_stream)
    assert rc == capi.HY_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)


@pytest.mark.parametrize("R,C,B", [(16, 256, 1), (100, 512, 4), (2048, 2048, 8), (6176, 2048, 8), (33, 4608, 7)])
@pytest.mark.parametrize("norm", [False, True])
def test_batch_gemv_q4(L, R, C, B, norm):
    run(L, 1, R, C, B, norm)


@pytest.mark.parametrize("fmt", [0, 1])
def test_batch_gemv_accumulate(L, fmt):
    run(L, fmt, 257, 2048, 6, True, accumulate=True)


@pytest.mark.parametrize("fmt,C", [(0, 1024), (1, 2048)])
def test_batch_gemv_swiglu(L, fmt, C):
    run(L, fmt, 512, C, 8, True, swiglu=True)


def test_batch_of_one_equals_each_token_alone(L):
    """Tokens do not interact: a batch of 8 gives each token's batch-1 result."""
    torch = _torch()
    rng = np.random.default_rng(4)
    R, C = 700, 2048
    W = q4_weights(3, 5, R, C)
    tw, keep = dev_tensor(W, 1)
    x = torch.from_numpy(rng.standard_normal((8, C)).astype(np.float32)).cuda()
    g = torch.ones(C, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    yb = torch.empty((8, R), device="cuda")
    assert L.hy_op_gemv_batch(ctypes.byref(tw), None, 1, R, C, 8, x.data_ptr(), C, g.data_ptr(), 1e-6, yb.data_ptr(), R,
                              0, st) == 0
    for b in range(8):
        y1 = torch.empty((1, R), device="cuda")
        assert L.hy_op_gemv_batch(ctypes.byref(tw), None, 1, R, C, 1, x[b].data_ptr(), C, g.data_ptr(), 1e-6,
                                  y1.data_ptr(), R, 0, st) == 0
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_np(y1)[0], to_np(yb)[b])
    del keep


@pytest.mark.parametrize("fmt,C,swiglu", [(0, 5824, False), (0, 4672, True), (1, 11264, False), (1, 8704, True)])
def test_batch_gemv_at_the_documented_column_limits(L, fmt, C, swiglu):
    """The widest inputs include/hybrid.h promises for hy_op_gemv_batch (bf16
    5824, or 4672 with an up matrix; 4-bit 11264, or 8704 with an up matrix),
    a full batch of 8, where the token vectors take the most shared memory."""
    run(L, fmt, 160, C, 8, True, swiglu=swiglu)
