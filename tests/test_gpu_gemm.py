"""Parity of the prompt GEMM (tcgen05 tensor cores, TMA-staged tiles, TMEM
accumulator), called through the C ABI, against FP64 products of the exact
bf16 weights with the exact (normalised) activations.

Tolerance: the activations reach the tensor cores as two bf16 parts hi + lo
(relative representation error 2^-16), the weights are exact and the products
accumulate in FP32, so each output is within (2^-16 + gamma_(K+64) + 16 u32)
* sum|w * xhat| of the exact value; the SwiGLU pair adds the activation's
error and the hi/lo split of its result (2^-16 relative)."""
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


def inputs(M, N, K, seed, pair=False):
    rng = np.random.default_rng(seed)
    W = gen.f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    W2 = gen.f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32)) if pair else None
    x = rng.standard_normal((M, K)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, K).astype(np.float32)
    return W, W2, x, g


def xhat_of(x, g, norm):
    if not norm:
        return x.astype(np.float64)
    return np.stack([orc.rmsnorm(r, g, 1e-6) for r in x])


@pytest.mark.parametrize("M,N,K", [(1, 1, 8), (5, 300, 256), (128, 256, 2560), (300, 6176, 2560), (129, 257, 2048),
                                   (1000, 2560, 9216), (2048, 3072, 2560), (77, 2560, 4096)])
@pytest.mark.parametrize("norm", [False, True])
def test_gemm_parity(L, M, N, K, norm):
    torch = _torch()
    W, _, x, g = inputs(M, N, K, M * 7 + N + K)
    Wd, xd, gd = bf16_tensor(W), torch.from_numpy(x).cuda(), torch.from_numpy(g).cuda()
    y = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(L.hy_op_gemm_workspace(M, K), dtype=torch.uint8, device="cuda")
    rc = L.hy_op_gemm(Wd.data_ptr(), N, K, M, xd.data_ptr(), K, gd.data_ptr() if norm else None, 1e-6, y.data_ptr(), N,
                      0, ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0, L.hy_last_error()
    torch.cuda.synchronize()
    xh = xhat_of(x, g, norm)
    Ww = gen.bf16_bits_to_f32(W).astype(np.float64)
    ref = xh @ Ww.T
    tol = (2.0 ** -16 + gamma(K + 64) + 16 * U32) * (np.abs(xh) @ np.abs(Ww).T) + 1e-30
    err = np.abs(to_np(y) - ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, f"{len(bad)} of {M * N} outside the bound, first {bad[:3].tolist()}, worst {(err / tol).max():.3g}"


def test_gemm_accumulates_into_the_residual(L):
    torch = _torch()
    M, N, K = 200, 2560, 2048
    W, _, x, _ = inputs(M, N, K, 3)
    y0 = np.random.default_rng(4).standard_normal((M, N)).astype(np.float32)
    Wd, xd, y = bf16_tensor(W), torch.from_numpy(x).cuda(), torch.from_numpy(y0.copy()).cuda()
    ws = torch.empty(L.hy_op_gemm_workspace(M, K), dtype=torch.uint8, device="cuda")
    assert L.hy_op_gemm(Wd.data_ptr(), N, K, M, xd.data_ptr(), K, None, 0.0, y.data_ptr(), N, 1, ws.data_ptr(),
                        torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    Ww = gen.bf16_bits_to_f32(W).astype(np.float64)
    xh = x.astype(np.float64)
    ref = y0 + xh @ Ww.T
    tol = (2.0 ** -16 + gamma(K + 64) + 16 * U32) * (np.abs(xh) @ np.abs(Ww).T + np.abs(y0)) + 1e-30
    assert np.all(np.abs(to_np(y) - ref) <= tol)


@pytest.mark.parametrize("M,N,K", [(64, 512, 256), (200, 1000, 2560), (130, 9216, 2560)])
def test_gemm_swiglu_pair(L, M, N, K):
    torch = _torch()
    Wg, Wu, x, g = inputs(M, N, K, N + K, pair=True)
    Wgd, Wud, xd, gd = bf16_tensor(Wg), bf16_tensor(Wu), torch.from_numpy(x).cuda(), torch.from_numpy(g).cuda()
    hh = torch.empty((M, N), dtype=torch.int16, device="cuda")
    hl = torch.empty((M, N), dtype=torch.int16, device="cuda")
    ws = torch.empty(L.hy_op_gemm_workspace(M, K), dtype=torch.uint8, device="cuda")
    assert L.hy_op_gemm_swiglu(Wgd.data_ptr(), Wud.data_ptr(), N, K, M, xd.data_ptr(), K, gd.data_ptr(), 1e-6,
                               hh.data_ptr(), hl.data_ptr(), N, ws.data_ptr(),
                               torch.cuda.current_stream().cuda_stream) == 0, L.hy_last_error()
    torch.cuda.synchronize()
    h = (gen.bf16_bits_to_f32(to_np(hh).view(np.uint16)).astype(np.float64) +
         gen.bf16_bits_to_f32(to_np(hl).view(np.uint16)).astype(np.float64))
    xh = xhat_of(x, g, True)
    Wg_, Wu_ = (gen.bf16_bits_to_f32(w).astype(np.float64) for w in (Wg, Wu))
    a, u = xh @ Wg_.T, xh @ Wu_.T
    sa, su = np.abs(xh) @ np.abs(Wg_).T, np.abs(xh) @ np.abs(Wu_).T
    ref = a / (1 + np.exp(-a)) * u
    rel = 2.0 ** -16 + gamma(K + 64) + 16 * U32
    tol = 1.1 * rel * sa * np.abs(u) + rel * su * np.abs(a) + (2.0 ** -15 + 64 * U32) * np.abs(ref) + 1e-30
    err = np.abs(h - ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, f"{len(bad)} of {M * N} outside the bound, worst {(err / tol).max():.3g}"
