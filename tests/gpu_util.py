"""Helpers shared by the GPU parity tests (tolerances and comparisons).

Floating-point tolerance for a single dot product of n terms computed in FP32
(any summation order) against the FP64 oracle: the standard worst-case bound
|fl(sum) - sum| <= gamma_n * sum|terms|, gamma_n = n u / (1 - n u), u = 2^-24,
plus a few ulps of the result for the scaling applied before or after it.
"""
from __future__ import annotations

import numpy as np

U32 = 2.0 ** -24


def gamma(n: int) -> float:
    return n * U32 / (1 - n * U32)


def assert_dot_close(got, ref, absdot, n: int, what: str = "", extra_ulps: float = 16.0):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = gamma(n) * np.asarray(absdot, dtype=np.float64) + extra_ulps * U32 * np.abs(ref) + 1e-30
    err = np.abs(got - ref)
    bad = np.nonzero(err > tol)[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {got.size} outside the FP32 dot-product bound; "
                           f"worst index {bad[np.argmax((err / tol)[bad])]}, err {err[bad].max():.3g}")


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def to_np(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def bf16_tensor(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_bits(t) -> np.ndarray:
    import torch
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
