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


# ---------------------------------------------------------------- attention
#
# Element-wise bound for the split-KV decode attention (FP32 kernel) against
# the FP64 oracle, per (query head j, output dim d).  With s_t the exact scaled
# scores, p_t their softmax and o the exact output, a kernel that computes
# every score with an error delta_t and every exponential with a relative
# error eps_t returns, to first order,
#     o_d + sum_t p_t (delta_t + eps_t) (V_td - o_d) + (sum rounding) ,
# because a common shift of all scores cancels in the softmax.  So
#     |err_d| <= sum_t p_t (delta_t + eps_t) |V_td - o_d| + rel_sum * sum_t p_t |V_td|
# with
#   delta_t = gamma(hd+16) * scale * sum_i |q_i K_ti|           (FP32 dot product)
#           + scale * sum_i dq_i |K_ti|,  dq_i = 6 u (|a_i| + |b_i|) (RoPE of the
#             FP32 projection pair (a, b) with FP32 cos/sin, then the scale)
#           + [t = T] 2^-8 scale * sum_{i in F} |q_i K_Ti|      (F: elements of the
#             new key row near a bf16 rounding boundary, where the kernel's
#             FP32 rotation may round to the neighbouring code; the value row
#             is rounded from the same FP32 projection value on both sides)
#   eps_t   = 2 (2^-21 + 2 u |s_t - max s|)                      (two fast
#             exponentials: the online softmax and the split combine)
#   rel_sum = gamma(npos + nsplit + 64) + 2^-21 (tiles + 4) + 2 u (max s - min s)
#             (FP32 sums of p V and of p, and the per-tile rescales)
# plus 16 u |o_d|.
# The tests take ATTN_SAFETY times this bound.
ATTN_SAFETY = 4.0


def bf16_tie_mask(x, err):
    """Elements of x (FP64) whose bf16 code (rounded through FP32) can change
    when x moves by up to err: the FP32 computation of x may round either way."""
    from synth import gen
    x = np.asarray(x, dtype=np.float64)
    lo = gen.f32_to_bf16_bits((x - err).astype(np.float32))
    hi = gen.f32_to_bf16_bits((x + err).astype(np.float32))
    return lo != hi


def rope_pair_abs(v):
    """|a_i| + |b_i| for each element of a rotate-half pair (i, i + hd/2)."""
    v = np.asarray(v, dtype=np.float64)
    return np.abs(v) + np.abs(np.roll(v, v.shape[-1] // 2, axis=-1))


def attention_tolerance(yq, q, Kw, Vw, npos, ref, nsplit, tile_positions=64, k_flip=None):
    """Per-element bound [nq][hd] (see above).  yq: FP32 projection of the
    queries before RoPE [nq][hd]; q: the rotated queries (FP64) [nq][hd]; Kw,
    Vw: widened caches [nkv][>=npos][hd] holding the new row at npos - 1; ref:
    the exact output [nq][hd]; nsplit: split count of the kernel; k_flip:
    [nkv][hd] mask of new-key elements whose bf16 code may differ (None: none)."""
    yq = np.asarray(yq, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    nq, hd = q.shape
    nkv = Kw.shape[0]
    G = nq // nkv
    scale = 1.0 / np.sqrt(hd)
    T = npos - 1
    tol = np.zeros_like(q)
    ntile = -(-npos // max(nsplit, 1) // tile_positions) + 2
    for j in range(nq):
        g = j // G
        Kg = Kw[g, :npos].astype(np.float64)
        Vg = Vw[g, :npos].astype(np.float64)
        aK = np.abs(Kg)
        s = Kg @ q[j] * scale
        M = s.max()
        p = np.exp(s - M)
        p /= p.sum()
        absd = aK @ np.abs(q[j]) * scale
        delta = gamma(hd + 16) * absd + aK @ (6 * U32 * rope_pair_abs(yq[j]) * scale)
        if k_flip is not None:
            delta[T] += 2.0 ** -8 * scale * np.sum(k_flip[g] * np.abs(q[j]) * aK[T])
        eps = 2 * (2.0 ** -21 + 2 * U32 * np.abs(s - M))
        term1 = ((delta + eps) * p) @ np.abs(Vg - ref[j])
        rel_sum = gamma(npos + nsplit + 64) + 2.0 ** -21 * (ntile + 4) + 2 * U32 * (M - s.min())
        term2 = rel_sum * (p @ np.abs(Vg))
        tol[j] = ATTN_SAFETY * (term1 + term2) + 16 * U32 * np.abs(ref[j]) + 1e-30
    return tol


def assert_elementwise(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{what}: {len(bad)} of {got.size} elements outside their bound; first {bad[:4].tolist()}, "
                           f"worst err/tol {(err / tol).max():.3g}")


# ---------------------------------------------------------------- Gated DeltaNet
#
# Per state row bound for the in-place delta rule (FP32 kernel) against the
# FP64 oracle (whose state is stored in FP32).  One step maps a state row S_i
# (value row i, over the key index) to
#     S_i' = alpha S_i + d_i k,  d_i = beta (v_i - alpha u_i),  u_i = S_i . k,
# i.e. S_i' = alpha S_i (I - beta k k^T) + beta v_i k^T.  ||k|| = 1 and
# 0 < beta < 1 make (I - beta k k^T) a contraction, so an error Delta_i already
# in the row is carried as ||alpha Delta_i (I - beta k k^T)|| <= alpha ||Delta_i||
# and the row's 2-norm error obeys
#     B_i(t) = alpha B_i(t-1) + e_i(t)
# with the step's own error (first order):
#   e_i = e_a ||S_i|| + |Delta d_i| + |d_i| e_k + 3 u ||S_i'|| + u |d_i|
#   |Delta d_i| = e_b |v_i - alpha u_i| + beta (e_v + e_a |u_i| + alpha |Delta u_i|) + 3 u |d_i|
#   |Delta u_i| = gamma(dk + 8) sum_j |S_ij k_j| + ||S_i|| e_k
# where the inputs' errors come from the FP32 conv (taps over the ring), the
# fast-exponential SiLU and sigmoid, and the L2 normalisation:
#   e_a = 2^-19 alpha, e_b = 2^-19 beta,
#   e_v = 2^-19 |v_i| + 1.1 gamma(conv_k + 4) A_i          (A: sum over taps |w u|)
#   e_k = 2 (1.1 gamma(conv_k + 4) ||A_k|| / ||silu(c_k)|| + 2^-19 + gamma(dk + 8))
#   e_q = e_k-form for q, divided by sqrt(dk) (q is scaled by dk^-1/2).
# The output o_i = S_i' . q then errs by at most
#     B_i ||q|| + ||S_i'|| e_q + gamma(dk + 8) sum_j |S'_ij q_j| + 16 u |o_i|.
# The tests take GDN_SAFETY times these bounds.
GDN_SAFETY = 4.0


def gdn_step_bounds(S_prev, qh, kh, v, alpha, beta, A_q, A_k, A_v, c_q, c_k, S_new, o_ref, B_prev, conv_k):
    """One head, one step.  S_prev, S_new: the oracle's FP32 state rows
    [dv][dk] before and after; qh, kh: normalised (and for q scaled) vectors;
    v: value inputs [dv]; A_*: conv sums of |tap * input| per channel; c_q, c_k:
    SiLU outputs before normalisation; o_ref: the oracle's outputs [dv];
    B_prev: the rows' carried bound [dv].  Returns (B [dv], o_tol [dv])."""
    dv, dk = S_prev.shape
    S = S_prev.astype(np.float64)
    Sn = S_new.astype(np.float64)
    u = S @ kh
    d = beta * (v - alpha * u)
    nS = np.linalg.norm(S, axis=1)
    nSn = np.linalg.norm(Sn, axis=1)
    cg = 1.1 * gamma(conv_k + 4)
    e_k = 2 * (cg * np.linalg.norm(A_k) / max(np.linalg.norm(c_k), 1e-30) + 2.0 ** -19 + gamma(dk + 8))
    e_q = 2 * (cg * np.linalg.norm(A_q) / max(np.linalg.norm(c_q), 1e-30) + 2.0 ** -19 + gamma(dk + 8)) / np.sqrt(dk)
    e_a, e_b = 2.0 ** -19 * alpha, 2.0 ** -19 * beta
    e_v = 2.0 ** -19 * np.abs(v) + cg * A_v
    du = gamma(dk + 8) * (np.abs(S) @ np.abs(kh)) + nS * e_k
    dd = e_b * np.abs(v - alpha * u) + beta * (e_v + e_a * np.abs(u) + alpha * du) + 3 * U32 * np.abs(d)
    e = e_a * nS + dd + np.abs(d) * e_k + 3 * U32 * nSn + U32 * np.abs(d)
    B = alpha * B_prev + e
    o_tol = (B * np.linalg.norm(qh) + nSn * e_q + gamma(dk + 8) * (np.abs(Sn) @ np.abs(qh))) + 16 * U32 * np.abs(o_ref)
    return B, o_tol


def gdn_reference_step(y, conv_w, hist, S, nh, dk, dv, K, B_prev=None):
    """One Gated DeltaNet step of a layer by the oracle, with the per-row
    bounds of gdn_step_bounds.  y: projection output (q|k|v|a|b) as FP64;
    conv_w: bf16 taps [CC][K]; hist: the oracle's conv history [K-1][CC];
    S: FP32 state [nh][dv][dk].  Returns (o, hist', S', B [nh][dv], o_tol [nh*dv])."""
    from oracle import oracle as orc
    from synth import gen
    CC = 2 * nh * dk + nh * dv
    y = np.asarray(y, dtype=np.float64)
    w = gen.bf16_bits_to_f32(conv_w).astype(np.float64)
    A = np.abs(w[:, K - 1]) * np.abs(y[:CC])
    for j in range(K - 1):
        A += np.abs(w[:, j]) * np.abs(hist[j])
    c, hist_new = orc.conv_step(y[:CC], hist, conv_w, K)
    o = np.zeros(nh * dv)
    S_new = np.array(S, dtype=np.float32, copy=True)
    B = np.zeros((nh, dv)) if B_prev is None else np.array(B_prev, dtype=np.float64)
    o_tol = np.zeros(nh * dv)
    for h in range(nh):
        qs, ks, vs = slice(h * dk, (h + 1) * dk), slice(nh * dk + h * dk, nh * dk + (h + 1) * dk), \
            slice(2 * nh * dk + h * dv, 2 * nh * dk + (h + 1) * dv)
        q = orc.l2norm(c[qs], 1e-6) / np.sqrt(dk)
        k = orc.l2norm(c[ks], 1e-6)
        v = c[vs]
        a = orc.lib().orc_sigmoid(float(y[CC + h]))
        b = orc.lib().orc_sigmoid(float(y[CC + nh + h]))
        o[h * dv:(h + 1) * dv], S_new[h] = orc.gdn_step(S[h], q, k, v, a, b)
        B[h], o_tol[h * dv:(h + 1) * dv] = gdn_step_bounds(S[h], q, k, v, a, b, A[qs], A[ks], A[vs], c[qs], c[ks],
                                                           S_new[h], o[h * dv:(h + 1) * dv], B[h], K)
    return o, hist_new, S_new, B, o_tol


def assert_gdn_rows(S_got, S_ref, B, what=""):
    """Every state row within GDN_SAFETY times its carried bound."""
    err = np.linalg.norm(np.asarray(S_got, dtype=np.float64) - np.asarray(S_ref, dtype=np.float64), axis=-1)
    tol = GDN_SAFETY * B + 1e-30
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (f"{what}: {len(bad)} state rows outside their bound; first (head, row) {bad[:4].tolist()}, "
                           f"worst err/tol {(err / tol).max():.3g}")
