"""The element-wise bounds the GPU parity tests use, checked on the CPU
before they are trusted: an independent FP32 evaluation of the same step
(numpy float32, another summation order) stays inside them, and a plausible
kernel mistake confined to one head, one dimension or one state row falls
outside them.  So the bounds are neither so loose that a local fault hides
nor so tight that correct FP32 arithmetic fails."""
import numpy as np
import pytest

from oracle import oracle as orc
from synth import gen
from tests.gpu_util import (ATTN_SAFETY, GDN_SAFETY, assert_elementwise, assert_gdn_rows, attention_tolerance,
                            gdn_reference_step)

F = np.float32


# ------------------------------------------------------------------ attention

def attention_fp32(yq, K, V, T, nsplit, theta=1e4, tile=64, wrong_kv_head=None, drop_split=None, drop_pos=None,
                   rope_pos=None):
    """FP32 split-KV attention with an online softmax per tile (numpy)."""
    nq, hd = yq.shape
    nkv = K.shape[0]
    G = nq // nkv
    half = hd // 2
    ang = (T if rope_pos is None else rope_pos) * theta ** (-2.0 * np.arange(half) / hd)
    cs, sn = np.cos(ang).astype(F), np.sin(ang).astype(F)
    scale = F(1.0 / np.sqrt(hd))
    a, b = yq[:, :half].astype(F), yq[:, half:].astype(F)
    q = np.concatenate([(a * cs - b * sn) * scale, (b * cs + a * sn) * scale], axis=1).astype(F)
    L = T + 1
    o = np.zeros((nq, hd), dtype=F)
    for j in range(nq):
        g = j // G
        if wrong_kv_head is not None and j == wrong_kv_head:
            g = (g + 1) % nkv
        Kg, Vg = K[g, :L].astype(F), V[g, :L].astype(F)
        ms, ls, os_ = [], [], []
        for s in range(nsplit):
            p0, p1 = s * L // nsplit, (s + 1) * L // nsplit
            m, l, acc = F(-np.inf), F(0), np.zeros(hd, dtype=F)
            for t0 in range(p0, p1, tile):
                t1 = min(p1, t0 + tile)
                sc = (Kg[t0:t1] @ q[j]).astype(F)
                if drop_pos is not None and t0 <= drop_pos < t1:
                    sc[drop_pos - t0] = -np.inf
                mn = max(m, sc.max())
                e = np.exp((sc - mn).astype(F)).astype(F)
                corr = F(np.exp(F(m - mn))) if m != -np.inf else F(0)
                l = F(l * corr + e.sum(dtype=F))
                acc = (acc * corr + e @ Vg[t0:t1]).astype(F)
                m = mn
            if drop_split is not None and s == drop_split:
                continue
            ms.append(m)
            ls.append(l)
            os_.append(acc)
        M = max(ms)
        w = [F(np.exp(F(mi - M))) if li > 0 else F(0) for mi, li in zip(ms, ls)]
        den = sum(F(wi * li) for wi, li in zip(w, ls))
        o[j] = sum(wi * oi for wi, oi in zip(w, os_)) / den
    return o


def attention_case(nq, nkv, hd, T, seed):
    rng = np.random.default_rng(seed)
    K = gen.f32_to_bf16_bits(rng.uniform(-1, 1, (nkv, T + 1, hd)).astype(np.float32))
    V = gen.f32_to_bf16_bits(rng.uniform(-1, 1, (nkv, T + 1, hd)).astype(np.float32))
    y = rng.standard_normal((nq + 2 * nkv) * hd).astype(np.float32)
    yq = y[:nq * hd].reshape(nq, hd)
    q = np.stack([orc.rope(yq[j].astype(np.float64), T) for j in range(nq)])
    Kw, Vw = gen.bf16_bits_to_f32(K), gen.bf16_bits_to_f32(V)
    ref = orc.attention(q, K, V, T + 1)
    return yq, q, K, V, Kw, Vw, ref


@pytest.mark.parametrize("nq,nkv,hd,T,nsplit", [(4, 2, 64, 0, 1), (4, 2, 64, 200, 3), (16, 4, 128, 700, 16),
                                                 (16, 2, 256, 300, 8)])
def test_attention_bound_admits_fp32_and_catches_local_faults(nq, nkv, hd, T, nsplit):
    yq, q, K, V, Kw, Vw, ref = attention_case(nq, nkv, hd, T, seed=T + hd)
    tol = attention_tolerance(yq, q, Kw, Vw, T + 1, ref, nsplit)
    got = attention_fp32(yq, Kw, Vw, T, nsplit)
    assert_elementwise(got, ref, tol, "FP32 evaluation")
    # the bound has room for FP32 arithmetic, but not for much more than its safety factor
    assert np.max(np.abs(got - ref) / tol) < 1.0
    # one query head reading the next kv head
    if nkv > 1:
        bad = attention_fp32(yq, Kw, Vw, T, nsplit, wrong_kv_head=nq - 1)
        with pytest.raises(AssertionError):
            assert_elementwise(bad, ref, tol)
    # one split left out of the combine
    if T + 1 >= 2 * nsplit and nsplit > 1:
        bad = attention_fp32(yq, Kw, Vw, T, nsplit, drop_split=nsplit - 1)
        with pytest.raises(AssertionError):
            assert_elementwise(bad, ref, tol)
    if T > 0:
        # the first position of the last split left out (an off-by-one at a split boundary)
        bad = attention_fp32(yq, Kw, Vw, T, nsplit, drop_pos=(nsplit - 1) * (T + 1) // nsplit)
        with pytest.raises(AssertionError):
            assert_elementwise(bad, ref, tol)
        # the query rotated for the previous position
        bad = attention_fp32(yq, Kw, Vw, T, nsplit, rope_pos=T - 1)
        with pytest.raises(AssertionError):
            assert_elementwise(bad, ref, tol)


# ------------------------------------------------------------------ Gated DeltaNet

def gdn_fp32_step(y, conv_w, ring, S, t, nh, dk, dv, K, stale_row=None):
    """FP32 decode step (numpy float32): conv over the ring, SiLU, L2 norms,
    gates, rank-1 update in place, outputs."""
    CC = 2 * nh * dk + nh * dv
    w = gen.bf16_bits_to_f32(conv_w).astype(F)
    acc = np.zeros(CC, dtype=F)
    for j in range(K - 1):
        acc = (acc + w[:, j] * ring[(t - (K - 1) + j) % K]).astype(F)
    acc = (acc + w[:, K - 1] * y[:CC].astype(F)).astype(F)
    ring[t % K] = y[:CC]
    c = (acc / (F(1) + np.exp(-acc))).astype(F)
    o = np.zeros(nh * dv, dtype=F)
    for h in range(nh):
        q = c[h * dk:(h + 1) * dk]
        k = c[nh * dk + h * dk:nh * dk + (h + 1) * dk]
        v = c[2 * nh * dk + h * dv:2 * nh * dk + (h + 1) * dv]
        qs = F(1) / (np.sqrt(F(np.dot(q, q)) + F(1e-6)) * np.sqrt(F(dk)))
        ks = F(1) / np.sqrt(F(np.dot(k, k)) + F(1e-6))
        kq, qq = (k * ks).astype(F), (q * qs).astype(F)
        a = F(1) / (F(1) + np.exp(-F(y[CC + h])))
        b = F(1) / (F(1) + np.exp(-F(y[CC + nh + h])))
        u = (S[h] @ kq).astype(F)
        d = (b * (v - a * u)).astype(F)
        Sn = (a * S[h] + d[:, None] * kq[None, :]).astype(F)
        if stale_row is not None and h == stale_row[0]:
            Sn[stale_row[1]] = S[h][stale_row[1]]
        S[h] = Sn
        o[h * dv:(h + 1) * dv] = S[h] @ qq
    return o


@pytest.mark.parametrize("nh,dk,dv,steps", [(4, 64, 64, 10), (16, 128, 128, 5), (2, 256, 40, 6)])
def test_gdn_bounds_admit_fp32_and_catch_a_stale_row(nh, dk, dv, steps):
    K = 4
    CC = 2 * nh * dk + nh * dv
    rng = np.random.default_rng(nh * dk + dv)
    conv_w = gen.f32_to_bf16_bits((rng.standard_normal((CC, K)) * 0.5).astype(np.float32))
    ring = np.zeros((K, CC), dtype=F)
    S32 = np.zeros((nh, dv, dk), dtype=F)
    hist = np.zeros((K - 1, CC))
    S_ref = np.zeros((nh, dv, dk), dtype=np.float32)
    B = None
    worst = 0.0
    for t in range(steps):
        y = rng.standard_normal(CC + 2 * nh).astype(np.float32)
        o32 = gdn_fp32_step(y, conv_w, ring, S32, t, nh, dk, dv, K)
        o_ref, hist, S_ref, B, o_tol = gdn_reference_step(y.astype(np.float64), conv_w, hist, S_ref, nh, dk, dv, K, B)
        assert_gdn_rows(S32, S_ref, B, f"step {t}")
        assert_elementwise(o32, o_ref, GDN_SAFETY * o_tol, f"step {t} outputs")
        err = np.linalg.norm(S32.astype(np.float64) - S_ref, axis=-1)
        worst = max(worst, float((err / (GDN_SAFETY * B + 1e-30)).max()))
    assert worst < 1.0
    # one state row left stale in the next step
    S_bad = S32.copy()
    ring_bad = ring.copy()
    y = rng.standard_normal(CC + 2 * nh).astype(np.float32)
    gdn_fp32_step(y, conv_w, ring_bad, S_bad, steps, nh, dk, dv, K, stale_row=(nh - 1, dv // 2))
    _, _, S_ref2, B2, _ = gdn_reference_step(y.astype(np.float64), conv_w, hist, S_ref, nh, dk, dv, K, B)
    with pytest.raises(AssertionError):
        assert_gdn_rows(S_bad, S_ref2, B2)
