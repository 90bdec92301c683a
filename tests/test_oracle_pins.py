"""Pins of the FP64 oracle against closed forms, invariants, special cases,
library routines and brute force (CPU only).

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong nibble order) fails it.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import oracle as orc
from synth import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def rand_bf16(shape, scale=1.0, rng=RNG):
    return gen.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def widen(bits):
    return gen.bf16_bits_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------ formats

def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_ieee_format_golden():
    for kind, expr, bits in _golden_lines("ieee_formats.txt"):
        value = float(eval(expr))  # arithmetic literals only
        if kind == "bf16":
            assert orc.to_bf16(value) == int(bits, 16), expr
        else:
            assert orc.fp16_to_double(int(bits, 16)) == value, expr


def test_bf16_widen_exact():
    b = np.arange(0, 65536, 97, dtype=np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]  # finite codes only
    for x in b[:400]:
        assert orc.bf16_to_double(int(x)) == float(gen.bf16_bits_to_f32(np.array([x]))[0])
        assert orc.to_bf16(orc.bf16_to_double(int(x))) == int(x)


def test_fp16_matches_numpy_all_finite():
    codes = np.arange(0, 65536, dtype=np.uint16)
    vals = codes.view(np.float16).astype(np.float64)
    fin = np.isfinite(vals)
    for c in codes[fin][::61]:
        assert orc.fp16_to_double(int(c)) == float(np.array([c], dtype=np.uint16).view(np.float16)[0])


# ------------------------------------------------------------ 4-bit blocks

def _q4_golden():
    d = {ln[0]: ln[1:] for ln in _golden_lines("q4_block.txt")}
    sc = int(d["scale_bits"][0], 16)
    qs = np.array([int(x, 16) for x in d["bytes"]], dtype=np.uint8)
    vals = np.array([float(x) for x in d["values"]])
    return qs, sc, vals


def test_q4_block_golden():
    qs, sc, vals = _q4_golden()
    w = (qs.reshape(1, 16), np.array([[sc]], dtype=np.uint16))
    np.testing.assert_array_equal(orc.mat_row(w, 0), vals)


def test_q4_every_nibble_round_trips_and_all_eight_is_zero():
    for pos in range(32):
        for nib in range(16):
            qs = np.full(16, 0x88, dtype=np.uint8)  # all elements 0
            b = pos % 16
            qs[b] = (qs[b] & 0xF0) | nib if pos < 16 else (qs[b] & 0x0F) | (nib << 4)
            row = orc.mat_row((qs.reshape(1, 16), np.array([[0x3C00]], dtype=np.uint16)), 0)
            expect = np.zeros(32)
            expect[pos] = nib - 8
            np.testing.assert_array_equal(row, expect)


def test_q4_scales_per_block_and_row():
    # two rows of two blocks each; each block all-nibble 9 (value +1) -> row entries equal the block scale
    qs = np.full((2, 32), 0x99, dtype=np.uint8)
    scales = np.array([[0x3C00, 0x4000], [0x3800, 0xC400]], dtype=np.uint16)  # 1, 2, 0.5, -4
    m = (qs, scales)
    np.testing.assert_array_equal(orc.mat_row(m, 0), np.r_[np.full(32, 1.0), np.full(32, 2.0)])
    np.testing.assert_array_equal(orc.mat_row(m, 1), np.r_[np.full(32, 0.5), np.full(32, -4.0)])


# ------------------------------------------------------------ GEMV

@pytest.mark.parametrize("rows,cols", [(1, 8), (7, 13), (33, 257), (64, 512)])
def test_gemv_equals_numpy_matmul(rows, cols):
    W = rand_bf16((rows, cols))
    x = RNG.standard_normal(cols)
    y = orc.gemv(W, x)
    ref = widen(W) @ x
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_gemv_q4_equals_numpy_on_widened_rows():
    rows, cols = 9, 96
    qs = RNG.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    sc = (RNG.uniform(0.5, 2.0, size=(rows, cols // 32)).astype(np.float16)).view(np.uint16)
    m = (qs, sc)
    dense = np.stack([orc.mat_row(m, r) for r in range(rows)])
    x = RNG.standard_normal(cols)
    np.testing.assert_allclose(orc.gemv(m, x), dense @ x, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ norms

def test_rmsnorm_constant_vector_gives_sign_times_gain():
    g = RNG.uniform(0.5, 2.0, 37).astype(np.float32)
    for c in (3.5, -0.25):
        y = orc.rmsnorm(np.full(37, c), g, 0.0)
        np.testing.assert_allclose(y, np.sign(c) * g.astype(np.float64), rtol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance():
    x = RNG.standard_normal(256)
    one = np.ones(256, dtype=np.float32)
    y = orc.rmsnorm(x, one, 0.0)
    assert abs(np.sqrt(np.mean(y * y)) - 1.0) < 1e-14
    np.testing.assert_allclose(orc.rmsnorm(7.0 * x, one, 0.0), y, rtol=1e-13)
    # eps keeps a zero vector finite
    assert np.all(orc.rmsnorm(np.zeros(8), one[:8], 1e-6) == 0.0)


def test_l2norm_unit_norm_and_direction():
    v = RNG.standard_normal(64)
    u = orc.l2norm(v, 0.0)
    assert abs(np.linalg.norm(u) - 1.0) < 1e-14
    np.testing.assert_allclose(u * np.linalg.norm(v), v, rtol=1e-13)


# ------------------------------------------------------------ RoPE

def test_rope_position_zero_is_identity():
    v = RNG.standard_normal(64)
    np.testing.assert_array_equal(orc.rope(v, 0), v)


def test_rope_preserves_norm_and_depends_on_relative_position():
    hd = 64
    q, k = RNG.standard_normal(hd), RNG.standard_normal(hd)
    for pos in (1, 17, 4096):
        assert abs(np.linalg.norm(orc.rope(q, pos)) - np.linalg.norm(q)) < 1e-12
    s1 = orc.rope(q, 30) @ orc.rope(k, 11)
    s2 = orc.rope(q, 30 + 977) @ orc.rope(k, 11 + 977)
    assert abs(s1 - s2) < 1e-10


def test_rope_pairs_half_apart_with_geometric_frequencies():
    # hd = 4: pair (0, 2) turns by pos * 1 rad, pair (1, 3) by pos * theta^(-1/2) rad
    hd, theta, pos = 4, 1e4, 3
    v = np.array([1.0, 2.0, 3.0, 4.0])
    r = orc.rope(v, pos, theta)
    ang02 = math.atan2(r[2], r[0]) - math.atan2(v[2], v[0])
    ang13 = math.atan2(r[3], r[1]) - math.atan2(v[3], v[1])
    assert abs(math.remainder(ang02 - pos * 1.0, 2 * math.pi)) < 1e-12
    assert abs(math.remainder(ang13 - pos * theta ** -0.5, 2 * math.pi)) < 1e-12
    # each pair keeps its own length (no mixing across pairs)
    assert abs(math.hypot(r[0], r[2]) - math.hypot(1, 3)) < 1e-12
    assert abs(math.hypot(r[1], r[3]) - math.hypot(2, 4)) < 1e-12


# ------------------------------------------------------------ causal conv

def _silu(x):
    return x * scipy.special.expit(x)


def test_conv_one_hot_taps_delay_the_input():
    C, K, T = 5, 4, 9
    seq = RNG.standard_normal((T, C))
    for tap in range(K):
        w = np.zeros((C, K), dtype=np.float32)
        w[:, tap] = 1.0
        wb = gen.f32_to_bf16_bits(w)
        st = np.zeros((K - 1, C))
        for t in range(T):
            out, st = orc.conv_step(seq[t], st, wb, K)
            src = t - (K - 1) + tap
            expect = _silu(seq[src]) if src >= 0 else np.zeros(C)  # zeros before t = 0
            np.testing.assert_allclose(out, expect, rtol=1e-14, atol=1e-15)


def test_conv_is_linear_in_taps_before_silu():
    C, K = 3, 4
    w = rand_bf16((C, K), 0.3)
    hist = RNG.standard_normal((K - 1, C))
    u = RNG.standard_normal(C)
    out, st = orc.conv_step(u, hist, w, K)
    pre = (widen(w)[:, :K - 1] * hist.T).sum(1) + widen(w)[:, K - 1] * u
    # silu is invertible on the sampled range via its monotone branch check
    np.testing.assert_allclose(out, _silu(pre), rtol=1e-13)
    np.testing.assert_array_equal(st[:-1], hist[1:])
    np.testing.assert_array_equal(st[-1], u)


# ------------------------------------------------------------ gated delta rule

def test_gdn_alpha1_beta0_leaves_state_unchanged():
    S = RNG.standard_normal((6, 4)).astype(np.float32)
    q, k, v = RNG.standard_normal(4), RNG.standard_normal(4), RNG.standard_normal(6)
    o, S2 = orc.gdn_step(S, q, k, v, 1.0, 0.0)
    np.testing.assert_array_equal(S2, S)
    np.testing.assert_allclose(o, S.astype(np.float64) @ q, rtol=1e-12)


def test_gdn_alpha0_beta1_writes_outer_product_non_square():
    # dv = 3, dk = 5: a transposed state or a swapped k/v would not even match shapes
    S = RNG.standard_normal((3, 5)).astype(np.float32)
    q, k, v = RNG.standard_normal(5), RNG.standard_normal(5), RNG.standard_normal(3)
    o, S2 = orc.gdn_step(S, q, k, v, 0.0, 1.0)
    np.testing.assert_allclose(S2, np.outer(v, k).astype(np.float32), rtol=1e-6)
    np.testing.assert_allclose(o, S2.astype(np.float64) @ q, rtol=1e-12)


def test_gdn_pure_decay():
    S = RNG.standard_normal((4, 4)).astype(np.float32)
    _, S2 = orc.gdn_step(S, np.zeros(4), np.ones(4) / 2, np.zeros(4), 0.25, 0.0)
    np.testing.assert_allclose(S2, 0.25 * S, rtol=1e-7)


def test_gdn_delta_rule_writes_value_at_unit_key():
    dk, dv = 16, 8
    S = RNG.standard_normal((dv, dk)).astype(np.float32)
    k = orc.l2norm(RNG.standard_normal(dk), 0.0)
    v = RNG.standard_normal(dv)
    _, S2 = orc.gdn_step(S, np.zeros(dk), k, v, 1.0, 1.0)
    np.testing.assert_allclose(S2.astype(np.float64) @ k, v, rtol=1e-5, atol=1e-5)


def test_gdn_associative_memory_over_orthonormal_keys():
    dk, dv = 8, 5
    Q, _ = np.linalg.qr(RNG.standard_normal((dk, dk)))
    vals = RNG.standard_normal((dk, dv))
    S = np.zeros((dv, dk), dtype=np.float32)
    for j in range(dk):
        _, S = orc.gdn_step(S, np.zeros(dk), Q[:, j], vals[j], 1.0, 1.0)
    for j in range(dk):
        np.testing.assert_allclose(S.astype(np.float64) @ Q[:, j], vals[j], atol=1e-5)


def test_gdn_partial_beta_interpolates_old_and_new():
    # alpha = 1, unit k: S'k = (1 - beta) S k + beta v
    dk, dv = 6, 4
    S = RNG.standard_normal((dv, dk)).astype(np.float32)
    k = orc.l2norm(RNG.standard_normal(dk), 0.0)
    v = RNG.standard_normal(dv)
    beta = 0.3
    _, S2 = orc.gdn_step(S, np.zeros(dk), k, v, 1.0, beta)
    np.testing.assert_allclose(S2.astype(np.float64) @ k, (1 - beta) * (S.astype(np.float64) @ k) + beta * v,
                               atol=1e-5)


# ------------------------------------------------------------ attention

def _kv(nkv, cap, hd, rng=RNG):
    return rand_bf16((nkv, cap, hd), 1.0, rng), rand_bf16((nkv, cap, hd), 1.0, rng)


def test_attention_single_position_returns_value_row():
    q = RNG.standard_normal((4, 32))
    K, V = _kv(2, 5, 32)
    o = orc.attention(q, K, V, 1)
    for j in range(4):
        np.testing.assert_allclose(o[j], widen(V[j // 2, 0]), rtol=1e-15)


def test_attention_equal_keys_average_values_per_kv_group():
    nq, nkv, hd, T = 6, 3, 16, 11
    K, V = _kv(nkv, T, hd)
    K[:] = K[:, :1, :]  # every position has the same key per group
    q = RNG.standard_normal((nq, hd))
    o = orc.attention(q, K, V, T)
    for j in range(nq):
        np.testing.assert_allclose(o[j], widen(V[j // 2]).mean(0), rtol=1e-12)


def test_attention_matches_library_softmax_bruteforce():
    nq, nkv, hd, cap, T = 4, 2, 8, 12, 9
    K, V = _kv(nkv, cap, hd)
    q = RNG.standard_normal((nq, hd))
    o = orc.attention(q, K, V, T)
    for j in range(nq):
        g = j // (nq // nkv)
        s = widen(K[g, :T]) @ q[j] / math.sqrt(hd)
        np.testing.assert_allclose(o[j], scipy.special.softmax(s) @ widen(V[g, :T]), rtol=1e-12)


@pytest.mark.parametrize("nsplit", [1, 2, 3, 4, 8, 16])
def test_split_lse_combine_equals_single_pass(nsplit):
    nq, nkv, hd = 4, 2, 16
    for T in sorted({1, max(nsplit - 1, 1), nsplit, nsplit + 1, 1000}):
        K, V = _kv(nkv, 1000, hd)
        q = RNG.standard_normal((nq, hd)) * 2.0
        np.testing.assert_allclose(orc.attention(q, K, V, T, nsplit), orc.attention(q, K, V, T), rtol=1e-12,
                                   atol=1e-14)


# ------------------------------------------------------------ argmax / top-k / softmax

def test_argmax_lowest_index_on_ties_and_fp32_decision():
    v = np.array([0.5, 2.0, -1.0, 2.0, 1.0])
    assert orc.argmax(v) == 1
    # differ only below FP32 resolution: decided as a tie -> lowest index
    w = np.array([1.0, 1.0 + 1e-12, 0.0])
    assert orc.argmax(w) == 0
    r = RNG.standard_normal(100_003)
    assert orc.argmax(r) == int(np.argmax(r.astype(np.float32)))


def test_topk_equals_full_stable_sort():
    rng = np.random.default_rng(7)
    for trial in range(2000):
        n, k = 256, 8
        if trial % 3 == 0:
            r = rng.integers(-6, 6, n).astype(np.float64)  # many ties
        else:
            r = rng.standard_normal(n)
        ids = orc.topk(r, k)
        order = np.lexsort((np.arange(n), -r.astype(np.float32)))  # descending value, ascending index
        np.testing.assert_array_equal(ids, order[:k])


def test_softmax_over_selected_equals_renormalised_full_softmax():
    r = RNG.standard_normal(256) * 0.9
    ids = orc.topk(r, 8)
    p_sel = orc.softmax(r[ids])
    full = scipy.special.softmax(r)
    np.testing.assert_allclose(p_sel, full[ids] / full[ids].sum(), rtol=1e-13)
    np.testing.assert_allclose(orc.softmax(r), full, rtol=1e-13)


# ------------------------------------------------------------------ int8 KV cache
# One cached vector -> int8 codes and one FP32 scale ("hanzo-engine...",
# "System Architecture": int8 KV with one f32 scale per vector).

def test_int8_quant_worked_example():
    """amax 1: scale 1/127; -0.5 * 127 = -63.5 is a tie and goes to the even
    -64; 0.25 * 127 = 31.75 rounds to 32."""
    q, s = orc.quant_i8([1.0, -0.5, 0.25, 0.0])
    np.testing.assert_array_equal(q, [127, -64, 32, 0])
    assert s == float(np.float32(1.0) / np.float32(127.0))


def test_int8_quant_invariants():
    rng = np.random.default_rng(12)
    for n in (1, 7, 64, 128, 256):
        x = rng.standard_normal(n) * rng.uniform(1e-3, 30)
        q, s = orc.quant_i8(x)
        i = int(np.argmax(np.abs(x)))
        assert abs(int(q[i])) == 127 and np.sign(q[i]) == np.sign(x[i])
        assert np.all(np.abs(q.astype(np.int32)) <= 127)
        # every element within half a step of its code (plus the FP32 rounding of the inputs)
        assert np.all(np.abs(x - q.astype(np.float64) * s) <= s * (0.5 + 1e-5) + 1e-6 * np.abs(x))
        qn, sn = orc.quant_i8(-x)
        np.testing.assert_array_equal(qn, -q)
        assert sn == s
    q, s = orc.quant_i8(np.zeros(16))
    assert s == 0.0 and not q.any()


def test_int8_attention_equals_bf16_attention_on_exact_values():
    """Codes with scale 2^-7 give values code / 128, exact in bf16: the int8
    attention then equals the bf16 one."""
    rng = np.random.default_rng(3)
    nq, nkv, hd, cap, npos = 4, 2, 16, 9, 7
    Kq = rng.integers(-127, 128, (nkv, cap, hd)).astype(np.int8)
    Vq = rng.integers(-127, 128, (nkv, cap, hd)).astype(np.int8)
    Ks = np.full((nkv, cap), 2.0 ** -7, dtype=np.float32)
    Vs = np.full((nkv, cap), 2.0 ** -7, dtype=np.float32)
    q = rng.standard_normal((nq, hd))
    Kb = gen.f32_to_bf16_bits((Kq.astype(np.float32) / 128.0))
    Vb = gen.f32_to_bf16_bits((Vq.astype(np.float32) / 128.0))
    np.testing.assert_allclose(orc.attention_i8(q, Kq, Ks, Vq, Vs, npos), orc.attention(q, Kb, Vb, npos),
                               rtol=1e-12, atol=1e-14)


def test_int8_attention_brute_force():
    rng = np.random.default_rng(4)
    nq, nkv, hd, cap, npos = 6, 3, 8, 6, 5
    Kq = rng.integers(-127, 128, (nkv, cap, hd)).astype(np.int8)
    Vq = rng.integers(-127, 128, (nkv, cap, hd)).astype(np.int8)
    Ks = rng.uniform(0.001, 0.02, (nkv, cap)).astype(np.float32)
    Vs = rng.uniform(0.001, 0.02, (nkv, cap)).astype(np.float32)
    q = rng.standard_normal((nq, hd))
    got = orc.attention_i8(q, Kq, Ks, Vq, Vs, npos)
    for j in range(nq):
        g = j // (nq // nkv)
        K = Kq[g, :npos].astype(np.float64) * Ks[g, :npos, None]
        V = Vq[g, :npos].astype(np.float64) * Vs[g, :npos, None]
        sc = K @ q[j] / np.sqrt(hd)
        p = np.exp(sc - sc.max())
        np.testing.assert_allclose(got[j], (p / p.sum()) @ V, rtol=1e-12, atol=1e-14)
