"""Parity of each decode-step kernel, called through the C ABI, against the
FP64 oracle on seeded inputs: ragged and tiled shapes, the configurations'
full sizes (sampled rows where the full output is large), and edge cases."""
import ctypes

import numpy as np
import pytest

from oracle import oracle as orc
from synth import gen
from tests.gpu_util import (GDN_SAFETY, assert_dot_close, assert_elementwise, assert_gdn_rows, attention_tolerance,
                            bf16_bits, bf16_tensor, bf16_tie_mask, gdn_reference_step, rope_pair_abs, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L(gpu):
    from bandwidth_bound_hybrid_gb300 import build, capi
    build.build()
    return capi.lib()


def _torch():
    import torch
    return torch


def stream():
    return _torch().cuda.current_stream().cuda_stream


def rand_bf16(rng, shape, scale=0.02):
    return gen.f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def widen(bits):
    return gen.bf16_bits_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ GEMV

GEMV_SHAPES = [(1, 8), (7, 24), (100, 256), (33, 520), (777, 2560), (2560, 2048), (2560, 9216), (6176, 2560),
               (5120, 2048), (257, 2048), (2048, 4096)]


@pytest.mark.parametrize("R,C", GEMV_SHAPES)
@pytest.mark.parametrize("norm", [False, True])
def test_gemv_parity(L, R, C, norm):
    torch = _torch()
    rng = np.random.default_rng(R * 7919 + C)
    W = rand_bf16(rng, (R, C))
    x = rng.standard_normal(C).astype(np.float32)
    g = rng.uniform(0.5, 1.5, C).astype(np.float32)
    y = torch.full((R,), 7.0, dtype=torch.float32, device="cuda")
    Wd, xd, gd = bf16_tensor(W), torch.from_numpy(x).cuda(), torch.from_numpy(g).cuda()  # held until synchronised
    rc = L.hy_op_gemv(Wd.data_ptr(), R, C, xd.data_ptr(), gd.data_ptr() if norm else None, 1e-6, y.data_ptr(), 0,
                      stream())
    assert rc == 0
    torch.cuda.synchronize()
    xn = orc.rmsnorm(x, g, 1e-6) if norm else x.astype(np.float64)
    ref = orc.gemv(W, xn)
    absdot = np.abs(widen(W)) @ np.abs(xn)
    assert_dot_close(to_np(y), ref, absdot, C + 64, f"gemv {R}x{C}")


def test_gemv_accumulate_adds_to_output(L):
    torch = _torch()
    rng = np.random.default_rng(5)
    R, C = 300, 2560
    W = rand_bf16(rng, (R, C))
    x = rng.standard_normal(C).astype(np.float32)
    y0 = rng.standard_normal(R).astype(np.float32)
    y = torch.from_numpy(y0.copy()).cuda()
    Wd, xd = bf16_tensor(W), torch.from_numpy(x).cuda()
    assert L.hy_op_gemv(Wd.data_ptr(), R, C, xd.data_ptr(), None, 0.0, y.data_ptr(), 1, stream()) == 0
    torch.cuda.synchronize()
    ref = y0.astype(np.float64) + orc.gemv(W, x)
    assert_dot_close(to_np(y), ref, np.abs(widen(W)) @ np.abs(x) + np.abs(y0), C + 64, "gemv accumulate")


def test_gemv_full_lm_head_sampled_rows(L):
    torch = _torch()
    from synth import device, workloads
    R, C = 151936, 2560
    W = torch.empty((R, C), dtype=torch.bfloat16, device="cuda")
    device.fill_normal_bf16(W, 0, workloads.GLOBAL_TID["lm_head"])
    rng = np.random.default_rng(11)
    x = rng.standard_normal(C).astype(np.float32)
    y = torch.empty(R, dtype=torch.float32, device="cuda")
    xd = torch.from_numpy(x).cuda()
    assert L.hy_op_gemv(W.data_ptr(), R, C, xd.data_ptr(), None, 0.0, y.data_ptr(), 0, stream()) == 0
    torch.cuda.synchronize()
    rows = np.unique(np.r_[0, 1, R - 1, rng.integers(0, R, 600)])
    Wh = bf16_bits(W[torch.from_numpy(rows).cuda()])
    # the generator's device copy must equal its host copy on these rows
    from synth import host
    for r in rows[:8]:
        np.testing.assert_array_equal(Wh[list(rows).index(r)], host.normal_bf16(0, workloads.GLOBAL_TID["lm_head"], C,
                                                                                start=int(r) * C))
    ref = orc.gemv(Wh, x)
    assert_dot_close(to_np(y)[rows], ref, np.abs(widen(Wh)) @ np.abs(x), C + 64, "lm head rows")


@pytest.mark.parametrize("R,C", [(512, 256), (9216, 2560), (1000, 2048), (3, 8)])
def test_gemv_swiglu_parity(L, R, C):
    torch = _torch()
    rng = np.random.default_rng(R + C)
    Wg, Wu = rand_bf16(rng, (R, C)), rand_bf16(rng, (R, C))
    x = rng.standard_normal(C).astype(np.float32)
    g = np.ones(C, dtype=np.float32)
    h = torch.empty(R, dtype=torch.float32, device="cuda")
    Wgd, Wud, xd, gd = bf16_tensor(Wg), bf16_tensor(Wu), torch.from_numpy(x).cuda(), torch.from_numpy(g).cuda()
    assert L.hy_op_gemv_swiglu(Wgd.data_ptr(), Wud.data_ptr(), R, C, xd.data_ptr(), gd.data_ptr(), 1e-6,
                               h.data_ptr(), stream()) == 0
    torch.cuda.synchronize()
    xn = orc.rmsnorm(x, g, 1e-6)
    a, b = orc.gemv(Wg, xn), orc.gemv(Wu, xn)
    ref = np.array([orc.lib().orc_silu(float(v)) for v in a]) * b
    # error of silu(a)*b from the two dot products: |d silu| <= 1.1, plus the activation's few ulps
    absd_a = np.abs(widen(Wg)) @ np.abs(xn)
    absd_b = np.abs(widen(Wu)) @ np.abs(xn)
    from tests.gpu_util import gamma
    tol = 1.1 * gamma(C + 64) * absd_a * np.abs(b) + gamma(C + 64) * absd_b * np.abs(a) + 64 * 2.0 ** -24 * (
        np.abs(ref) + 1e-30)
    assert np.all(np.abs(to_np(h) - ref) <= tol)


@pytest.mark.parametrize("R,C", [(1, 8), (1000, 256), (151936, 2560)])
def test_gemv_argmax(L, R, C):
    torch = _torch()
    rng = np.random.default_rng(R)
    W = rand_bf16(rng, (R, C))
    x = rng.standard_normal(C).astype(np.float32)
    ws = torch.zeros(L.hy_op_argmax_workspace(), dtype=torch.uint8, device="cuda")
    logits = torch.empty(R, dtype=torch.float32, device="cuda")
    out = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    Wd, xd = bf16_tensor(W), torch.from_numpy(x).cuda()
    for _ in range(2):  # twice: the workspace must come back zeroed
        assert L.hy_op_gemv_argmax(Wd.data_ptr(), R, C, xd.data_ptr(), None, 0.0, logits.data_ptr(), out.data_ptr(),
                                   ws.data_ptr(), stream()) == 0
        torch.cuda.synchronize()
        gl = to_np(logits)
        assert int(out.item()) == int(np.argmax(gl.astype(np.float32)))  # the kernel's own logits
        assert int(ws[:4].view(torch.int32).item()) == 0
    ref = orc.gemv(W, x)
    top = int(orc.argmax(ref))
    srt = np.sort(ref)
    if R > 1 and srt[-1] - srt[-2] > 1e-3:
        assert int(out.item()) == top


def test_argmax_ties_pick_lowest_index(L):
    torch = _torch()
    rng = np.random.default_rng(3)
    R, C = 4000, 256
    W = rand_bf16(rng, (R, C))
    x = rng.standard_normal(C).astype(np.float32)
    best = int(np.argmax(orc.gemv(W, x)))
    # copy the best row to two later rows and one earlier row in other CTAs: the earliest copy must win
    dup = [3990, 2500, 17]
    for r in dup:
        W[r] = W[best]
    ws = torch.zeros(L.hy_op_argmax_workspace(), dtype=torch.uint8, device="cuda")
    out = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    Wd, xd = bf16_tensor(W), torch.from_numpy(x).cuda()
    assert L.hy_op_gemv_argmax(Wd.data_ptr(), R, C, xd.data_ptr(), None, 0.0, None, out.data_ptr(), ws.data_ptr(),
                               stream()) == 0
    torch.cuda.synchronize()
    assert int(out.item()) == min(dup + [best])


# ------------------------------------------------------------------ Gated DeltaNet

@pytest.mark.parametrize("nh,dk,dv,steps", [(4, 64, 64, 12), (16, 128, 128, 9), (2, 256, 40, 7), (3, 128, 16, 5)])
def test_gdn_step_sequence(L, nh, dk, dv, steps):
    """Consecutive steps of one layer: after every step each state row is
    within its carried per-row bound and each output element within its own
    bound (tests/gpu_util.py, derivation there)."""
    torch = _torch()
    K = 4
    CC = 2 * nh * dk + nh * dv
    rng = np.random.default_rng(nh * dk + dv)
    conv_w = gen.f32_to_bf16_bits((rng.standard_normal((CC, K)) * 0.5).astype(np.float32))
    cw = bf16_tensor(conv_w)
    ring = torch.zeros((K, CC), dtype=torch.float32, device="cuda")
    S = torch.zeros((nh, dv, dk), dtype=torch.float32, device="cuda")
    o = torch.empty(nh * dv, dtype=torch.float32, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist = np.zeros((K - 1, CC))
    S_ref = np.zeros((nh, dv, dk), dtype=np.float32)
    B = None
    for t in range(steps):
        y = rng.standard_normal(CC + 2 * nh).astype(np.float32)
        pos.fill_(t)
        yd = torch.from_numpy(y).cuda()
        assert L.hy_op_gdn_step(yd.data_ptr(), cw.data_ptr(), ring.data_ptr(), S.data_ptr(), o.data_ptr(), nh, dk,
                                dv, K, pos.data_ptr(), stream()) == 0
        torch.cuda.synchronize()
        o_ref, hist, S_ref, B, o_tol = gdn_reference_step(y.astype(np.float64), conv_w, hist, S_ref, nh, dk, dv, K, B)
        assert_gdn_rows(to_np(S), S_ref, B, f"step {t}")
        assert_elementwise(to_np(o), o_ref, GDN_SAFETY * o_tol, f"step {t} outputs")


def test_gdn_state_stays_in_place_other_heads_untouched(L):
    """The kernel writes only the state rows of the layer it is given."""
    torch = _torch()
    nh, dk, dv, K = 2, 64, 32, 4
    CC = 2 * nh * dk + nh * dv
    big = torch.full((3, nh, dv, dk), 5.0, dtype=torch.float32, device="cuda")
    S = big[1]
    ring = torch.zeros((K, CC), dtype=torch.float32, device="cuda")
    o = torch.empty(nh * dv, dtype=torch.float32, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.randn(CC + 2 * nh, device="cuda")
    cw = torch.zeros((CC, K), dtype=torch.bfloat16, device="cuda")
    assert L.hy_op_gdn_step(y.data_ptr(), cw.data_ptr(), ring.data_ptr(), S.data_ptr(), o.data_ptr(), nh, dk, dv, K,
                            pos.data_ptr(), stream()) == 0
    torch.cuda.synchronize()
    assert torch.all(big[0] == 5.0) and torch.all(big[2] == 5.0)
    assert not torch.all(big[1] == 5.0)


# ------------------------------------------------------------------ attention

def run_attention(L, rng, nq, nkv, hd, cap, T, nsplit):
    torch = _torch()
    Kc = rand_bf16(rng, (nkv, cap, hd), 1.0)
    Vc = rand_bf16(rng, (nkv, cap, hd), 1.0)
    y = rng.standard_normal((nq + 2 * nkv) * hd).astype(np.float32)
    Kd, Vd = bf16_tensor(Kc), bf16_tensor(Vc)
    table = torch.empty((cap, hd // 2, 2), dtype=torch.float32, device="cuda")
    assert L.hy_op_rope_table(table.data_ptr(), cap, hd, 1e4, stream()) == 0
    ln = torch.tensor([T], dtype=torch.int32, device="cuda")
    o = torch.empty(nq * hd, dtype=torch.float32, device="cuda")
    ws = torch.zeros(L.hy_op_attention_workspace(nq, nkv, hd, nsplit), dtype=torch.uint8, device="cuda")
    yd = torch.from_numpy(y).cuda()
    assert L.hy_op_attention(yd.data_ptr(), Kd.data_ptr(), Vd.data_ptr(), cap, nq, nkv, hd, ln.data_ptr(),
                             table.data_ptr(), nsplit, o.data_ptr(), ws.data_ptr(), stream()) == 0
    torch.cuda.synchronize()
    ref, Kr, Vr, tol = attention_reference(y, Kc, Vc, nq, nkv, hd, T, nsplit)
    return to_np(o).reshape(nq, hd), ref, bf16_bits(Kd), bf16_bits(Vd), Kr, Vr, ws, tol


def attention_reference(y, Kc, Vc, nq, nkv, hd, T, nsplit):
    """The oracle's attention at position T (rotate, append the bf16 k/v row,
    single-pass softmax over [0, T]) and the element-wise bound of the kernel's
    result (nsplit 0: the automatic count, at most 32)."""
    yd = y.astype(np.float64)
    q = np.stack([orc.rope(yd[j * hd:(j + 1) * hd], T) for j in range(nq)])
    Kr, Vr = Kc.copy(), Vc.copy()
    k_rot = np.zeros((nkv, hd))
    for g in range(nkv):
        kpre = yd[(nq + g) * hd:(nq + g + 1) * hd]
        k_rot[g] = orc.rope(kpre, T)
        v = yd[(nq + nkv + g) * hd:(nq + nkv + g + 1) * hd]
        Kr[g, T] = [orc.to_bf16(e) for e in k_rot[g]]
        Vr[g, T] = [orc.to_bf16(e) for e in v]
    ref = orc.attention(q, Kr, Vr, T + 1)
    kpre = yd[nq * hd:(nq + nkv) * hd].reshape(nkv, hd)
    k_flip = bf16_tie_mask(k_rot, 8 * 2.0 ** -24 * rope_pair_abs(kpre))
    tol = attention_tolerance(y[:nq * hd].reshape(nq, hd), q, widen(Kr), widen(Vr), T + 1, ref,
                              nsplit if nsplit > 0 else 32, k_flip=k_flip)
    return ref, Kr, Vr, tol


ATTN_CASES = [(4, 2, 64, 0), (4, 2, 64, 1), (4, 2, 64, 127), (4, 2, 64, 128), (4, 2, 64, 129),
              (16, 4, 128, 5), (16, 4, 128, 63), (16, 4, 128, 64), (16, 4, 128, 65), (16, 4, 128, 1000),
              (16, 4, 128, 4095), (16, 2, 256, 31), (16, 2, 256, 33), (16, 2, 256, 2303), (8, 8, 128, 300)]


@pytest.mark.parametrize("nq,nkv,hd,T", ATTN_CASES)
@pytest.mark.parametrize("nsplit", [1, 3, 16, 32, 64, 0])
def test_attention_parity(L, nq, nkv, hd, T, nsplit):
    rng = np.random.default_rng(T * 31 + hd + nsplit)
    cap = T + 3
    o, ref, Kg, Vg, Kr, Vr, ws, tol = run_attention(L, rng, nq, nkv, hd, cap, T, nsplit)
    assert_elementwise(o, ref, tol, f"attention T={T} nsplit={nsplit}")
    # appended rows: the bf16 code is decided in FP32 on both sides; allow one-ulp flips at rounding ties
    for got, want in ((Kg[:, T], Kr[:, T]), (Vg[:, T], Vr[:, T])):
        diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
        assert diff.max() <= 1 and (diff > 0).mean() < 0.01
    # only row T was written
    np.testing.assert_array_equal(Kg[:, :T], Kr[:, :T])
    np.testing.assert_array_equal(Kg[:, T + 1:], Kr[:, T + 1:])
    # the arrival counts (low 16 bits of each kv head's counter) are back to zero
    assert int((ws[:16].view(_torch().int32) & 0xFFFF).sum().item()) == 0


@pytest.mark.parametrize("nsplit", [1, 2, 4, 8, 16])
def test_attention_long_context_32k(L, nsplit):
    rng = np.random.default_rng(nsplit)
    T = 32768 + 127
    o, ref, *_, tol = run_attention(L, rng, 16, 4, 128, T + 1, T, nsplit)
    assert_elementwise(o, ref, tol, f"attention T={T} nsplit={nsplit}")
