"""The int8 KV cache (one FP32 scale per cached k or v vector): the attention
kernel through hy_op_attention_i8 against the oracle's int8 attention, and
whole models with kv_format 1 against the oracle's int8 path and against the
bf16 cache.

Tolerances: the cached rows before the new position are given to both sides
as the same codes and scales, so the attention bound of the bf16 tests
applies to their dequantised values; the new k and v vectors are quantised
by both sides from FP32 values that may differ in the last bits (the RoPE of
k in FP32 on the GPU, in FP64 on the oracle), so a code may differ by one
step only where the oracle's product lies within those bits of a rounding
boundary, and the bound gets that step for those elements."""
import dataclasses

import numpy as np
import pytest

from bandwidth_bound_hybrid_gb300 import capi
from oracle import oracle as orc
from synth import workloads
from tests.gpu_util import assert_elementwise, attention_tolerance, rel_l2, to_np

pytestmark = pytest.mark.gpu

U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def L(gpu):
    from bandwidth_bound_hybrid_gb300 import build
    build.build()
    return capi.lib()


def _torch():
    import torch
    return torch


def flip_candidates(x):
    """Elements of x whose int8 code can change under an FP32 perturbation of
    x by a few ulps (the amax scale moves with it)."""
    x = np.asarray(x, dtype=np.float64)
    lo, _ = orc.quant_i8(x * (1 - 8 * U32))
    hi, _ = orc.quant_i8(x * (1 + 8 * U32))
    mid, _ = orc.quant_i8(x)
    return (lo != mid) | (hi != mid)


@pytest.mark.parametrize("nq,nkv,hd,T,nsplit", [(4, 2, 64, 0, 1), (4, 2, 64, 200, 3), (16, 4, 128, 1000, 16),
                                                 (16, 4, 128, 4095, 0), (16, 2, 256, 2303, 32), (8, 8, 128, 37, 4),
                                                 (16, 4, 128, 3000, 64)])
def test_attention_int8_cache(L, nq, nkv, hd, T, nsplit):
    torch = _torch()
    rng = np.random.default_rng(T * 7 + hd + nsplit)
    cap = T + 5
    cap4 = (cap + 3) & ~3
    Kq = rng.integers(-127, 128, (nkv, cap, hd)).astype(np.int8)
    Vq = rng.integers(-127, 128, (nkv, cap, hd)).astype(np.int8)
    Ks = np.zeros((nkv, cap4), dtype=np.float32)
    Vs = np.zeros((nkv, cap4), dtype=np.float32)
    Ks[:, :cap] = rng.uniform(0.004, 0.012, (nkv, cap))
    Vs[:, :cap] = rng.uniform(0.004, 0.012, (nkv, cap))
    y = rng.standard_normal((nq + 2 * nkv) * hd).astype(np.float32)
    d = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (Kq, Ks, Vq, Vs, y)]
    table = torch.empty((cap, hd // 2, 2), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert L.hy_op_rope_table(table.data_ptr(), cap, hd, 1e4, st) == 0
    ln = torch.tensor([T], dtype=torch.int32, device="cuda")
    o = torch.empty(nq * hd, dtype=torch.float32, device="cuda")
    ws = torch.zeros(L.hy_op_attention_workspace(nq, nkv, hd, nsplit), dtype=torch.uint8, device="cuda")
    assert L.hy_op_attention_i8(d[4].data_ptr(), d[0].data_ptr(), d[1].data_ptr(), d[2].data_ptr(), d[3].data_ptr(),
                                cap, nq, nkv, hd, ln.data_ptr(), table.data_ptr(), nsplit, o.data_ptr(),
                                ws.data_ptr(), st) == 0, L.hy_last_error()
    torch.cuda.synchronize()
    # oracle: rotate, quantise the new k and v rows, attend over [0, T]
    yd = y.astype(np.float64)
    q = np.stack([orc.rope(yd[j * hd:(j + 1) * hd], T) for j in range(nq)])
    Kr, Vr, Ksr, Vsr = Kq.copy(), Vq.copy(), Ks[:, :cap].copy(), Vs[:, :cap].copy()
    kflip = np.zeros((nkv, hd), dtype=bool)
    vflip = np.zeros((nkv, hd), dtype=bool)
    for g in range(nkv):
        k = orc.rope(yd[(nq + g) * hd:(nq + g + 1) * hd], T)
        v = yd[(nq + nkv + g) * hd:(nq + nkv + g + 1) * hd]
        Kr[g, T], Ksr[g, T] = orc.quant_i8(k)
        Vr[g, T], Vsr[g, T] = orc.quant_i8(v)
        kflip[g], vflip[g] = flip_candidates(k), flip_candidates(v)
    ref = orc.attention_i8(q, Kr, Ksr, Vr, Vsr, T + 1)
    # the appended codes and scales
    gK, gKs, gV, gVs = (to_np(t) for t in d[:4])
    for got, want, fl in ((gK[:, T], Kr[:, T], kflip), (gV[:, T], Vr[:, T], vflip)):
        diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
        assert diff.max() <= 1 and not np.any(diff[~fl])
    np.testing.assert_allclose(gKs[:, T], Ksr[:, T], rtol=4 * U32)
    np.testing.assert_allclose(gVs[:, T], Vsr[:, T], rtol=4 * U32)
    np.testing.assert_array_equal(gK[:, :T], Kq[:, :T])
    np.testing.assert_array_equal(gV[:, :T], Vq[:, :T])
    # outputs: the bf16 bound on the dequantised values, plus one code step at the candidates of the new row
    Kw = Kr.astype(np.float64) * Ksr[..., None]
    Vw = Vr.astype(np.float64) * Vsr[..., None]
    tol = attention_tolerance(y[:nq * hd].reshape(nq, hd), q, Kw, Vw, T + 1, ref, nsplit if nsplit > 0 else 32)
    G = nq // nkv
    for j in range(nq):
        g = j // G
        sc = Kw[g, :T + 1] @ q[j] / np.sqrt(hd)
        p = np.exp(sc - sc.max())
        p /= p.sum()
        dk = Ksr[g, T] * np.sum(kflip[g] * np.abs(q[j])) / np.sqrt(hd)  # score change of the new row
        tol[j] += 4 * (p[T] * dk * np.abs(Vw[g, T] - ref[j]) + p[T] * Vsr[g, T] * vflip[g] +
                       8 * U32 * p[T] * np.abs(Vw[g, T]))
    assert_elementwise(to_np(o).reshape(nq, hd), ref, tol, f"int8 attention T={T}")


KV8_TINY = dataclasses.replace(workloads.TINY, name="tiny-kv8", kv_format=1)


def test_tiny_int8_cache_against_the_oracle(L):
    """Tiny hybrid with the int8 cache, 128-token prompt and 16 decode steps,
    per-layer hidden and logits against the oracle's int8 path."""
    from tests.test_gpu_model import run_parity
    run_parity(KV8_TINY, 128, 16)


def test_dense4b_truncated_int8_cache_against_the_oracle(L):
    shape = dataclasses.replace(workloads.DENSE4B, name="dense4b-l4-kv8", n_layers=4, attn_layers=(3,), vocab=4096,
                                kv_format=1)
    from tests.test_gpu_model import run_parity
    run_parity(shape, 40, 3)


def test_int8_cache_greedy_ids_follow_the_bf16_cache(L):
    """128 greedy steps of the tiny model, both caches fed the bf16 path's
    tokens: the int8 cache picks the same token wherever the bf16 logits'
    top-2 margin exceeds 0.05, and (measured) almost everywhere else."""
    torch = _torch()
    from bandwidth_bound_hybrid_gb300.model import HybridModel
    shape = workloads.TINY
    dev_w = workloads.device_weights(shape)
    steps = 128
    prompt = workloads.prompt_ids(workloads.WORKLOADS["tiny"], n=32)
    mb = HybridModel(shape, dev_w, [32 + steps + 1])
    m8 = HybridModel(KV8_TINY, dev_w, [32 + steps + 1])
    lb = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    l8 = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    toks = torch.from_numpy(prompt).cuda()
    mb.prefill(0, toks, lb)
    m8.prefill(0, toks, l8)
    ib = torch.empty(1, dtype=torch.int32, device="cuda")
    i8 = torch.empty(1, dtype=torch.int32, device="cuda")
    same = gated = 0
    for s in range(steps):
        torch.cuda.synchronize()
        gb, g8 = to_np(lb), to_np(l8)
        srt = np.sort(gb)
        if srt[-1] - srt[-2] > 0.05:
            gated += 1
            assert int(np.argmax(g8)) == int(np.argmax(gb)), f"step {s}"
        same += int(np.argmax(g8)) == int(np.argmax(gb))
        assert rel_l2(g8, gb) < 2e-2
        nxt = torch.tensor([int(np.argmax(gb))], dtype=torch.int32, device="cuda")
        mb.decode_step(0, nxt, ib, lb)
        m8.decode_step(0, nxt, i8, l8)
    print(f"int8 cache: {same} of {steps} greedy ids equal to the bf16 cache's ({gated} margin-gated)")
    assert same >= 0.95 * steps
    assert mb.check_device() == 0 and m8.check_device() == 0
    mb.close()
    m8.close()
