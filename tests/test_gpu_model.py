"""Whole decode-step parity through the C ABI against the FP64 oracle.

Gates (the method's stated tolerances): per-layer hidden relative L2 <= 5e-3,
final-logit relative L2 <= 1e-2; greedy ids bit-exact wherever the oracle's
top-2 logit margin exceeds 0.05; router expert ids bit-exact (as a set)
wherever the gap between the k-th and (k+1)-th router logit exceeds 1e-3.
Both sides consume the oracle's greedy token at every step (teacher forcing),
so one near-tie cannot cascade.
"""
import dataclasses

import numpy as np
import pytest

from bandwidth_bound_hybrid_gb300 import capi
from oracle import oracle as orc
from synth import workloads
from tests.gpu_util import rel_l2, to_np

pytestmark = pytest.mark.gpu

HIDDEN_TOL, LOGIT_TOL, ID_MARGIN, ROUTER_GAP = 5e-3, 1e-2, 0.05, 1e-3


@pytest.fixture(scope="module")
def built(gpu):
    from bandwidth_bound_hybrid_gb300 import build
    build.build()
    return True


def make(shape, capacity, flags=capi.HY_FLAG_DEBUG, splits=0, host=True):
    from bandwidth_bound_hybrid_gb300.model import HybridModel
    dev_w = workloads.device_weights(shape)
    model = HybridModel(shape, dev_w, [capacity], splits=splits, flags=flags)
    ref = orc.Oracle(shape, workloads.host_weights(shape), capacity) if host else None
    return model, ref


def compare_step(model, ref_out, logits, shape, step, router=False):
    import torch
    torch.cuda.synchronize()
    for l in range(shape.n_layers):
        h = to_np(model.debug_hidden(l))
        e = rel_l2(h, ref_out["hidden"][l])
        assert e <= HIDDEN_TOL, f"step {step} layer {l}: hidden rel-L2 {e:.3g}"
    e = rel_l2(to_np(logits), ref_out["logits"])
    assert e <= LOGIT_TOL, f"step {step}: logits rel-L2 {e:.3g}"
    if router and shape.ffn == 0:
        for l in range(shape.n_layers):
            rl = ref_out["router_logits"][l][:shape.n_experts]
            srt = np.sort(rl)[::-1]
            if srt[shape.top_k - 1] - srt[shape.top_k] > ROUTER_GAP:
                _, ids = model.debug_router(l)
                assert set(to_np(ids).tolist()) == set(ref_out["router_ids"][l].tolist()), f"step {step} layer {l}"
    return rel_l2(to_np(logits), ref_out["logits"])


def greedy_ok(gpu_id, ref_logits):
    srt = np.sort(ref_logits)
    if srt[-1] - srt[-2] > ID_MARGIN:
        return gpu_id == int(orc.argmax(ref_logits))
    return True


def run_parity(shape, prompt_len, n_decode, capacity=None, prefill_path=True, seed_seq=0):
    import torch
    capacity = capacity or prompt_len + n_decode + 1
    model, ref = make(shape, capacity, flags=capi.HY_FLAG_DEBUG)
    prompt = workloads.host.uniform_ids(1 + seed_seq, workloads.PROMPT_TID, prompt_len, shape.vocab)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    ids = torch.empty(1, dtype=torch.int32, device="cuda")
    want_router = shape.ffn == 0
    if prefill_path:
        model.prefill(0, torch.from_numpy(prompt).cuda(), logits)
        for t in prompt:
            r = ref.forward(int(t), want_router=want_router)
        compare_step(model, r, logits, shape, "prefill", router=want_router)
    else:
        for i, t in enumerate(prompt):
            model.decode_step(0, torch.tensor([int(t)], dtype=torch.int32, device="cuda"), ids, logits)
            r = ref.forward(int(t), want_router=want_router)
            compare_step(model, r, logits, shape, i, router=want_router)
            assert greedy_ok(int(ids.item()), r["logits"])
    matched = 0
    for s in range(n_decode):
        nxt = int(orc.argmax(r["logits"]))
        model.decode_step(0, torch.tensor([nxt], dtype=torch.int32, device="cuda"), ids, logits)
        r = ref.forward(nxt, want_router=want_router)
        compare_step(model, r, logits, shape, f"decode {s}", router=want_router)
        assert greedy_ok(int(ids.item()), r["logits"]), f"decode {s}"
        matched += int(int(ids.item()) == int(orc.argmax(r["logits"])))
    assert model.seq_len(0) == prompt_len + n_decode
    assert model.check_device() == 0
    assert model.step_kernels() > 1
    model.close()
    return matched


def test_tiny_full_parity(built):
    """Tiny hybrid: 128-token prompt, then 16 greedy decode steps."""
    w = workloads.WORKLOADS["tiny"]
    run_parity(w.shape, w.prompt_len, w.decode_steps)


def test_tiny_per_token_parity_through_decode_steps(built):
    run_parity(workloads.TINY, 40, 4, prefill_path=False)


def test_dense4b_truncated_depth_parity(built):
    """Full widths of the dense 4B-shaped model (hidden 2560, FFN 9216, vocab
    151936, 16x128 DeltaNet heads, 16/4x128 GQA), first 4 layers (3 DeltaNet +
    1 attention)."""
    shape = dataclasses.replace(workloads.DENSE4B, name="dense4b-l4", n_layers=4, attn_layers=(3,))
    run_parity(shape, 6, 3)


def test_moe_truncated_depth_parity(built):
    """Full widths of the MoE 35B-A3B-shaped model (256 experts of 512, top-8
    + shared, 16/2x256 GQA), first 4 layers."""
    shape = dataclasses.replace(workloads.MOE35B, name="moe-l4", n_layers=4, attn_layers=(3,))
    run_parity(shape, 5, 3)


@pytest.mark.parametrize("flags", [capi.HY_FLAG_NO_GRAPH, capi.HY_FLAG_NO_PDL, capi.HY_FLAG_NO_GRAPH | capi.HY_FLAG_NO_PDL])
def test_graph_and_pdl_do_not_change_results(built, flags):
    import torch
    shape = dataclasses.replace(workloads.DENSE4B, name="dense4b-l4", n_layers=4, attn_layers=(3,), vocab=4096)
    prompt = workloads.host.uniform_ids(7, workloads.PROMPT_TID, 20, shape.vocab)
    outs = []
    for f in (0, flags):
        model, _ = make(shape, 32, flags=f, host=False)
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        ids = torch.empty(1, dtype=torch.int32, device="cuda")
        model.prefill(0, torch.from_numpy(prompt).cuda())
        seq = []
        for _ in range(5):
            model.decode_step(0, ids if seq else torch.tensor([1], dtype=torch.int32, device="cuda"), ids, logits)
            torch.cuda.synchronize()
            seq.append((int(ids.item()), to_np(logits).copy()))
        outs.append(seq)
        model.close()
    for (a, la), (b, lb) in zip(*outs):
        assert a == b
        np.testing.assert_array_equal(la, lb)


def test_capacity_is_checked_before_launch(built):
    import torch
    shape = workloads.TINY
    model, _ = make(shape, 6, flags=0, host=False)
    toks = torch.arange(6, dtype=torch.int32, device="cuda")
    ids = torch.empty(1, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.HybridError) as ei:
        model.prefill(0, torch.arange(7, dtype=torch.int32, device="cuda"))
    assert ei.value.code == capi.HY_ERR_CAPACITY and model.seq_len(0) == 0
    model.prefill(0, toks)
    assert model.seq_len(0) == 6
    with pytest.raises(capi.HybridError) as ei:
        model.decode_step(0, toks[:1], ids)
    assert ei.value.code == capi.HY_ERR_CAPACITY and model.seq_len(0) == 6
    model.reset(0)
    assert model.seq_len(0) == 0
    model.decode_step(0, toks[:1], ids)
    assert model.check_device() == 0
    model.close()


def test_reset_replays_identically(built):
    import torch
    shape = workloads.TINY
    model, _ = make(shape, 64, flags=0, host=False)
    prompt = torch.from_numpy(workloads.prompt_ids(workloads.WORKLOADS["tiny"], n=30)).cuda()
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    runs = []
    for _ in range(2):
        model.reset(0)
        model.prefill(0, prompt, logits)
        torch.cuda.synchronize()
        runs.append(to_np(logits).copy())
    np.testing.assert_array_equal(runs[0], runs[1])
    model.close()


def test_out_of_range_token_sets_guard_not_fault(built):
    import torch
    shape = workloads.TINY
    model, _ = make(shape, 8, flags=0, host=False)
    ids = torch.empty(1, dtype=torch.int32, device="cuda")
    model.decode_step(0, torch.tensor([shape.vocab + 5], dtype=torch.int32, device="cuda"), ids)
    assert model.check_device() & capi.HY_GUARD_BAD_INDEX
    assert model.check_device() == 0  # cleared after reading
    model.close()


def test_host_buffer_step_matches_device_step(built):
    import torch
    shape = workloads.TINY
    a, _ = make(shape, 16, flags=0, host=False)
    b, _ = make(shape, 16, flags=0, host=False)
    ids_d = torch.empty(1, dtype=torch.int32, device="cuda")
    lg_d = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    tok_h = torch.tensor([17], dtype=torch.int32).pin_memory()
    ids_h = torch.empty(1, dtype=torch.int32).pin_memory()
    lg_h = torch.empty(shape.vocab, dtype=torch.float32).pin_memory()
    for _ in range(3):
        a.decode_step(0, tok_h.cuda(), ids_d, lg_d)
        b.decode_step_host(0, tok_h, ids_h, lg_h)
        torch.cuda.synchronize()
        assert int(ids_d.item()) == int(ids_h.item())
        np.testing.assert_array_equal(to_np(lg_d), lg_h.numpy())
        tok_h[0] = int(ids_h.item())
    a.close()
    b.close()


def test_moe_with_511_experts(built):
    """511 routed experts (the header's limit: the router's 512th row gates the
    shared expert) at batch 1, against the oracle with the router ids checked."""
    shape = dataclasses.replace(workloads.TINY, name="tiny-moe-e511", vocab=512, ffn=0, n_experts=511, top_k=8,
                                expert_ffn=64, shared_ffn=64)
    run_parity(shape, 8, 3)

