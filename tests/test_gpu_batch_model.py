"""Batched decode (several sequences per step, one weight stream) and 4-bit
block weights, through the C ABI, against the FP64 oracle run on each
sequence alone.

Gates as for single-sequence decode: per-layer hidden relative L2 <= 5e-3
(first token of a step), final-logit relative L2 <= 1e-2 for every sequence,
greedy ids bit-exact where the oracle's top-2 margin exceeds 0.05.  Every
sequence consumes its own oracle's greedy token (teacher forcing)."""
import dataclasses

import numpy as np
import pytest

from bandwidth_bound_hybrid_gb300 import capi
from oracle import oracle as orc
from synth import workloads
from tests.gpu_util import rel_l2, to_np

pytestmark = pytest.mark.gpu

HIDDEN_TOL, LOGIT_TOL, ID_MARGIN = 5e-3, 1e-2, 0.05

# a tiny MoE hybrid whose widths suit 4-bit blocks (multiples of 256)
TINY_MOE_Q4 = workloads.ModelShape("tiny-moe-q4", n_layers=2, hidden=256, vocab=1024, ffn=0, gdn_heads=4, gdn_dk=64,
                                   gdn_dv=64, attn_q_heads=4, attn_kv_heads=2, head_dim=64, attn_layers=(1,),
                                   n_experts=16, top_k=4, expert_ffn=256, shared_ffn=256, weight_format=1)


@pytest.fixture(scope="module")
def built(gpu):
    from bandwidth_bound_hybrid_gb300 import build
    build.build()
    return True


def prompts_for(shape, lens, seed=3):
    return [workloads.host.uniform_ids(seed + i, workloads.PROMPT_TID, n, shape.vocab) for i, n in enumerate(lens)]


def run(shape, prompt_lens, n_steps, flags=capi.HY_FLAG_DEBUG, check_hidden=True):
    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    B = len(prompt_lens)
    host_w = workloads.host_weights(shape)
    model = HybridModel(shape, workloads.device_weights(shape), [n + n_steps + 1 for n in prompt_lens], flags=flags)
    refs = [orc.Oracle(shape, host_w, n + n_steps + 1) for n in prompt_lens]
    prompts = prompts_for(shape, prompt_lens)
    last = []
    for s, (ref, pr) in enumerate(zip(refs, prompts)):
        lg = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        model.prefill(s, torch.from_numpy(pr).cuda(), lg)
        for t in pr:
            r = ref.forward(int(t))
        torch.cuda.synchronize()
        e = rel_l2(to_np(lg), r["logits"])
        assert e <= LOGIT_TOL, f"sequence {s} after prefill: logits rel-L2 {e:.3g}"
        if check_hidden and s == B - 1:  # the last prefill step ran sequence s alone
            for l in range(shape.n_layers):
                eh = rel_l2(to_np(model.debug_hidden(l)), r["hidden"][l])
                assert eh <= HIDDEN_TOL, f"prefill of sequence {s}, layer {l}: hidden rel-L2 {eh:.3g}"
        last.append(r)
    seqs = list(range(B))
    logits = torch.empty((B, shape.vocab), dtype=torch.float32, device="cuda")
    ids = torch.empty(B, dtype=torch.int32, device="cuda")
    for step in range(n_steps):
        nxt = [int(orc.argmax(r["logits"])) for r in last]
        model.decode_batch(seqs, torch.tensor(nxt, dtype=torch.int32, device="cuda"), ids, logits)
        last = [ref.forward(t) for ref, t in zip(refs, nxt)]
        torch.cuda.synchronize()
        got = to_np(logits)
        gid = to_np(ids)
        for s in range(B):
            e = rel_l2(got[s], last[s]["logits"])
            assert e <= LOGIT_TOL, f"step {step} sequence {s}: logits rel-L2 {e:.3g}"
            srt = np.sort(last[s]["logits"])
            if srt[-1] - srt[-2] > ID_MARGIN:
                assert int(gid[s]) == int(orc.argmax(last[s]["logits"])), f"step {step} sequence {s}"
        if check_hidden:
            for l in range(shape.n_layers):
                eh = rel_l2(to_np(model.debug_hidden(l)), last[0]["hidden"][l])
                assert eh <= HIDDEN_TOL, f"step {step} layer {l}: hidden rel-L2 {eh:.3g}"
    for s, n in enumerate(prompt_lens):
        assert model.seq_len(s) == n + n_steps
    assert model.check_device() == 0
    model.close()


def test_tiny_q4_moe_one_sequence(built):
    """4-bit weights: prefill and decode run the batched path with one sequence."""
    run(TINY_MOE_Q4, [12], 4)


def test_tiny_q4_moe_batch_of_eight_ragged(built):
    run(TINY_MOE_Q4, [3, 9, 5, 12, 7, 4, 10, 6], 4)


def test_tiny_bf16_dense_batch_of_three(built):
    """bf16 weights, several sequences: batched tensor-core projections (the
    activations rounded to bf16 for the MMA)."""
    run(workloads.TINY, [5, 9, 14], 4)


def test_moe35b_q4_truncated_batch(built):
    """The 4-bit MoE 35B-A3B shape at full widths (256 experts of 512, top-8
    + shared, 16/2x256 GQA, vocab 151936), first 2 layers (DeltaNet +
    attention), four sequences: the union of up to 32 selected experts."""
    shape = dataclasses.replace(workloads.MOE35B_Q4, name="moe-q4-l2", n_layers=2, attn_layers=(1,))
    run(shape, [3, 5, 2, 4], 2)


@pytest.mark.parametrize("spread", ["", "0", "5"])
def test_ragged_batch_attention_splits(built, monkeypatch, spread):
    """Batched attention over strongly ragged contexts: the step's splits
    shared among the sequences in proportion to their lengths on the device
    (the default), one split count for every sequence (spread off), and 5
    splits for 4 sequences (one each, the largest remainder a second): every
    sequence against its own oracle."""
    if spread:
        monkeypatch.setenv("HY_ATTN_BATCH_SPREAD", spread)
    else:
        monkeypatch.delenv("HY_ATTN_BATCH_SPREAD", raising=False)
    run(TINY_MOE_Q4, [1, 150, 2, 40], 3)


def test_batch_rejects_repeated_and_full_sequences(built):
    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    shape = TINY_MOE_Q4
    model = HybridModel(shape, workloads.device_weights(shape), [4, 4], flags=0)
    ids = torch.empty(2, dtype=torch.int32, device="cuda")
    toks = torch.tensor([1, 2], dtype=torch.int32, device="cuda")
    with pytest.raises(capi.HybridError) as ei:
        model.decode_batch([0, 0], toks, ids)
    assert ei.value.code == capi.HY_ERR_ARG
    model.prefill(1, torch.arange(4, dtype=torch.int32, device="cuda"))
    with pytest.raises(capi.HybridError) as ei:
        model.decode_batch([0, 1], toks, ids)
    assert ei.value.code == capi.HY_ERR_CAPACITY and model.seq_len(0) == 0
    model.decode_batch([0], toks[:1], ids)
    assert model.seq_len(0) == 1 and model.check_device() == 0
    model.close()


def test_synthetic_fill(built):
    """hy_seq_fill_synthetic: the same seed gives the same cache (identical
    outputs for two sequences), another seed another cache; the length is set
    and bounded by the capacity."""
    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    shape = TINY_MOE_Q4
    model = HybridModel(shape, workloads.device_weights(shape), [40, 40, 40], flags=0)
    model.fill_synthetic(0, 30, seed=5)
    model.fill_synthetic(1, 30, seed=5)
    model.fill_synthetic(2, 30, seed=6)
    assert [model.seq_len(s) for s in range(3)] == [30, 30, 30]
    toks = torch.tensor([7, 7, 7], dtype=torch.int32, device="cuda")
    ids = torch.empty(3, dtype=torch.int32, device="cuda")
    lg = torch.empty((3, shape.vocab), dtype=torch.float32, device="cuda")
    model.decode_batch([0, 1, 2], toks, ids, lg)
    torch.cuda.synchronize()
    got = to_np(lg)
    assert np.all(np.isfinite(got))
    np.testing.assert_array_equal(got[0], got[1])
    assert np.abs(got[0] - got[2]).max() > 0
    with pytest.raises(capi.HybridError) as ei:
        model.fill_synthetic(0, 41)
    assert ei.value.code == capi.HY_ERR_CAPACITY and model.seq_len(0) == 31
    model.fill_synthetic(0, 0)
    assert model.seq_len(0) == 0 and model.check_device() == 0
    model.close()


def test_experts_read_counts_the_union(built):
    """hy_experts_read: per MoE layer a batched step reads the union of its
    tokens' picks once: between top_k and min(E, B top_k) experts; reading
    resets the count."""
    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    shape = TINY_MOE_Q4
    B = 8
    model = HybridModel(shape, workloads.device_weights(shape), [16] * B, flags=0)
    toks = torch.tensor(list(range(3, 3 + B)), dtype=torch.int32, device="cuda")
    ids = torch.empty(B, dtype=torch.int32, device="cuda")
    model.experts_read()
    model.decode_batch(list(range(B)), toks, ids)
    n = model.experts_read()
    layers = shape.n_layers  # every layer of this shape is MoE
    assert layers * shape.top_k <= n <= layers * min(shape.n_experts, B * shape.top_k)
    assert model.experts_read() == 0
    model.close()


def test_dense4b_truncated_batch_of_two(built):
    """bf16 at the dense 4B shape's full widths (hidden 2560, FFN 9216), first
    2 layers, two sequences: the down projection's 9216-wide token vectors do
    not fit the kernel's shared memory and run as column slices that
    accumulate in order."""
    shape = dataclasses.replace(workloads.DENSE4B, name="dense4b-l2", n_layers=2, attn_layers=(1,), vocab=4096)
    run(shape, [3, 5], 2)


def test_moe_top16_batch_of_four_at_the_pick_limit(built):
    """top_k 16 (the largest the header allows) for four sequences in one
    batched step: 64 routed picks, the most a batched MoE step holds."""
    shape = dataclasses.replace(workloads.TINY, name="tiny-moe-k16", vocab=512, ffn=0, n_experts=64, top_k=16,
                                expert_ffn=64, shared_ffn=64)
    run(shape, [5, 9, 12, 7], 2)
