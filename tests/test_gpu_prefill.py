"""The chunked prompt path (tensor-core GEMMs, for MoE models the grouped
expert GEMMs, and the prompt mixer kernels) against the FP64 oracle and against the token-by-token prefill through the
decode step: several chunks with a ragged last one, a prompt continued by a
second call (positions not starting at 0), a single-token prompt, and the
decode steps that follow, which read the caches the prefill left.

Tolerances as for the decode step: per-layer hidden rel-L2 <= 5e-3 and final
logits rel-L2 <= 1e-2 against the oracle; greedy ids where the oracle's top-2
margin exceeds 0.05.  The chunked and the token-by-token prefill compute the
same sums in another order (tensor-core GEMMs with bf16 hi + lo activations
instead of FP32 GEMVs), so they agree to 1e-4 (rel-L2 of logits and hidden)."""
import dataclasses
import os

import numpy as np
import pytest

from bandwidth_bound_hybrid_gb300 import capi
from oracle import oracle as orc
from synth import workloads
from tests.gpu_util import rel_l2, to_np

pytestmark = pytest.mark.gpu

HIDDEN_TOL, LOGIT_TOL, ID_MARGIN, SAME_TOL = 5e-3, 1e-2, 0.05, 1e-4


@pytest.fixture(scope="module")
def built(gpu):
    from bandwidth_bound_hybrid_gb300 import build
    build.build()
    return True


@pytest.fixture
def chunk_rows():
    old = os.environ.get("HY_PREFILL_CHUNK")

    def set_rows(n):
        os.environ["HY_PREFILL_CHUNK"] = str(n)

    yield set_rows
    if old is None:
        os.environ.pop("HY_PREFILL_CHUNK", None)
    else:
        os.environ["HY_PREFILL_CHUNK"] = old


def hidden_of(model, shape):
    return [to_np(model.debug_hidden(l)).copy() for l in range(shape.n_layers)]


def run(shape, segments, n_decode, seed=1, same_tol=SAME_TOL):
    """Prefill the prompt in `segments` (lengths of consecutive prefill calls),
    then decode n_decode greedy steps (the oracle's token), comparing the
    chunked model with the oracle and with the token-by-token model."""
    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    total = sum(segments)
    cap = total + n_decode + 1
    dev_w = workloads.device_weights(shape)
    fast = HybridModel(shape, dev_w, [cap], flags=capi.HY_FLAG_DEBUG)
    slow = HybridModel(shape, dev_w, [cap], flags=capi.HY_FLAG_DEBUG | capi.HY_FLAG_TOKEN_PREFILL)
    ref = orc.Oracle(shape, workloads.host_weights(shape), cap)
    prompt = workloads.host.uniform_ids(seed, workloads.PROMPT_TID, total, shape.vocab)
    lf = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    ls = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    i0 = 0
    for n in segments:
        toks = torch.from_numpy(prompt[i0:i0 + n]).cuda()
        fast.prefill(0, toks, lf)
        slow.prefill(0, toks, ls)
        for t in prompt[i0:i0 + n]:
            r = ref.forward(int(t), want_router=shape.is_moe)
        i0 += n
        torch.cuda.synchronize()
        hf, hs = hidden_of(fast, shape), hidden_of(slow, shape)
        for l in range(shape.n_layers):
            assert rel_l2(hf[l], r["hidden"][l]) <= HIDDEN_TOL, f"prefill to {i0}: layer {l} vs oracle"
            assert rel_l2(hf[l], hs[l]) <= same_tol, f"prefill to {i0}: layer {l} chunked vs token by token"
        if shape.is_moe:  # the last token picked the oracle's experts in every layer (or differs at a near-tie)
            for l in range(shape.n_layers):
                dev = sorted(to_np(fast.debug_router(l)[1]).tolist())
                if dev != sorted(int(i) for i in r["router_ids"][l]):
                    srt = np.sort(np.asarray(r["router_logits"][l][:shape.n_experts]))[::-1]
                    gap = srt[shape.top_k - 1] - srt[shape.top_k]
                    assert gap <= 1e-3 * max(1.0, abs(srt[0])), f"prefill to {i0}: layer {l} experts {dev}"
        assert rel_l2(to_np(lf), r["logits"]) <= LOGIT_TOL
        assert rel_l2(to_np(lf), to_np(ls)) <= same_tol
    assert fast.seq_len(0) == total and slow.seq_len(0) == total
    ids_f = torch.empty(1, dtype=torch.int32, device="cuda")
    ids_s = torch.empty(1, dtype=torch.int32, device="cuda")
    for s in range(n_decode):
        nxt = int(orc.argmax(r["logits"]))
        tok = torch.tensor([nxt], dtype=torch.int32, device="cuda")
        fast.decode_step(0, tok, ids_f, lf)
        slow.decode_step(0, tok, ids_s, ls)
        r = ref.forward(nxt)
        torch.cuda.synchronize()
        e = rel_l2(to_np(lf), r["logits"])
        assert e <= LOGIT_TOL, f"decode {s}: logits rel-L2 {e:.3g}"
        assert rel_l2(to_np(lf), to_np(ls)) <= same_tol, f"decode {s}: chunked vs token-by-token caches"
        hf = hidden_of(fast, shape)
        for l in range(shape.n_layers):
            assert rel_l2(hf[l], r["hidden"][l]) <= HIDDEN_TOL, f"decode {s} layer {l}"
        srt = np.sort(r["logits"])
        if srt[-1] - srt[-2] > ID_MARGIN:
            assert int(ids_f.item()) == int(orc.argmax(r["logits"]))
    assert fast.check_device() == 0 and slow.check_device() == 0
    fast.close()
    slow.close()


def test_tiny_prompt_in_ragged_chunks(built, chunk_rows):
    """Tiny hybrid, a 130-token prompt in chunks of 48 (48 + 48 + 34)."""
    chunk_rows(48)
    run(workloads.TINY, [130], 4)


def test_tiny_prompt_continued_by_a_second_call(built, chunk_rows):
    """Positions of the second call start at 57 (the conv ring and the KV
    rows of the first call are read back); then a single-token prefill."""
    chunk_rows(2048)
    run(workloads.TINY, [57, 70, 1], 3)


def test_dense4b_full_widths_truncated_depth(built, chunk_rows):
    """Full widths of the dense 4B-shaped model (hidden 2560, FFN 9216,
    16x128 DeltaNet heads, 16/4x128 GQA), 4 layers, vocab cut to 4096 for
    the oracle's sake; a 300-token prompt in chunks of 128 (two full M tiles
    of the GEMM and a ragged one)."""
    chunk_rows(128)
    shape = dataclasses.replace(workloads.DENSE4B, name="dense4b-l4-v4k", n_layers=4, attn_layers=(3,), vocab=4096)
    run(shape, [300], 2)


# a tiny bf16 MoE hybrid whose widths suit the GEMM's tensor copies (multiples of 8)
TINY_MOE = workloads.ModelShape("tiny-moe-bf16", n_layers=2, hidden=256, vocab=1024, ffn=0, gdn_heads=4, gdn_dk=64,
                                gdn_dv=64, attn_q_heads=4, attn_kv_heads=2, head_dim=64, attn_layers=(1,),
                                n_experts=16, top_k=4, expert_ffn=256, shared_ffn=256)


def test_tiny_moe_prompt_in_ragged_chunks(built, chunk_rows):
    """Tiny MoE hybrid (16 experts, top 4, shared expert), a 130-token prompt
    in chunks of 48: router GEMM, routing, the grouped expert GEMMs, the
    shared expert and the combine, against the oracle and the token-by-token
    prefill; then decode steps on the caches it left."""
    chunk_rows(48)
    run(TINY_MOE, [130], 4)


def test_moe_full_widths_truncated_depth(built, chunk_rows):
    """Full widths of the MoE 35B-A3B-shaped model (hidden 2048, 256 experts
    of 512, top 8, shared expert, 16x128 DeltaNet heads, 16/2x256 GQA), 4
    layers, vocab cut to 4096; a 200-token prompt in chunks of 128, so that
    experts take several grouped tiles or none."""
    chunk_rows(128)
    shape = dataclasses.replace(workloads.MOE35B, name="moe-l4-v4k", n_layers=4, attn_layers=(3,), vocab=4096)
    # a MoE layer's output sums top_k + 1 = 9 expert outputs, each with the rounding of the bf16 hi / lo parts
    # of its input and of its SwiGLU output; 9 such terms add about sqrt(9) = 3 times a dense FFN's rounding
    # difference between the two paths (1e-4 at dense widths)
    run(shape, [200], 2, same_tol=3 * SAME_TOL)


def test_prefill_refuses_past_capacity_with_nothing_launched(built):
    import torch

    from bandwidth_bound_hybrid_gb300.model import HybridModel
    model = HybridModel(workloads.TINY, workloads.device_weights(workloads.TINY), [16])
    toks = torch.zeros(17, dtype=torch.int32, device="cuda")
    with pytest.raises(capi.HybridError) as ei:
        model.prefill(0, toks)
    assert ei.value.code == capi.HY_ERR_CAPACITY
    assert model.seq_len(0) == 0
    model.close()
