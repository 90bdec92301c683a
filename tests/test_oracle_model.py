"""Whole-model oracle checks (CPU only).

The pages print no worked example of a whole decode step, so the composition
is pinned only through degenerate cases that reduce it to pinned parts:
zeroed mixer/FFN outputs leave the residual stream at the embedding, a MoE
whose experts are identical reduces to one SwiGLU FFN, and the hybrid
schedule touches exactly the state of the layers it names.
"""
import dataclasses

import numpy as np

from oracle import oracle as orc
from synth import gen, workloads

TINY = workloads.TINY


def tiny_weights():
    return workloads.host_weights(TINY)


def test_tiny_runs_and_is_deterministic():
    w = tiny_weights()
    a, b = orc.Oracle(TINY, w, 32), orc.Oracle(TINY, w, 32)
    ids = workloads.prompt_ids(workloads.WORKLOADS["tiny"], n=6)
    for t in ids:
        ra, rb = a.forward(int(t)), b.forward(int(t))
        assert np.all(np.isfinite(ra["logits"])) and np.all(np.isfinite(ra["hidden"]))
        np.testing.assert_array_equal(ra["logits"], rb["logits"])
    assert a.len == 6


def test_zero_outputs_leave_residual_at_embedding():
    w = tiny_weights()
    for l in range(TINY.n_layers):
        w[f"l{l}.w_o"] = np.zeros_like(w[f"l{l}.w_o"])
        w[f"l{l}.w_down"] = np.zeros_like(w[f"l{l}.w_down"])
    o = orc.Oracle(TINY, w, 8)
    tok = 77
    r = o.forward(tok)
    emb = gen.bf16_bits_to_f32(w["embed"][tok]).astype(np.float64)
    for l in range(TINY.n_layers):
        np.testing.assert_array_equal(r["hidden"][l], emb)
    xn = orc.rmsnorm(emb, w["final_norm"], TINY.rms_eps)
    ref = gen.bf16_bits_to_f32(w["lm_head"]).astype(np.float64) @ xn
    np.testing.assert_allclose(r["logits"], ref, rtol=1e-11, atol=1e-12)


def test_hybrid_schedule_touches_only_its_own_state():
    w = tiny_weights()
    o = orc.Oracle(TINY, w, 8)
    o.forward(5)
    o.forward(9)
    # layer 0 is Gated DeltaNet: its state moved; layer 1 is attention: two cached rows
    assert np.abs(o.gdn_state(0)).sum() > 0
    K, V = o.kv_cache(0)
    assert np.all(K[:, 2:] == 0) and np.any(K[:, :2] != 0) and np.any(V[:, :2] != 0)


def test_moe_with_identical_experts_reduces_to_one_ffn():
    H = 64
    shape = dataclasses.replace(TINY, name="moe-tiny", n_layers=1, hidden=H, vocab=50, ffn=0, gdn_heads=2,
                                gdn_dk=32, gdn_dv=32, attn_layers=(), n_experts=6, top_k=3, expert_ffn=32,
                                shared_ffn=32)
    w = workloads.host_weights(shape)
    Fe = shape.expert_ffn
    # every routed expert equal to the shared expert
    for src, dst in (("sh_gate", "exp_gate"), ("sh_up", "exp_up"), ("sh_down", "exp_down")):
        w[f"l0.{dst}"] = np.broadcast_to(w[f"l0.{src}"], w[f"l0.{dst}"].shape).copy()
    w["l0.w_o"] = np.zeros_like(w["l0.w_o"])  # isolate the FFN
    o = orc.Oracle(shape, w, 4)
    tok = 3
    r = o.forward(tok, want_router=True)
    emb = gen.bf16_bits_to_f32(w["embed"][tok]).astype(np.float64)
    xn = orc.rmsnorm(emb, w["l0.norm2"], shape.rms_eps)
    g = orc.gemv(w["l0.sh_gate"], xn)
    u = orc.gemv(w["l0.sh_up"], xn)
    ffn = orc.gemv(w["l0.sh_down"], g / (1 + np.exp(-g)) * u)
    gs = 1 / (1 + np.exp(-r["router_logits"][0][shape.n_experts]))
    # routed weights sum to one, so the routed part equals one FFN; plus the gated shared expert
    np.testing.assert_allclose(r["hidden"][0], emb + ffn + gs * ffn, rtol=1e-10, atol=1e-12)
    rl = r["router_logits"][0][:shape.n_experts]
    np.testing.assert_array_equal(r["router_ids"][0], orc.topk(rl, shape.top_k))
    assert Fe == 32


def _unions(shape, n_tok=8):
    """Distinct experts the router picks per layer for n_tok random tokens
    (each from an empty cache)."""
    w = workloads.host_weights(shape)
    toks = workloads.host.uniform_ids(1, 5, n_tok, shape.vocab)
    ids = np.array([orc.Oracle(shape, w, 4).forward(int(t), want_hidden=False, want_router=True)["router_ids"]
                    for t in toks])
    return [len(set(ids[:, l, :].ravel())) for l in range(shape.n_layers)]


def test_4bit_value_distribution_concentrates_routing():
    """The 4-bit workload's values are uniform in [-8, 7] (mean -0.5), so
    every 4-bit row carries a common component and the tokens' hidden states
    come to share a direction: a few layers in, 8 random tokens pick far fewer
    distinct experts than the 57 of uniform routing.  The bf16 model, whose
    weights have mean 0, keeps near-uniform routing."""
    cut = dict(n_layers=5, attn_layers=(3,))
    q4 = _unions(dataclasses.replace(workloads.MOE35B_Q4, name="q4-l5", **cut))
    bf = _unions(dataclasses.replace(workloads.MOE35B, name="bf16-l5", **cut))
    assert min(q4[:2]) >= 45 and max(q4[3:]) <= 25, q4
    assert min(bf) >= 45, bf
