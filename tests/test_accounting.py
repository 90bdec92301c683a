"""Byte accounting of a decode step, pinned to the figures the pages print
(tests/golden/strata_figures.txt) and to per-config totals worked out from the model shapes."""
import os

from bandwidth_bound_hybrid_gb300 import accounting as acc
from synth import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "strata_figures.txt")


def golden():
    with open(GOLDEN) as f:
        return {ln.split()[0]: ln.split()[1:] for ln in f if ln.strip() and not ln.startswith("#")}


def test_state_and_kv_sizes_match_the_page():
    g = golden()
    nh, dk, dv, b = map(int, g["gdn_state_layer_bytes"])
    assert acc.gdn_state_bytes_per_layer(nh, dk, dv) == b  # 2.0 MB
    assert 24 * acc.gdn_state_bytes_per_layer(nh, dk, dv) == int(g["gdn_state_24_layers_bytes"][0])  # 48.0 MB
    n_attn, nkv, hd, kv = map(int, g["kv_per_token"])
    assert acc.kv_bytes_per_token(n_attn, nkv, hd) == kv  # 32 KB per token


def test_roofline_formula_reproduces_the_page():
    g = golden()
    bw, gb, tok = map(float, g["roofline"])
    ceil = acc.roofline_tokens_per_s(bw, gb * 1e9)
    assert abs(ceil - tok) < 0.05
    got, frac = map(float, g["fraction"])
    assert abs(got / ceil - frac) < 0.001


def test_dense4b_step_bytes():
    s = workloads.DENSE4B
    b = acc.step_bytes(s, 4352)
    # weights: every linear layer once (3.264 B params) -> ~6.53 GB
    assert 6.50e9 < b.weights < 6.56e9
    # 16 KB of K+V per token over 8 layers (4 kv heads x 128 x bf16 x 2)
    assert acc.kv_bytes_per_token(8, 4, 128) == 16384
    assert b.kv_read == 16384 * 4352
    assert 6.60e9 < b.total < 6.70e9


def test_moe_step_bytes_counts_selected_experts_only():
    s = workloads.MOE35B
    b = acc.step_bytes(s, 2304)
    assert 4.25e9 < b.weights < 4.40e9
    more = acc.step_bytes(s, 2304, experts_touched=16)
    per_expert = 3 * 512 * 2048 * 2 * s.n_layers
    assert more.weights - b.weights == 8 * per_expert


def test_kernels_per_step():
    assert acc.kernels_per_step(workloads.DENSE4B) == 32 * 5 + 1
    assert acc.kernels_per_step(workloads.MOE35B) == 40 * 6 + 1


def test_expected_union_against_a_direct_simulation():
    """E (1 - (1 - k/E)^B): the expected number of distinct experts B tokens
    pick, each taking k of E uniformly without replacement, checked against
    sampling (and its end points)."""
    import numpy as np
    assert acc.expected_union(256, 8, 1) == 8.0
    assert abs(acc.expected_union(16, 16, 3) - 16.0) < 1e-12
    rng = np.random.default_rng(0)
    E, k, B = 256, 8, 8
    sizes = [len(set(np.concatenate([rng.choice(E, k, replace=False) for _ in range(B)]))) for _ in range(4000)]
    assert abs(np.mean(sizes) - acc.expected_union(E, k, B)) < 0.3  # 57.42; sampling error ~0.05


def test_batch_step_bytes_count_the_union_once_and_each_sequence_state_and_kv():
    s = workloads.MOE35B_Q4
    ctx = [1000, 2000, 3000, 4000]
    one = acc.step_bytes(s, 0, 10)
    b = acc.batch_step_bytes(s, ctx, 10)
    assert b.state == len(ctx) * one.state
    assert b.kv_read == acc.kv_bytes_per_token(10, s.attn_kv_heads, s.head_dim) * sum(ctx)
    assert b.kv_write == len(ctx) * one.kv_write
    # the weights once, plus one embedding row per further token
    assert b.weights == one.weights + (len(ctx) - 1) * s.hidden * acc.BF16
    # a fractional union adds that fraction of one expert's three matrices per layer
    per_exp = 3 * acc.linear_bytes(s.expert_ffn, s.hidden, 1)
    frac = acc.batch_step_bytes(s, ctx, 10.25)
    assert frac.weights - b.weights == round(s.n_layers * per_exp * 0.25)


def test_batch_gemv_bytes():
    assert acc.gemv_batch_bytes(16, 256, 8, 0) == 16 * 256 * 2 + 8 * (256 + 16) * 4
    assert acc.gemv_batch_bytes(16, 256, 8, 1) == 16 * 128 + 16 * 8 * 2 + 8 * (256 + 16) * 4
