"""Byte accounting of a decode step, pinned to the figures the pages print
(tests/golden/strata_figures.txt) and to the survey's per-config totals."""
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
