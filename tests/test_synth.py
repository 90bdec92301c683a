"""The seeded input generator: published SplitMix64 vectors, and agreement of
its numpy definition with the host C copy (CPU only)."""
import os

import numpy as np

from synth import gen, host, workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_vectors():
    with open(os.path.join(GOLDEN, "splitmix64_state0.txt")) as f:
        expect = [int(ln, 16) for ln in f if ln.strip() and not ln.startswith("#")]
    # tensor stream (seed 0, id 0) has key mix64(0) = 0, so its words are the state-0 sequence
    assert gen.stream_key(0, 0) == 0
    got = [int(w) for w in gen.words(0, 0, 0, 3)]
    assert got == expect


def test_host_copy_matches_numpy_definition():
    for seed, tid, n, start in [(0, 5, 1000, 0), (3, 1_000_002, 4097, 123456789)]:
        np.testing.assert_array_equal(host.normal_bf16(seed, tid, n, start=start),
                                      gen.normal_bf16(seed, tid, n, start=start))
        np.testing.assert_array_equal(host.uniform_ids(seed, tid, n, 151936, start=start),
                                      gen.uniform_ids(seed, tid, n, 151936, start=start))
    np.testing.assert_array_equal(host.q4_packed(9, 77, 1001), gen.q4_packed(9, 77, 1001))
    np.testing.assert_array_equal(host.q4_scales(9, 77, 999), gen.q4_scales(9, 77, 999, gen.Q4_S0))


def test_normal_weights_have_requested_moments():
    w = gen.bf16_bits_to_f32(host.normal_bf16(0, 42, 2_000_000)).astype(np.float64)
    assert abs(w.mean()) < 1e-4
    assert abs(w.std() - 0.02) < 2e-4


def test_q4_weights_rms_close_to_dense():
    qs, sc = workloads.host_tensor(workloads.MOE35B_Q4, workloads.TensorSpec("t", 99, (64, 2048), workloads.Q4))
    lo = (qs & 0xF).astype(np.float64) - 8
    hi = (qs >> 4).astype(np.float64) - 8
    s = sc.view(np.float16).astype(np.float64)
    rms = np.sqrt(np.mean(np.concatenate([lo.ravel(), hi.ravel()]) ** 2) * np.mean(s ** 2))
    assert 0.017 < rms < 0.023


def test_ids_in_range_and_spread():
    ids = host.uniform_ids(1, workloads.PROMPT_TID, 100_000, 151936)
    assert ids.min() >= 0 and ids.max() < 151936
    assert len(np.unique(ids)) > 70_000


def test_tensor_table_parameter_counts():
    s = workloads.DENSE4B
    specs = {t.name: t for t in workloads.tensor_specs(s)}
    assert specs["l0.w_in"].dims == (3 * 16 * 128 + 2 * 16, 2560)
    assert specs["l3.w_in"].dims == ((16 + 8) * 128, 2560)
    assert "l3.conv_w" not in specs and "l0.conv_w" in specs
    assert sum(1 for l in range(32) if s.is_attn(l)) == 8
    m = workloads.MOE35B
    assert sum(1 for l in range(40) if m.is_attn(l)) == 10
    assert {t.name: t for t in workloads.tensor_specs(m)}["l0.router"].dims == (257, 2048)
