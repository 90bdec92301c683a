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


def test_cache_fill_values_follow_their_definition():
    """The cache-fill stream: value i is the top 24 bits of the i-th
    SplitMix64 output of a generator seeded with the key, mapped to
    [-1, 1) * scale; checked element by element through the scalar
    SplitMix64 of this module and exact rational arithmetic."""
    from fractions import Fraction
    key = 123456789 * workloads.FILL_SEED_MULT + 3 * 64 + 1
    v = gen.fill_values(key, 4096, 1.0)
    for i in (0, 1, 2, 77, 4095):
        z = gen.mix64_int(key + (i + 1) * gen.GOLDEN)
        assert Fraction(float(v[i])) == Fraction(z >> 40, 1 << 23) - 1
    assert v.dtype == np.float32 and v.min() >= -1.0 and v.max() < 1.0
    assert abs(float(v.mean())) < 0.05 and abs(float(v.var()) - 1 / 3) < 0.02
    s = gen.fill_values(key, 4096, 0.01)
    np.testing.assert_array_equal(s, v * np.float32(0.01))


def test_synthetic_cache_layout():
    """Host copy of hy_seq_fill_synthetic: one K and one V array per attention
    layer, [nkv, length, hd] bf16 bits, each kv head its own stream from row
    0; the DeltaNet states one stream over [n_gdn, nh, dv, dk]."""
    s = workloads.TINY
    c = workloads.synthetic_cache(s, 37, seed=5)
    assert len(c["k"]) == len(c["v"]) == 1
    assert c["k"][0].shape == (s.attn_kv_heads, 37, s.head_dim) and c["k"][0].dtype == np.uint16
    base = 5 * workloads.FILL_SEED_MULT
    np.testing.assert_array_equal(c["v"][0][1].ravel(),
                                  gen.f32_to_bf16_bits(gen.fill_values(base + 1 * 64 + 1, 37 * s.head_dim)))
    longer = workloads.synthetic_cache(s, 50, seed=5)
    np.testing.assert_array_equal(longer["k"][0][:, :37], c["k"][0])  # rows do not depend on the length
    assert c["state"].shape == (1, s.gdn_heads, s.gdn_dv, s.gdn_dk) and c["state"].dtype == np.float32
    assert np.abs(c["state"]).max() < workloads.FILL_STATE_SCALE
    assert not np.array_equal(workloads.synthetic_cache(s, 37, seed=6)["k"][0], c["k"][0])
