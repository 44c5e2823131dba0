"""The seeded input generator: published SplitMix64 test vector, determinism,
bf16 rounding, distribution moments and the Zipf bias.  CPU only."""
import math

import numpy as np

import synth


def test_splitmix64_known_answer():
    # Outputs of the SplitMix64 reference implementation (Vigna's splitmix64.c)
    # seeded with 1234567.
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(v) for v in synth.splitmix64(1234567, 0, 5)] == want
    # counter based: a slice equals the same outputs of the full stream
    full = synth.splitmix64(99, 0, 1000)
    assert np.array_equal(synth.splitmix64(99, 637, 100), full[637:737])


def test_normal_moments_and_slices():
    v = synth.normal_f32(7, 2_000_000, 0.5).astype(np.float64)
    assert abs(v.mean()) < 3 * 0.5 / math.sqrt(v.size)
    assert abs(v.std() / 0.5 - 1) < 3e-3
    a = synth.normal(5, (100, 64), 0.1, bf16=True)
    b = synth.normal(5, (40, 64), 0.1, bf16=True, start=30 * 64)
    assert np.array_equal(a[30:70], b)


def test_round_bf16_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e-3],
                 np.float32)
    r = synth.round_bf16(x)
    assert r[0] == 1.0
    assert r[1] == 1.0                      # tie -> even (1.0)
    assert r[2] == 1.0 + 4 * 2 ** -8        # tie -> even (1 + 2^-6)
    assert r[3] == 1.0
    assert r[4] == -2.5
    bits = r.view(np.uint32)
    assert (bits & 0xFFFF == 0).all()
    assert abs(r[5] - 3.0e-3) <= 3.0e-3 * 2 ** -8


def test_zipf_bias_popularity():
    b = synth.zipf_bias(3, 128, 1.1).astype(np.float64)
    pi = np.exp(b)
    assert abs(pi.sum() - 1) < 1e-5
    ranks = np.sort(pi)[::-1]
    want = np.arange(1, 129, dtype=np.float64) ** -1.1
    want /= want.sum()
    assert np.allclose(ranks, want, rtol=1e-5)
    assert sorted(synth.permutation(3, 128)) == list(range(128))


def test_expert_slice_matches_full_tensor():
    w = synth.WORKLOADS["tiny_fp32_n16_k4_d64_f128_b4"]
    L = synth.make_layer(w)
    g, u, dn = synth.make_expert(w, 0, 5)
    assert np.array_equal(g, L["w_gate"][5]) and np.array_equal(u, L["w_up"][5])
    assert np.array_equal(dn, L["w_down"][5])
