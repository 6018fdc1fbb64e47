"""Pins for the seeded input generator (CPU side)."""
import json
import os

import numpy as np

import synth
from tests.conftest import GOLDEN


def test_splitmix64_published_vector():
    g = json.load(open(os.path.join(GOLDEN, "splitmix64_seed0.json")))
    w = synth.words(0, 0, 0, 3)
    assert [int(x) for x in w] == [int(h, 16) for h in g["outputs_hex"]]


def test_slices_are_consistent():
    a = synth.normal(3, synth.STREAM_K, 0, 1000)
    b = synth.normal(3, synth.STREAM_K, 400, 200)
    np.testing.assert_array_equal(a[400:600], b)
    c = synth.normal(3, synth.STREAM_V, 0, 1000)
    assert not np.array_equal(a, c)


def test_normal_moments_and_support():
    z = synth.normal(1, synth.STREAM_Q, 0, 400_000)
    assert abs(z.mean()) < 0.01 and abs(z.var() - 1.0) < 0.01
    assert np.abs(z).max() < 3.47
    y = synth.normal(1, synth.STREAM_LSE, 0, 400_000, mu=10.0, sigma=2.0)
    assert abs(y.mean() - 10.0) < 0.02 and abs(y.std() - 2.0) < 0.02


def test_bernoulli_rate():
    b = synth.bernoulli(2, synth.STREAM_LSE_DROP, 0, 1_000_000, 0.05)
    assert abs(b.mean() - 0.05) < 0.002


def test_f16_pack_word():
    g = json.load(open(os.path.join(GOLDEN, "pack_f16.json")))
    bits = synth.round_to(np.array(g["values"], dtype=np.float32), "f16")
    word = int(bits[0]) | (int(bits[1]) << 16)
    assert word == int(g["packed_word_hex"], 16)


def test_bf16_round_to_nearest_even():
    # 1 + 2^-8 is exactly halfway between bf16 neighbours 1 and 1 + 2^-7: ties to even (1.0)
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 (odd mantissa) and 1 + 2^-6: rounds up
    x = np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -(1.0 + 2**-8), 1.0 + 2**-8 + 2**-20, 0.0, -0.0],
                 dtype=np.float32)
    got = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x))
    np.testing.assert_array_equal(got, np.array([1.0, 1.0 + 2**-6, -1.0, 1.0 + 2**-7, 0.0, -0.0],
                                                 dtype=np.float32))
    assert np.signbit(got[5])


def test_lse_partials_masks():
    P, RH = 8, 50_000
    lse = synth.lse_partials(5, P, RH)
    dead_rows = np.all(np.isneginf(lse), axis=0)
    frac_dead_entries = np.isneginf(lse).mean()
    assert 0.04 < frac_dead_entries < 0.06
    row_drawn = synth.bernoulli(5, synth.STREAM_ROW_DROP, 0, RH, 0.001)
    assert np.all(dead_rows[row_drawn])
    part = synth.lse_partials(5, P, RH, start_rh=1000, count_rh=77)
    np.testing.assert_array_equal(part, lse[:, 1000:1077])
