"""Pins of the seeded input generator (the module both sides draw inputs from)."""
import math

import numpy as np

import synth
from golden_io import lines


def test_splitmix64_published_outputs():
    parts = list(lines("splitmix64.txt"))
    seed = int(parts[0][1])
    expected = [int(p[1], 16) for p in parts[1:]]
    assert [synth.u64(seed, i) for i in range(len(expected))] == expected


def test_uniform_is_top_53_bits():
    for c in range(5):
        x = synth.u64(123, c)
        assert synth.uniform(123, c) == (x >> 11) * 2.0**-53


def test_fills_are_counter_based_and_thread_invariant():
    seed = synth.stream_seed(7, 3)
    full = synth.normal(seed, 3_000_000, "f32")  # several threads
    part = synth.normal(seed, 1000, "f32", offset=2_500_000)  # one thread, offset
    assert np.array_equal(full[2_500_000:2_501_000], part)
    b16 = synth.normal(seed, 1000, "bf16", offset=2_500_000)
    # bf16 bits are the RNE rounding of the same fp32 values
    f = part.view(np.uint32).astype(np.uint64)
    rne = ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(b16, rne)


def test_normal_moments():
    x = synth.normal(synth.stream_seed(11, 2), 2_000_000, "f64")
    assert abs(x.mean()) < 5e-3
    assert abs(x.var() - 1.0) < 5e-3
    kurt = ((x - x.mean()) ** 4).mean() / x.var() ** 2
    assert abs(kurt - 3.0) < 0.05


def test_length_mix_shape():
    n = 200_000
    lens = synth.lengths_mix(synth.stream_seed(5, 1), n)
    short = (lens >= 32) & (lens <= 511)
    mid = (lens >= 512) & (lens <= 2047)
    long_ = (lens >= 2048) & (lens <= 4095)
    assert np.all(short | mid | long_)
    for frac, want in ((short.mean(), 0.70), (mid.mean(), 0.25), (long_.mean(), 0.05)):
        assert abs(frac - want) < 4 * math.sqrt(want * (1 - want) / n)
    # within a component the draw is uniform: residues mod 16 are flat
    counts = np.bincount(lens % 16, minlength=16) / n
    assert np.all(np.abs(counts - 1 / 16) < 0.005)


def test_permutation():
    p = synth.permutation(99, 1000)
    assert sorted(p.tolist()) == list(range(1000))
    assert not np.array_equal(p, np.arange(1000))
    assert np.array_equal(p, synth.permutation(99, 1000))
