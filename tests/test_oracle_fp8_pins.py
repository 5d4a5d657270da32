"""Pins of the oracle's FP8 (E4M3) codes, append and decode.

The code table is checked against published facts of the OCP E4M3 format
(largest finite 448, smallest normal 2^-6, smallest subnormal 2^-9, 1.0 =
0x38, NaN = S.1111.111, 254 finite non-zero values, monotone in the code),
and the encoder against an exact rational nearest-value search written here
(ties to the even code, saturation past 448).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _magnitudes():
    """The 127 finite E4M3 magnitudes by code 0x00..0x7E, from the bit layout (exact rationals)."""
    out = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        out.append(Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return out


def test_code_table_facts():
    v = oracle.e4m3_value(np.arange(256, dtype=np.uint8))
    assert v[0x38] == 1.0 and v[0x7E] == 448.0 and v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and v[0x80] == 0.0 and np.signbit(v[0x80])
    finite = v[np.isfinite(v)]
    assert len(finite) == 254 and len(set(np.abs(finite[finite != 0]).tolist())) == 126
    assert np.all(np.diff(v[:0x7F]) > 0) and np.array_equal(v[0x80:0xFF], -v[:0x7F])
    assert [Fraction(x) for x in v[:0x7F]] == _magnitudes()


def _nearest(x):
    """Exact nearest finite E4M3 code of fp32 x (ties to the even code, saturating past 448)."""
    mags = _magnitudes()
    a = abs(Fraction(float(x)))
    best = min(range(0x7F), key=lambda c: (abs(mags[c] - a), c & 1))
    return best | (0x80 if np.signbit(x) else 0)


def test_encoder_matches_exact_search():
    mags = [float(m) for m in _magnitudes()]
    mids = [(a + b) / 2 for a, b in zip(mags, mags[1:])]  # every tie
    rng = np.random.default_rng(0)
    xs = np.concatenate([mags, mids, [448.0, 464.0, 470.0, 1e6, 2.0 ** -10, 2.0 ** -11, 0.0],
                         rng.standard_normal(300) * 10.0, rng.standard_normal(200) * 1e-2]).astype(np.float32)
    xs = np.concatenate([xs, -xs])
    got = oracle.e4m3_encode(xs)
    want = np.array([_nearest(x) for x in xs], np.uint8)
    assert np.array_equal(got, want)


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_value(codes).astype(np.float32))
    assert np.array_equal(back, codes)


def test_append_quantises_within_half_a_step():
    rng = np.random.default_rng(3)
    nb, hkv, bs, d = 6, 2, 16, 8
    kn = rng.standard_normal((20, hkv, d)).astype(np.float32)
    vn = (rng.standard_normal((20, hkv, d)) * 3).astype(np.float32)
    kp = np.zeros((nb, hkv, bs, d), np.uint8)
    vp = np.zeros((nb, hkv, bs, d), np.uint8)
    slots = np.array([3 * bs + i for i in range(16)] + [5 * bs + i for i in range(4)], np.int64)
    oracle.reshape_and_cache_fp8(kn, vn, kp, vp, slots, 0.05, 0.2)
    for i, s in enumerate(slots):
        kh = oracle.e4m3_value(kp[s // bs, :, s % bs]) * np.float32(0.05)
        vh = oracle.e4m3_value(vp[s // bs, :, s % bs]) * np.float32(0.2)
        # three mantissa bits: relative error at most 2^-4 in the normal range
        assert np.all(np.abs(kh - kn[i]) <= 2.0 ** -4 * np.abs(kn[i]) + 0.05 * 2.0 ** -10)
        assert np.all(np.abs(vh - vn[i]) <= 2.0 ** -4 * np.abs(vn[i]) + 0.2 * 2.0 ** -10)
    assert np.all(kp[:3] == 0) and np.all(vp[4] == 0)


def test_fp8_decode_closed_forms():
    """One token: the output is exactly its dequantised value row; all keys equal: the mean of the values."""
    rng = np.random.default_rng(5)
    nb, hkv, bs, d, hq = 4, 2, 16, 8, 4
    kp = rng.integers(0, 0x7E, (nb, hkv, bs, d)).astype(np.uint8)
    vp = rng.integers(0, 0x7E, (nb, hkv, bs, d)).astype(np.uint8)
    q = rng.standard_normal((2, hq, d)).astype(np.float32)
    tables = np.array([[2, 0], [1, 3]], np.int32)
    out = oracle.decode_attention_fp8(q, kp, vp, 0.5, 0.25, tables, np.array([1, 20], np.int32), 0.3)
    for h in range(hq):
        assert np.array_equal(out[0, h], oracle.e4m3_value(vp[2, h // 2, 0]) * 0.25)
    kp[1], kp[3] = kp[1, :, :1], kp[1, :, :1]  # every key of sequence 1 the same row
    kp[3] = kp[1, :, :1]
    out = oracle.decode_attention_fp8(q, kp, vp, 0.5, 0.25, tables, np.array([1, 20], np.int32), 0.3)
    vals = np.concatenate([oracle.e4m3_value(vp[1]), oracle.e4m3_value(vp[3])[:, :4]], axis=1) * 0.25
    for h in range(hq):
        assert np.allclose(out[1, h], vals[h // 2].mean(axis=0), rtol=0, atol=1e-12)
