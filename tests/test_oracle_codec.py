"""Pins of the oracle's E4M3 codec against the format definition and libraries.

E4M3 per the OCP 8-bit floating point specification / "FP8 Formats for Deep
Learning" (bias 7, no infinities, S.1111.111 NaN, max 448); the layer's
contract asks for round-half-to-even with saturation at +-448.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from tests.conftest import GOLDEN


def _finite_codes():
    return [c for c in range(256) if (c & 0x7F) != 0x7F]


def test_exhaustive_round_trip_all_256_codes():
    table = oracle.e4m3_table()
    assert np.isnan(table[0x7F]) and np.isnan(table[0xFF])
    finite = _finite_codes()
    assert len(finite) == 254
    vals = table[finite].astype(np.float32)
    assert np.all(vals.astype(np.float64) == table[finite]), "every E4M3 value is exact in FP32"
    enc = oracle.e4m3_encode(vals)
    assert np.array_equal(enc, np.array(finite, dtype=np.uint8))
    enc2 = oracle.e4m3_encode_arith(vals)
    assert np.array_equal(enc2, np.array(finite, dtype=np.uint8))


def test_magnitudes_are_strictly_increasing_and_span_format():
    t = oracle.e4m3_table()[:0x7F]
    assert np.all(np.diff(t) > 0)
    assert t[0] == 0.0 and t[1] == 2.0 ** -9 and t[0x7E] == 448.0
    assert t[8] == 2.0 ** -6 and t[7] == 0.875 * 2.0 ** -6
    # sign symmetry
    neg = oracle.e4m3_table()[0x80:0xFF]
    assert np.all(neg == -t) or np.all(np.abs(neg) == t)
    assert np.signbit(oracle.e4m3_table()[0x80])


def test_golden_ocp_values():
    path = os.path.join(GOLDEN, "e4m3_ocp_values.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert len(rows) >= 20
    for val_s, code_s in rows:
        v = np.float32(float(val_s))
        code = int(code_s, 16)
        got = int(oracle.e4m3_encode(np.array([v]))[0])
        assert got == code, (val_s, hex(got), code_s)
        dec = oracle.e4m3_decode(np.array([code], dtype=np.uint8))[0]
        assert dec == float(val_s) and np.signbit(dec) == np.signbit(float(val_s))


def test_every_midpoint_rounds_to_even_code():
    t = oracle.e4m3_table()[:0x7F]
    lo = np.arange(0, 0x7E)
    mids = ((t[lo] + t[lo + 1]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (t[lo] + t[lo + 1]) / 2), "midpoints exact in FP32"
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(oracle.e4m3_encode(mids), want)
    assert np.array_equal(oracle.e4m3_encode(-mids), want | 0x80)
    # one FP32 ulp either side of the midpoint decides by distance
    above = np.nextafter(mids, np.float32(np.inf))
    below = np.nextafter(mids, np.float32(0))
    assert np.array_equal(oracle.e4m3_encode(above), (lo + 1).astype(np.uint8))
    assert np.array_equal(oracle.e4m3_encode(below), lo.astype(np.uint8))


def test_saturation_and_specials():
    vals = np.array([448, 449, 463.99, 464, 480, 1e6, np.inf, 3.4e38], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(vals) == 0x7E)
    assert np.all(oracle.e4m3_encode(-vals) == 0xFE)
    nan = oracle.e4m3_encode(np.array([np.nan], dtype=np.float32))[0]
    assert nan & 0x7F == 0x7F
    assert oracle.e4m3_encode(np.array([0.0], dtype=np.float32))[0] == 0x00
    assert oracle.e4m3_encode(np.array([-0.0], dtype=np.float32))[0] == 0x80
    tiny = np.array([1e-30, 2.0 ** -11, 2.0 ** -126, 1e-45], dtype=np.float32)
    assert np.all(oracle.e4m3_encode(tiny) == 0x00)
    assert np.all(oracle.e4m3_encode(-tiny) == 0x80)


def _random_probe_values(n, seed):
    rng = np.random.default_rng(seed)
    mant = rng.uniform(-1, 1, n)
    expo = rng.integers(-14, 10, n)
    v = (mant * np.exp2(expo)).astype(np.float32)
    return v


def test_brute_force_matches_independent_arithmetic_encoder():
    v = _random_probe_values(1 << 20, 11)
    assert np.array_equal(oracle.e4m3_encode(v), oracle.e4m3_encode_arith(v))


def _torch_e4m3_codes(v: np.ndarray) -> np.ndarray:
    # torch's CPU cast rounds half to even but turns |v| > 464 into NaN instead
    # of saturating, so clamp to the finite range first.
    t = torch.from_numpy(np.clip(v, -448, 448).astype(np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_matches_torch_float8_e4m3fn_cast():
    v = _random_probe_values(1 << 20, 12)
    t = oracle.e4m3_table()[:0x7F]
    mids = ((t[:-1] + t[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    assert np.array_equal(oracle.e4m3_encode(v), _torch_e4m3_codes(v))


def test_matches_ml_dtypes_float8_e4m3fn():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    v = _random_probe_values(1 << 18, 13)
    v = np.clip(v, -448, 448)
    got = oracle.e4m3_encode(v)
    ref = v.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(got, ref)
