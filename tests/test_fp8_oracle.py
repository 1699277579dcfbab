"""Pins of the E4M3 / E5M2 oracle (oracle/fp8.py) against the formats'
definitions: fixed points of the encodings, exhaustive round trips, ties to
even, saturation, brute-force nearest values, and the scaling reading."""
import numpy as np
import pytest

from oracle import fp8 as F


@pytest.mark.parametrize("fmt,byte,value", [
    ("e4m3", 0x7E, 448.0), ("e4m3", 0x01, 2.0 ** -9), ("e4m3", 0x08, 2.0 ** -6),
    ("e4m3", 0x38, 1.0), ("e4m3", 0xC0, -2.0), ("e4m3", 0x3C, 1.5), ("e4m3", 0x00, 0.0),
    ("e5m2", 0x7B, 57344.0), ("e5m2", 0x01, 2.0 ** -16), ("e5m2", 0x04, 2.0 ** -14),
    ("e5m2", 0x3C, 1.0), ("e5m2", 0xBE, -1.5), ("e5m2", 0x40, 2.0),
])
def test_fixed_points_of_the_encodings(fmt, byte, value):
    assert F.decode(np.array([byte]), fmt)[0] == value
    assert F.encode(np.array([value]), fmt)[0] == byte


def _finite_bytes(fmt):
    b = np.arange(256, dtype=np.uint8)
    if fmt == "e4m3":  # S.1111.111 is NaN
        return b[(b & 0x7F) != 0x7F]
    return b[(b & 0x7C) != 0x7C]  # E5M2 exponent 11111: infinities and NaNs


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_every_finite_byte_round_trips(fmt):
    b = _finite_bytes(fmt)
    assert np.array_equal(F.encode(F.decode(b, fmt), fmt), b)
    assert np.array_equal(F.round_fp8(F.decode(b, fmt), fmt), F.decode(b, fmt))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_rounding_is_to_the_nearest_value_ties_to_even(fmt):
    vals = np.unique(F.decode(_finite_bytes(fmt), fmt))
    rng = np.random.default_rng(0)
    fmax = F.FORMATS[fmt][2]
    x = np.concatenate([rng.uniform(-fmax, fmax, 4000),
                        rng.standard_normal(4000) * 2.0 ** rng.integers(-18, 4, 4000)])
    r = F.round_fp8(x, fmt)
    d = np.abs(x[:, None] - vals[None, :])
    best = d.min(axis=1)
    assert np.array_equal(np.abs(x - r), best)  # r is a nearest value
    # ties: the midpoints between neighbours go to the one with the even mantissa
    mids = (vals[1:] + vals[:-1]) / 2
    rm = F.round_fp8(mids, fmt)
    codes = F.encode(rm, fmt)
    assert np.all((codes & 1) == 0)


def test_specific_roundings():
    e = lambda v: F.round_fp8(np.array([v]), "e4m3")[0]  # noqa: E731
    assert e(1.0625) == 1.0          # halfway 1 | 1.125 -> even mantissa
    assert e(1.1875) == 1.25         # halfway 1.125 | 1.25 -> even
    assert e(1.07) == 1.125
    assert e(500.0) == 448.0 and e(-1e9) == -448.0   # saturation
    assert e(2.0 ** -10) == 0.0      # half the smallest subnormal -> even (0)
    assert e(3 * 2.0 ** -10) == 2.0 ** -8
    assert F.round_fp8(np.array([60000.0]), "e5m2")[0] == 57344.0


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_quantize_maps_amax_to_fmax_and_scales_back(fmt):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(5000) * 3.0).astype(np.float32)
    q, sinv = F.quantize(x, fmt)
    v = F.decode(q, fmt)
    fmax = F.FORMATS[fmt][2]
    assert np.max(np.abs(v)) == fmax
    # relative error of the dequantised values: one rounding to m bits
    m = F.FORMATS[fmt][0]
    big = np.abs(x) > np.max(np.abs(x)) * 2.0 ** -5
    rel = np.abs(v[big] * sinv - x[big]) / np.abs(x[big])
    assert rel.max() <= 2.0 ** -(m + 1) * (1 + 1e-6)
    assert F.quantize(np.zeros(8, np.float32), fmt)[1] == 1.0


def test_gemm_is_the_product_of_the_decoded_operands():
    rng = np.random.default_rng(2)
    a, sa = F.quantize(rng.standard_normal((5, 7)).astype(np.float32), "e4m3")
    b, sb = F.quantize(rng.standard_normal((3, 7)).astype(np.float32), "e5m2")
    c = F.gemm_fp8(a, "e4m3", sa, b, "e5m2", sb)
    A, B = F.decode(a, "e4m3"), F.decode(b, "e5m2")
    for i in range(5):
        for j in range(3):
            ref = sum(A[i, k] * B[j, k] for k in range(7)) * float(sa) * float(sb)
            assert abs(c[i, j] - ref) <= 1e-12 * max(1.0, abs(ref))
