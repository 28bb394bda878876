"""Pins of oracle.e5m2 against the OCP E5M2 definition, the IEEE half
precision format it truncates, and a library cast."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import e5m2
from tests.conftest import GOLDEN

with open(os.path.join(GOLDEN, "e5m2_ocp_values.json")) as f:
    OCP = json.load(f)

FINITE = np.array([c for c in range(256) if (c & 0x7F) <= 0x7B], dtype=np.uint8)


@pytest.mark.parametrize("e", OCP["values"], ids=lambda e: e["name"])
def test_named_values(e):
    v = e5m2.decode([e["code"]])[0]
    assert v == e["value"] and np.signbit(v) == np.signbit(e["value"])
    assert int(e5m2.encode(np.float32(e["value"]), 1.0)) == e["code"]


def test_infinity_and_nan_codes():
    for c, name in OCP["infinity_codes"].items():
        assert e5m2.decode([int(c)])[0] == float(name)
    for c in OCP["nan_codes"]:
        assert np.isnan(e5m2.decode([c])[0])
    assert int(e5m2.encode(np.float32("nan"), 1.0)) == e5m2.NAN_CODE


def test_table_is_the_upper_byte_of_ieee_half():
    # E5M2 has the sign, exponent width and bias of IEEE binary16 and keeps
    # its two leading mantissa bits: code c is the half-precision number with
    # bit pattern c << 8 (numpy's float16 decodes it independently)
    half = (np.arange(256, dtype=np.uint16) << 8).view(np.float16).astype(np.float64)
    same = (half == e5m2.E5M2_VALUES) | (np.isnan(half) & np.isnan(e5m2.E5M2_VALUES))
    assert same.all()
    assert np.array_equal(np.signbit(half[~np.isnan(half)]), np.signbit(e5m2.E5M2_VALUES[~np.isnan(half)]))


def test_all_finite_codes_round_trip():
    vals = e5m2.decode(FINITE).astype(np.float32)
    assert np.array_equal(e5m2.encode(vals, 1.0), FINITE)


def test_positive_codes_strictly_increase():
    vals = e5m2.decode(np.arange(0x7C))
    assert np.all(np.diff(vals) > 0)
    assert np.array_equal(e5m2.decode(np.arange(0x80, 0xFC)), -vals)


def test_saturation_and_infinities():
    big = np.array([57344.0, 57345.0, 61439.0, 61440.0, 65536.0, 1e30, np.inf], dtype=np.float32)
    assert np.all(e5m2.encode(big, 1.0) == 0x7B)
    assert np.all(e5m2.encode(-big, 1.0) == 0xFB)


def test_ties_go_to_even_code():
    cases = {
        2.0 ** -17: 0x00,          # half of the smallest subnormal -> 0
        3 * 2.0 ** -17: 0x02,      # between 0x01 (2^-16) and 0x02 (2^-15)
        1.125: 0x3C,               # between 1.0 (0x3C) and 1.25 (0x3D)
        1.375: 0x3E,               # between 1.25 (0x3D) and 1.5 (0x3E)
        53248.0: 0x7A,             # between 49152 (0x7A) and 57344 (0x7B)
    }
    for x, code in cases.items():
        assert int(e5m2.encode(np.float32(x), 1.0)) == code, x
        assert int(e5m2.encode(np.float32(-x), 1.0)) == code | 0x80, x


def test_sign_of_zero_kept():
    assert int(e5m2.encode(np.float32(-0.0), 1.0)) == 0x80
    assert int(e5m2.encode(np.float32(-1e-12), 1.0)) == 0x80


def test_quotient_is_single_precision():
    # 1/3 in float32 is 0.33333334; the E5M2 neighbours are 0.3125 (exponent
    # field 13, mantissa 1 -> 0x35) and 0.375 (0x36): the nearest is 0x35,
    # computed by hand from the format
    assert int(e5m2.encode(np.float32(1.0), 3.0)) == 0x35
    q = e5m2.quotient_f32(np.float32(1.0), 3.0)
    assert q.dtype == np.float32 and q == np.float32(1.0) / np.float32(3.0)


def test_matches_library_cast_in_range():
    # within +-57344 round-to-nearest-even needs no saturation rule, so the
    # exhaustive search must agree with the library's float8_e5m2 cast
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 3000,
        rng.standard_normal(50000).astype(np.float32) * 1e-4,
        (e5m2.decode(np.arange(0x7B)) + e5m2.decode(np.arange(1, 0x7C))).astype(np.float32) / 2,
    ])
    x = x[np.abs(x) <= 57344]
    ours = e5m2.nearest_code(x)
    lib = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)
