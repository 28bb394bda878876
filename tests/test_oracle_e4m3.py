"""Pins of oracle.e4m3 against the OCP E4M3 definition and a library cast."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import e4m3
from tests.conftest import GOLDEN

with open(os.path.join(GOLDEN, "e4m3_ocp_values.json")) as f:
    OCP = json.load(f)


@pytest.mark.parametrize("e", OCP["values"], ids=lambda e: e["name"])
def test_named_values(e):
    v = e4m3.decode([e["code"]])[0]
    assert v == e["value"] and np.signbit(v) == np.signbit(e["value"])
    assert int(e4m3.encode(np.float32(e["value"]), 1.0)) == e["code"]


def test_nan_codes():
    for c in OCP["nan_codes"]:
        assert np.isnan(e4m3.decode([c])[0])
    assert int(e4m3.encode(np.float32("nan"), 1.0)) == e4m3.NAN_CODE


def test_all_finite_codes_round_trip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3.decode(codes).astype(np.float32)
    assert np.array_equal(e4m3.encode(vals, 1.0), codes)


def test_positive_codes_strictly_increase():
    vals = e4m3.decode(np.arange(0x7F))
    assert np.all(np.diff(vals) > 0)
    assert np.array_equal(e4m3.decode(np.arange(0x80, 0xFF)), -vals)


def test_saturation_and_infinities():
    big = np.array([448.0, 449.0, 464.0, 480.0, 1e6, np.inf], dtype=np.float32)
    assert np.all(e4m3.encode(big, 1.0) == 0x7E)
    assert np.all(e4m3.encode(-big, 1.0) == 0xFE)


def test_ties_go_to_even_code():
    cases = {
        2.0 ** -10: 0x00,          # half of the smallest subnormal -> 0
        3 * 2.0 ** -10: 0x02,      # between 0x01 and 0x02
        1.0625: 0x38,              # between 1.0 (0x38) and 1.125 (0x39)
        1.1875: 0x3A,              # between 1.125 (0x39) and 1.25 (0x3A)
        432.0: 0x7E,               # between 416 (0x7D) and 448 (0x7E)
    }
    for x, code in cases.items():
        assert int(e4m3.encode(np.float32(x), 1.0)) == code, x
        assert int(e4m3.encode(np.float32(-x), 1.0)) == code | 0x80, x


def test_sign_of_zero_kept():
    assert int(e4m3.encode(np.float32(-0.0), 1.0)) == 0x80
    assert int(e4m3.encode(np.float32(-1e-9), 1.0)) == 0x80


def test_quotient_is_single_precision():
    # 1/3 in float32 is 0.33333334; the nearest E4M3 value is 0.34375
    # (exponent field 5, mantissa 3 -> 0x2B), computed by hand from the format
    assert int(e4m3.encode(np.float32(1.0), 3.0)) == 0x2B
    q = e4m3.quotient_f32(np.float32(1.0), 3.0)
    assert q.dtype == np.float32 and q == np.float32(1.0) / np.float32(3.0)


def test_matches_library_cast_in_range():
    # within +-448 round-to-nearest-even needs no saturation rule, so the
    # exhaustive search must agree with the library's float8_e4m3fn cast
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * 60,
        rng.standard_normal(50000).astype(np.float32) * 0.01,
        (e4m3.decode(np.arange(0x7E)) + e4m3.decode(np.arange(1, 0x7F))).astype(np.float32) / 2,
    ])
    x = x[np.abs(x) <= 448]
    ours = e4m3.nearest_code(x)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)
