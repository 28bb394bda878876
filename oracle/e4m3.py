"""FP8 E4M3 KV storage (oracle; test infrastructure only).

Sources:

* "KV cache capacity planning ..." section 4: FP8 stores K/V as 8-bit floats;
  E4M3 spends more bits on the mantissa and has the narrower range; a scale
  factor sets the dynamic range (too large wastes resolution on small values,
  too small saturates the outliers); scales may be per tensor or per
  attention head.  Its reference list names the OCP 8-bit floating point
  specification, which defines the format used here.
* Same page, section 5: some kernels store FP8 and dequantise before compute.
* "What a KV cache is ..." section 3.3: E4M3 is 4 exponent bits, 3 mantissa bits.

The OCP E4M3 format: sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
exponent 0 encodes subnormals m/8 * 2^-6; exponent 1..15 encodes
(1 + m/8) * 2^(e-7); S.1111.111 is NaN; there is no infinity, so the largest
finite magnitude is 1.75 * 2^8 = 448 (code 0x7E).

Encoding reading (the pages fix no rounding rule): the stored code for x with
scale s is the E4M3 value nearest to the float32 quotient fl32(x / s), ties to
the even code, and magnitudes above 448 clamp to 448 (saturating, never NaN).
The sign of the quotient is kept, so -0.0 and tiny negatives give 0x80.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def _value_of_code(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** -6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


# value of each of the 256 codes, exactly (every one is a dyadic rational)
E4M3_VALUES = np.array([_value_of_code(c) for c in range(256)], dtype=np.float64)

# the finite non-negative magnitudes in code order 0x00..0x7E (strictly increasing)
_MAGNITUDES = E4M3_VALUES[:0x7F].copy()


def decode(codes) -> np.ndarray:
    """float64 value of each uint8 code (exact table lookup)."""
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


def quotient_f32(x, scale) -> np.ndarray:
    """fl32(fl32(x) / fl32(scale)): one IEEE single-precision division."""
    return np.asarray(x, dtype=np.float32) / np.float32(scale)


def nearest_code(q) -> np.ndarray:
    """Nearest E4M3 code to each float32 ``q`` by exhaustive search over the
    127 finite magnitudes, ties to the even code, saturating at 448."""
    q = np.asarray(q, dtype=np.float32)
    flat = q.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    chunk = 1 << 15
    for s in range(0, flat.size, chunk):
        part = flat[s:s + chunk]
        mag = np.abs(part.astype(np.float64))
        dist = np.abs(mag[:, None] - _MAGNITUDES[None, :])
        best = np.argmin(dist, axis=1)             # first (lower) code on a tie
        nxt = np.minimum(best + 1, 0x7E)
        tie = (nxt != best) & (dist[np.arange(best.size), nxt] == dist[np.arange(best.size), best])
        best = np.where(tie & (best % 2 == 1), nxt, best)   # prefer the even code
        best = np.where(mag >= E4M3_MAX, 0x7E, best)        # saturate (also +-inf)
        code = best.astype(np.uint8) | np.where(np.signbit(part), 0x80, 0).astype(np.uint8)
        code = np.where(np.isnan(part), NAN_CODE, code)
        out[s:s + chunk] = code
    return out.reshape(q.shape)


def encode(x, scale) -> np.ndarray:
    """E4M3 codes for values ``x`` (anything float32 holds exactly, e.g.
    fp16/bf16 inputs) stored with ``scale``: nearest_code(fl32(x / scale))."""
    return nearest_code(quotient_f32(x, scale))
