"""FP8 E5M2 KV storage (oracle; test infrastructure only).

Sources:

* "KV cache capacity planning ..." section 4: FP8 stores K/V as 8-bit floats;
  the common formats are E4M3 and E5M2; E5M2 has the wider exponent range and
  the lower precision; a scale factor sets the dynamic range, per tensor or
  per attention head.  Its reference list names the OCP 8-bit floating point
  specification, which defines the format used here.
* Same page, section 5: some kernels store FP8 and dequantise before compute.

The OCP E5M2 format: sign bit, 5 exponent bits with bias 15, 2 mantissa bits;
exponent 0 encodes subnormals m/4 * 2^-14; exponent 1..30 encodes
(1 + m/4) * 2^(e-15); exponent 31 with m = 0 is infinity and with m != 0 is
NaN.  The largest finite magnitude is 1.75 * 2^15 = 57344 (code 0x7B).

Encoding reading (the pages fix no rounding rule; the same reading as for
E4M3): the stored code for x with scale s is the E5M2 value nearest to the
float32 quotient fl32(x / s), ties to the even code; magnitudes above 57344,
infinities included, clamp to 57344 (saturating: a stored K/V is never
infinite); NaN stores the NaN code 0x7F; the sign of the quotient is kept, so
-0.0 and tiny negatives give 0x80.
"""
from __future__ import annotations

import numpy as np

E5M2_MAX = 57344.0
NAN_CODE = 0x7F
_MAX_CODE = 0x7B


def _value_of_code(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 2) & 0x1F
    man = code & 0x3
    if exp == 0x1F:
        return sign * float("inf") if man == 0 else float("nan")
    if exp == 0:
        return sign * (man / 4.0) * 2.0 ** -14
    return sign * (1.0 + man / 4.0) * 2.0 ** (exp - 15)


# value of each of the 256 codes, exactly (every finite one is a dyadic rational)
E5M2_VALUES = np.array([_value_of_code(c) for c in range(256)], dtype=np.float64)

# the finite non-negative magnitudes in code order 0x00..0x7B (strictly increasing)
_MAGNITUDES = E5M2_VALUES[:_MAX_CODE + 1].copy()


def decode(codes) -> np.ndarray:
    """float64 value of each uint8 code (exact table lookup)."""
    return E5M2_VALUES[np.asarray(codes, dtype=np.uint8)]


def quotient_f32(x, scale) -> np.ndarray:
    """fl32(fl32(x) / fl32(scale)): one IEEE single-precision division."""
    return np.asarray(x, dtype=np.float32) / np.float32(scale)


def nearest_code(q) -> np.ndarray:
    """Nearest E5M2 code to each float32 ``q`` by exhaustive search over the
    124 finite magnitudes, ties to the even code, saturating at 57344."""
    q = np.asarray(q, dtype=np.float32)
    flat = q.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    chunk = 1 << 15
    for s in range(0, flat.size, chunk):
        part = flat[s:s + chunk]
        mag = np.abs(part.astype(np.float64))
        with np.errstate(invalid="ignore"):
            dist = np.abs(mag[:, None] - _MAGNITUDES[None, :])
        best = np.argmin(np.nan_to_num(dist, nan=0.0, posinf=np.inf), axis=1)   # lower code on a tie
        nxt = np.minimum(best + 1, _MAX_CODE)
        idx = np.arange(best.size)
        tie = (nxt != best) & (dist[idx, nxt] == dist[idx, best])
        best = np.where(tie & (best % 2 == 1), nxt, best)     # prefer the even code
        best = np.where(mag >= E5M2_MAX, _MAX_CODE, best)     # saturate (also +-inf)
        code = best.astype(np.uint8) | np.where(np.signbit(part), 0x80, 0).astype(np.uint8)
        code = np.where(np.isnan(part), NAN_CODE, code)
        out[s:s + chunk] = code
    return out.reshape(q.shape)


def encode(x, scale) -> np.ndarray:
    """E5M2 codes for values ``x`` (anything float32 holds exactly, e.g.
    fp16/bf16 inputs) stored with ``scale``: nearest_code(fl32(x / scale))."""
    return nearest_code(quotient_f32(x, scale))
