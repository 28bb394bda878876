"""Exact float64 values of stored 16-bit bit patterns (oracle; test infrastructure only).

fp16 and bf16 values are exactly representable in float64, so the oracle
works on exact inputs.  bf16 is the upper half of an IEEE float32: shifting
the 16 bits left by 16 gives the float32 with the same value.
"""
from __future__ import annotations

import numpy as np


def f16_bits_to_f64(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_f64(bits) -> np.ndarray:
    wide = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return wide.view(np.float32).astype(np.float64)


def bits_to_f64(bits, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return f16_bits_to_f64(bits)
    if dtype == "bf16":
        return bf16_bits_to_f64(bits)
    raise ValueError(f"unknown 16-bit dtype {dtype!r}")
