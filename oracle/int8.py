"""INT8 KV cache with per-block min-max scaling (oracle; test infrastructure only).

Source: "What a KV cache is ..." section 3.3: each block's K (and V) is
quantised as

    q = round((k - k_min) / (k_max - k_min) * 255)

with the block's own k_min / k_max kept beside it (two scalars per block,
about 0.2 % extra memory).

Readings (the pages fix none of these):
* Granularity: one (min, max) pair per (physical block, KV head), for K and
  for V separately -- a block's slab of 16 tokens x head_dim of one head.  At
  d = 128 two 16-bit scalars per 2 KiB slab are the pages' 0.2 %; they are
  kept here as float32, stored per slab as (k_min, k_max, v_min, v_max).
* Only the rows that hold tokens enter min and max; the other rows of the
  block have code 0.
* Arithmetic in float32, in the formula's order, IEEE round to nearest:
  t = ((x - min) / (max - min)) * 255, q = round half to even of t, clamped to
  [0, 255]; max == min gives q = 0.  x is the float32 value of the 16-bit input.
* Decode for attention: min + q (max - min) / 255, exactly (float64 here).
* Appending a token to a block re-quantises it: the existing codes are first
  decoded in float32 as min + ((q * (max - min)) / 255) (in that order), the new
  row is added, min and max are taken over the block's rows so far, and
  every row is encoded again.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def encode_rows(values: np.ndarray):
    """Codes [rows, d] (uint8) and (min, max) as float32 for the float32 rows
    ``values`` (all of them hold tokens)."""
    x = np.asarray(values, dtype=F32)
    lo, hi = F32(x.min()), F32(x.max())
    span = F32(hi - lo)
    if span == 0:
        return np.zeros(x.shape, dtype=np.uint8), lo, hi
    t = ((x - lo) / span) * F32(255.0)          # float32 ops, left to right
    q = np.clip(np.rint(t), 0, 255).astype(np.uint8)
    return q, lo, hi


def decode_f64(codes: np.ndarray, lo, hi) -> np.ndarray:
    """Dequantised values for attention: min + q (max - min) / 255 in float64."""
    lo, hi = float(lo), float(hi)
    return lo + codes.astype(np.float64) * (hi - lo) / 255.0


def decode_f32(codes: np.ndarray, lo, hi) -> np.ndarray:
    """The float32 decode used before re-quantising: min + ((q * span) / 255)."""
    span = F32(F32(hi) - F32(lo))
    return F32(lo) + (codes.astype(F32) * span) / F32(255.0)


def quantize_pool(pool_f32: np.ndarray, rows_used=None):
    """Quantise a float32 pool [NB, H, 16, d]: codes [NB, H, 16, d] and
    params [NB, H, 2] (min, max).  rows_used[blk] (default 16) rows of each
    block hold tokens; the rest get code 0."""
    nb, nh, bs, d = pool_f32.shape
    codes = np.zeros(pool_f32.shape, dtype=np.uint8)
    params = np.zeros((nb, nh, 2), dtype=F32)
    for blk in range(nb):
        n = bs if rows_used is None else int(rows_used[blk])
        if n == 0:
            continue
        for h in range(nh):
            q, lo, hi = encode_rows(pool_f32[blk, h, :n])
            codes[blk, h, :n] = q
            params[blk, h] = (lo, hi)
    return codes, params


def append_row(codes: np.ndarray, params: np.ndarray, blk: int, head: int, row: int, new_row) -> None:
    """Write the float32 ``new_row`` at ``row`` of block ``blk``, head
    ``head``, re-quantising rows 0..row of that slab in place."""
    old = decode_f32(codes[blk, head, :row], params[blk, head, 0], params[blk, head, 1])
    rows = np.concatenate([old, np.asarray(new_row, dtype=F32)[None]], axis=0)
    q, lo, hi = encode_rows(rows)
    codes[blk, head, :row + 1] = q
    params[blk, head] = (lo, hi)
