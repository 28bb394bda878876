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


def encode_slabs(values: np.ndarray):
    """Codes (uint8, same shape) and per-slab (min, max) as float32 for a
    stack of slabs ``values`` [..., rows, d] (every row holds a token): each
    slab [rows, d] is encoded on its own with the formula above, its min and
    max taken over that slab alone."""
    x = np.asarray(values, dtype=F32)
    lo = x.min(axis=(-2, -1), keepdims=True)
    hi = x.max(axis=(-2, -1), keepdims=True)
    span = (hi - lo).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((x - lo) / span) * F32(255.0)      # float32 ops, left to right
    q = np.clip(np.rint(t), 0, 255)
    q = np.where(span == 0, 0, q).astype(np.uint8)
    return q, lo[..., 0, 0], hi[..., 0, 0]


def encode_rows(values: np.ndarray):
    """Codes [rows, d] (uint8) and (min, max) as float32 for the float32 rows
    ``values`` (all of them hold tokens): one slab of ``encode_slabs``."""
    q, lo, hi = encode_slabs(np.asarray(values, dtype=F32)[None])
    return q[0], F32(lo[0]), F32(hi[0])


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
    block hold tokens; the rest get code 0 (and a block with none gets
    (0, 0)).  Blocks with the same number of used rows are encoded together
    (slab by slab, as ``encode_slabs`` does)."""
    nb, nh, bs, d = pool_f32.shape
    codes = np.zeros(pool_f32.shape, dtype=np.uint8)
    params = np.zeros((nb, nh, 2), dtype=F32)
    used = np.full(nb, bs) if rows_used is None else np.asarray(rows_used).astype(np.int64)
    for n in np.unique(used):
        n = int(n)
        if n == 0:
            continue
        blks = np.nonzero(used == n)[0]
        for s in range(0, blks.size, 1024):    # bounded temporaries
            part = blks[s:s + 1024]
            q, lo, hi = encode_slabs(pool_f32[part, :, :n])
            codes[part, :, :n] = q
            params[part, :, 0] = lo
            params[part, :, 1] = hi
    return codes, params


def append_row(codes: np.ndarray, params: np.ndarray, blk: int, head: int, row: int, new_row) -> None:
    """Write the float32 ``new_row`` at ``row`` of block ``blk``, head
    ``head``, re-quantising rows 0..row of that slab in place."""
    old = decode_f32(codes[blk, head, :row], params[blk, head, 0], params[blk, head, 1])
    rows = np.concatenate([old, np.asarray(new_row, dtype=F32)[None]], axis=0)
    q, lo, hi = encode_rows(rows)
    codes[blk, head, :row + 1] = q
    params[blk, head] = (lo, hi)
