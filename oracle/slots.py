"""Slot mapping and append (oracle; test infrastructure only).

A token at logical position p of a sequence lives in logical block p // bs at
offset p % bs ("Series 03: why the KV cache eats memory ..." section 3.1: the
block table maps logical block i to a physical block).  Its physical slot in
the pool is therefore table[p // bs] * bs + p % bs; the cache tensor
(num_blocks, kv_heads, block_size, head_dim) stores that slot's row for head h
at [slot // bs, h, slot % bs, :].  The pages never write the formula; it is the
plainest reading of a block table over fixed-size blocks.

Appending ("KV Cache, the memory notepad ..." section 三: each decode step
appends the new token's K and V to the cache) is a bit copy of the new rows
into their slots; a negative slot means "skip this row".
"""
from __future__ import annotations

import numpy as np


def slot_of(table_row, position: int, block_size: int = 16) -> int:
    """Physical slot of logical ``position`` for one sequence's table row."""
    logical_block, offset = divmod(position, block_size)
    return int(table_row[logical_block]) * block_size + offset


def slot_mapping(block_tables, seq_idx, positions, block_size: int = 16) -> np.ndarray:
    """Slots for tokens t = 0..T-1, token t belonging to sequence
    ``seq_idx[t]`` at logical position ``positions[t]``.  A negative
    position gives slot -1 (a padding token that is not written)."""
    out = np.empty(len(positions), dtype=np.int64)
    for t, (b, p) in enumerate(zip(seq_idx, positions)):
        out[t] = -1 if p < 0 else slot_of(block_tables[b], int(p), block_size)
    return out


def append_rows(cache: np.ndarray, new_rows: np.ndarray, slots) -> None:
    """Write new_rows[t, h, :] to cache[slot // bs, h, slot % bs, :] for every
    token t with a non-negative slot.  Works on raw bit patterns (any dtype),
    so the copy is exact by construction."""
    block_size = cache.shape[2]
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), block_size)
        cache[blk, :, off, :] = new_rows[t]


def copy_blocks(cache: np.ndarray, pairs) -> None:
    """Copy-on-write data movement: for each (src, dst) in order, physical
    block dst of the cache takes the contents of block src, all heads and all
    rows ("Series 03 ..." section 3.3: the old block's contents are copied
    into the newly taken block).  Raw bit patterns, so exact by construction."""
    for src, dst in pairs:
        cache[int(dst)] = cache[int(src)]
