"""Pins of oracle.slots: slot arithmetic and append read back in order."""
import numpy as np

from oracle.attention import gather_sequence
from oracle.block_pool import BlockPool, SequenceTable
from oracle.slots import append_rows, slot_mapping, slot_of


def test_hand_example():
    # logical block 1 of table [7, 2, 9] is physical block 2; position 17 is
    # offset 1 in it -> slot 2 * 16 + 1
    assert slot_of([7, 2, 9], 17) == 33
    assert slot_of([7, 2, 9], 0) == 112
    assert slot_of([7, 2, 9], 47) == 159


def test_negative_position_is_padding():
    out = slot_mapping(np.array([[3, 4]]), [0, 0], [5, -1])
    assert out.tolist() == [3 * 16 + 5, -1]


def test_append_then_gather_reads_back_in_order():
    # what is appended at position p is what a reader of position p sees,
    # whatever physical blocks the pool handed out
    rng = np.random.default_rng(1)
    pool = BlockPool(40)
    pool_order = rng.permutation(40)
    pool._free = [int(i) for i in pool_order]     # scramble the free list
    cache = np.full((40, 2, 16, 8), -1, dtype=np.int64)
    seqs = [SequenceTable(pool) for _ in range(3)]
    written = {i: [] for i in range(3)}
    for step in range(60):
        b = int(rng.integers(3))
        pos = seqs[b].append_tokens(1)[0]
        rows = rng.integers(0, 1 << 30, size=(1, 2, 8))
        slots = slot_mapping({b: seqs[b].blocks}, [b], [pos])
        append_rows(cache, rows, slots)
        written[b].append(rows[0])
    for b in range(3):
        for g in range(2):
            got = gather_sequence(cache, seqs[b].blocks, seqs[b].length, g)
            assert np.array_equal(got, np.stack([w[g] for w in written[b]]))


def test_negative_slot_skipped():
    cache = np.zeros((2, 1, 16, 4), dtype=np.uint16)
    append_rows(cache, np.ones((2, 1, 4), dtype=np.uint16), [-1, 3])
    assert cache.sum() == 4 and cache[0, 0, 3].tolist() == [1, 1, 1, 1]
