"""Pins of oracle.block_pool against the allocator facts the pages state."""
import numpy as np
import pytest

from oracle.block_pool import BlockPool, PoolExhausted, SequenceTable, blocks_needed


def test_prompt_of_1200_tokens_takes_75_blocks():
    # "What a KV cache is ..." section 3.2: 1200 tokens -> 75 blocks of 16
    assert blocks_needed(1200) == 75
    pool = BlockPool(2048)
    seq = SequenceTable(pool)
    seq.append_tokens(1200)
    assert len(seq.blocks) == 75 and pool.num_free == 2048 - 75


def test_preallocated_pool_capacity():
    # same section: 2048 blocks x 16 tokens = 32768 tokens
    assert BlockPool(2048).capacity_tokens == 32768


@pytest.mark.parametrize("seed", range(5))
def test_waste_at_most_one_block(seed):
    # "Series 03" section 3.2: a block is taken only when the current one is
    # full, so the waste is the unused tail of the last block
    rng = np.random.default_rng(seed)
    pool = BlockPool(4096)
    seqs = [SequenceTable(pool) for _ in range(8)]
    for _ in range(200):
        s = seqs[rng.integers(len(seqs))]
        s.append_tokens(int(rng.integers(1, 40)))
    for s in seqs:
        assert len(s.blocks) == -(-s.length // 16)
        assert 0 <= s.wasted_slots() < 16
    used = sum(len(s.blocks) for s in seqs)
    assert pool.num_free == 4096 - used
    ids = [b for s in seqs for b in s.blocks]
    assert len(ids) == len(set(ids))          # no block handed out twice


def test_exhaustion_raises_and_leaves_state():
    # "What a KV cache is ..." section 4.2: overflow is a RuntimeError
    pool = BlockPool(3)
    seq = SequenceTable(pool)
    seq.append_tokens(40)                     # 3 blocks
    with pytest.raises(RuntimeError):
        seq.append_tokens(9)                  # would need a 4th block
    assert seq.length == 40 and len(seq.blocks) == 3
    with pytest.raises(PoolExhausted):
        pool.alloc()


def test_lengths_grow_by_appends():
    # "What a KV cache is ..." section 4.2: 100 prefill tokens + 1 decode = 101;
    # "KV Cache, the memory notepad ..." section 四: 5-token prompt + 3 decode steps = 8
    pool = BlockPool(16)
    a = SequenceTable(pool)
    a.append_tokens(100)
    a.append_tokens(1)
    assert a.length == 101
    b = SequenceTable(pool)
    b.append_tokens(5)
    for _ in range(3):
        b.append_tokens(1)
    assert b.length == 8


def test_shared_prefix_refcounts():
    # "Series 03" section 3.3: several tables reference one physical block;
    # a shared block returns to the pool only when no table references it
    pool = BlockPool(64)
    base = SequenceTable(pool)
    base.append_tokens(32)                    # 2 blocks
    forks = []
    for _ in range(3):
        f = SequenceTable(pool)
        f.share_prefix_from(base, 2)
        f.append_tokens(5)
        forks.append(f)
    for blk in base.blocks:
        assert pool.refcount(blk) == 4
    free_before = pool.num_free
    base.release()
    assert pool.num_free == free_before       # still referenced by the forks
    for f in forks:
        f.release()
    assert pool.num_free == 64


def test_lifo_policy():
    pool = BlockPool(8)
    got = [pool.alloc() for _ in range(3)]
    assert got == [0, 1, 2]
    pool.decref(1)
    assert pool.alloc() == 1
    with pytest.raises(ValueError):
        pool.decref(5)                        # never allocated
