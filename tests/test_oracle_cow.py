"""Pins of the oracle's copy-on-write ("Series 03 ..." section 3.3) and
agreement of the C-ABI host pool's copy-on-write with it (no GPU needed).

Section 3.3: block tables of several sequences may point at one physical
block; beam-search branches share the prefix blocks without copying, and only
when a branch writes its first token of its own into a shared block is a new
block taken, the old contents copied and the token written there, while the
other branches keep the old block.  Parallel samples share the prompt the
same way, so the common prefix is stored once plus small increments.
"""
import numpy as np
import pytest

from oracle import attention as oa
from oracle import slots as osl
from oracle.block_pool import BlockPool, PoolExhausted, SequenceTable


def _prompt(pool, n):
    s = SequenceTable(pool)
    s.append_tokens(n)
    return s


def test_fork_shares_without_copying():
    pool = BlockPool(32)
    parent = _prompt(pool, 40)                  # 3 blocks, the last one partial
    free0 = pool.num_free
    kids = [parent.fork() for _ in range(3)]
    assert pool.num_free == free0               # nothing allocated, nothing copied
    for k in kids:
        assert k.blocks == parent.blocks and k.length == parent.length
    assert all(pool.refcount(b) == 4 for b in parent.blocks)


def test_first_divergent_write_copies_and_last_sharer_writes_in_place():
    pool = BlockPool(32)
    parent = _prompt(pool, 40)
    kids = [parent.fork() for _ in range(2)]
    shared_last = parent.blocks[2]
    seqs = kids + [parent]
    pairs = []
    for s in seqs:
        (pos,) = s.append_tokens(1)            # position 40 lies in the shared third block
        pairs.append(s.prepare_write(pos))
    # the first two writers copy, the last one keeps the (now private) block
    assert pairs[0] is not None and pairs[1] is not None and pairs[2] is None
    assert pairs[0][0] == pairs[1][0] == shared_last
    assert pairs[0][1] != pairs[1][1] and shared_last not in (pairs[0][1], pairs[1][1])
    assert parent.blocks[2] == shared_last and pool.refcount(shared_last) == 1
    assert kids[0].blocks[2] == pairs[0][1] and kids[1].blocks[2] == pairs[1][1]
    # full prefix blocks stay shared
    assert all(pool.refcount(b) == 3 for b in parent.blocks[:2])
    assert [kid.blocks[:2] for kid in kids] == [parent.blocks[:2]] * 2


def test_private_block_needs_no_copy():
    pool = BlockPool(8)
    s = _prompt(pool, 5)
    (pos,) = s.append_tokens(1)
    assert s.prepare_write(pos) is None and pool.num_free == 7


def test_copy_on_write_exhaustion_changes_nothing():
    pool = BlockPool(1)
    s = _prompt(pool, 5)
    t = s.fork()
    with pytest.raises(PoolExhausted):
        t.prepare_write(5)
    assert t.blocks == s.blocks and pool.refcount(s.blocks[0]) == 2 and pool.num_free == 0


def test_copy_blocks_moves_all_heads_and_rows_bitwise():
    rng = np.random.default_rng(0)
    cache = rng.integers(0, 2 ** 16, size=(6, 2, 16, 8), dtype=np.uint16)
    before = cache.copy()
    osl.copy_blocks(cache, [(1, 4), (3, 5)])
    assert np.array_equal(cache[4], before[1]) and np.array_equal(cache[5], before[3])
    assert np.array_equal(cache[:4], before[:4])


@pytest.mark.parametrize("prompt_len", [37, 48, 5])
def test_beam_search_through_shared_blocks_equals_each_beams_history(prompt_len):
    # Brute force: every beam's attention over the paged cache (with sharing
    # and copy-on-write) equals attention over that beam's own token history
    # kept contiguously, step after step.
    rng = np.random.default_rng(prompt_len)
    n_kv, n_q, d, scale = 2, 4, 8, 8 ** -0.5
    pool = BlockPool(64)
    k_cache = np.full((64, n_kv, 16, d), np.nan)
    v_cache = np.full((64, n_kv, 16, d), np.nan)

    def write(seq, pos, k_row, v_row):
        slot = osl.slot_of(seq.blocks, pos)
        osl.append_rows(k_cache, k_row[None], [slot])
        osl.append_rows(v_cache, v_row[None], [slot])

    prompt = SequenceTable(pool)
    history = []
    for pos in prompt.append_tokens(prompt_len):
        k_row, v_row = rng.normal(size=(n_kv, d)), rng.normal(size=(n_kv, d))
        write(prompt, pos, k_row, v_row)
        history.append((k_row, v_row))
    beams = [prompt] + [prompt.fork() for _ in range(3)]
    hist = [list(history) for _ in beams]
    for _ in range(20):
        for i, beam in enumerate(beams):
            (pos,) = beam.append_tokens(1)
            pair = beam.prepare_write(pos)
            if pair is not None:
                osl.copy_blocks(k_cache, [pair])
                osl.copy_blocks(v_cache, [pair])
            k_row, v_row = rng.normal(size=(n_kv, d)), rng.normal(size=(n_kv, d))
            write(beam, pos, k_row, v_row)
            hist[i].append((k_row, v_row))
        for i, beam in enumerate(beams):
            q = rng.normal(size=(n_q, d))
            paged = oa.paged_decode_attention(q[None], k_cache, v_cache, [beam.blocks], [beam.length], scale)[0]
            ks = np.stack([k for k, _ in hist[i]])
            vs = np.stack([v for _, v in hist[i]])
            assert np.array_equal(paged, oa.contiguous_decode_attention(q, ks, vs, scale))
    # the prompt's full blocks are stored once for all beams; the rest is private
    full = prompt_len // 16
    per_beam = -(-(prompt_len + 20) // 16) - full
    assert pool.num_free == 64 - full - len(beams) * per_beam
    assert all(pool.refcount(b) == len(beams) for b in prompt.blocks[:full])


# ---------------------------------------------------------------------------
# the C-ABI host pool against the oracle
# ---------------------------------------------------------------------------
def _c_table(seqs, max_blocks):
    t = np.full((len(seqs), max_blocks), -1, dtype=np.int32)
    for i, s in enumerate(seqs):
        t[i, :len(s.blocks)] = s.blocks
    return t


@pytest.mark.parametrize("seed", range(6))
def test_c_prepare_append_matches_oracle(seed):
    pkv = pytest.importorskip("paged_kv_cache_153_gb300")
    rng = np.random.default_rng(seed)
    nb, max_blocks = 160, 12
    opool, cpool = BlockPool(nb), pkv.BlockPool(nb)
    seqs = []
    # prompts, allocated the same way on both sides
    for _ in range(4):
        n = int(rng.integers(1, 70))
        s = SequenceTable(opool)
        s.append_tokens(n)
        for b in s.blocks:
            assert cpool.alloc() == b
        seqs.append(s)
    # beams: forks of random sequences (incref on the C side)
    for _ in range(6):
        src = seqs[int(rng.integers(len(seqs)))]
        seqs.append(src.fork())
        for b in src.blocks:
            cpool.incref(b)
    for _ in range(25):
        pick = sorted(rng.choice(len(seqs), size=int(rng.integers(1, len(seqs) + 1)), replace=False))
        step = [seqs[i] for i in pick if seqs[i].length < 16 * max_blocks]
        if not step:
            continue
        table = _c_table(step, max_blocks)
        lens = np.array([s.length + 1 for s in step], dtype=np.int32)
        src, dst = pkv.pkv_prepare_append(cpool, table, lens)
        pairs = []
        for s in step:
            (pos,) = s.append_tokens(1)
            pr = s.prepare_write(pos)
            if pr is not None:
                pairs.append(pr)
        assert list(zip(src.tolist(), dst.tolist())) == pairs
        assert np.array_equal(table, _c_table(step, max_blocks))
        assert cpool.num_free == opool.num_free
        assert all(cpool.refcount(b) == opool.refcount(b) for b in range(nb))


def test_c_prepare_append_is_all_or_nothing():
    pkv = pytest.importorskip("paged_kv_cache_153_gb300")
    cpool = pkv.BlockPool(3)
    a = cpool.alloc()                      # one shared block ...
    cpool.incref(a)
    cpool.incref(a)
    b = cpool.alloc()                      # ... and one private full block
    table = np.array([[a, -1], [a, -1], [a, -1], [b, -1]], dtype=np.int32)
    # rows 0, 1 copy (2 blocks), row 2 writes in place, row 3 needs a new block: 3 > 1 free
    with pytest.raises(pkv.PkvError):
        pkv.pkv_prepare_append(cpool, table, np.array([5, 5, 5, 17], dtype=np.int32))
    assert table.tolist() == [[a, -1], [a, -1], [a, -1], [b, -1]]
    assert cpool.refcount(a) == 3 and cpool.num_free == 1


def test_c_pool_cow():
    pkv = pytest.importorskip("paged_kv_cache_153_gb300")
    cpool = pkv.BlockPool(4)
    a = cpool.alloc()
    assert cpool.cow(a) == a                # private: nothing to do
    cpool.incref(a)
    n = cpool.cow(a)
    assert n != a and cpool.refcount(a) == 1 and cpool.refcount(n) == 1 and cpool.num_free == 2
