"""Pins of the INT8 per-block min-max oracle ("What a KV cache is ..."
section 3.3: q = round((k - k_min) / (k_max - k_min) * 255), two scalars per
block)."""
import numpy as np
import pytest

from oracle import int8 as oi


def test_worked_example_of_the_formula():
    # k in {-1, 0, 1}: (k + 1) / 2 * 255 = 0, 127.5, 255 -> 0, 128 (half to even), 255
    q, lo, hi = oi.encode_rows(np.array([[-1.0, 0.0, 1.0]], dtype=np.float32))
    assert q.tolist() == [[0, 128, 255]] and (lo, hi) == (-1.0, 1.0)


@pytest.mark.parametrize("seed", range(4))
def test_range_ends_monotone_and_half_step_error(seed):
    rng = np.random.default_rng(seed)
    x = (rng.normal(size=(16, 128)) * rng.uniform(0.1, 10)).astype(np.float32)
    q, lo, hi = oi.encode_rows(x)
    assert q.flat[np.argmin(x)] == 0 and q.flat[np.argmax(x)] == 255
    order = np.argsort(x, axis=None)
    assert (np.diff(q.ravel()[order].astype(int)) >= 0).all()          # monotone
    err = np.abs(oi.decode_f64(q, lo, hi) - x.astype(np.float64))
    step = (float(hi) - float(lo)) / 255.0
    assert err.max() <= 0.5 * step * (1 + 1e-5)


def test_constant_block_is_exact():
    q, lo, hi = oi.encode_rows(np.full((5, 8), 0.75, dtype=np.float32))
    assert (q == 0).all() and np.array_equal(oi.decode_f64(q, lo, hi), np.full((5, 8), 0.75))


def test_requantising_without_a_range_change_keeps_the_codes():
    rng = np.random.default_rng(7)
    x = rng.normal(size=(12, 64)).astype(np.float32)
    q, lo, hi = oi.encode_rows(x)
    again, lo2, hi2 = oi.encode_rows(np.concatenate([oi.decode_f32(q[:-1], lo, hi), x[-1:]], axis=0))
    # rows 0..10 went through decode / encode, the range (set by raw values) may
    # only shrink if an extreme sat in those rows; where it is unchanged the codes are
    if (lo2, hi2) == (lo, hi):
        assert np.array_equal(again, q)


def test_append_row_by_row_tracks_the_values():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(16, 32)).astype(np.float32)
    codes = np.zeros((1, 1, 16, 32), dtype=np.uint8)
    params = np.zeros((1, 1, 2), dtype=np.float32)
    for r in range(16):
        oi.append_row(codes, params, 0, 0, r, x[r])
        lo, hi = params[0, 0]
        assert lo <= x[:r + 1].min() + 1e-6 and hi >= x[:r + 1].max() - 1e-6
        assert (codes[0, 0, r + 1:] == 0).all()
    dec = oi.decode_f64(codes[0, 0], *params[0, 0])
    # each re-quantisation adds at most half a step of the final range
    step = (float(params[0, 0, 1]) - float(params[0, 0, 0])) / 255.0
    assert np.abs(dec - x).max() <= 16 * 0.5 * step


def test_pool_quantisation_leaves_unused_rows_zero():
    rng = np.random.default_rng(1)
    pool = rng.normal(size=(3, 2, 16, 8)).astype(np.float32)
    codes, params = oi.quantize_pool(pool, rows_used=[16, 5, 0])
    assert (codes[1, :, 5:] == 0).all() and (codes[2] == 0).all() and (params[2] == 0).all()
    assert params[1, 0, 0] == pool[1, 0, :5].min() and params[1, 0, 1] == pool[1, 0, :5].max()


def test_worked_example_through_the_slab_encoder():
    # the same worked example as one slab of a stack, next to a constant slab
    x = np.array([[[-1.0, 0.0, 1.0]], [[2.5, 2.5, 2.5]]], dtype=np.float32)
    q, lo, hi = oi.encode_slabs(x)
    assert q.tolist() == [[[0, 128, 255]], [[0, 0, 0]]]
    assert lo.tolist() == [-1.0, 2.5] and hi.tolist() == [1.0, 2.5]


def test_each_slab_uses_only_its_own_range():
    # slabs of very different ranges side by side: each slab's extremes map to
    # 0 and 255 and its codes stay within half a step of its own values (a min
    # or max taken over the wrong axes would break one of these)
    rng = np.random.default_rng(11)
    x = (rng.normal(size=(5, 3, 16, 32)) * np.array([0.01, 1.0, 100.0])[None, :, None, None]).astype(np.float32)
    q, lo, hi = oi.encode_slabs(x)
    assert q.shape == x.shape and lo.shape == hi.shape == (5, 3)
    for i in range(5):
        for h in range(3):
            s = x[i, h]
            assert lo[i, h] == s.min() and hi[i, h] == s.max()
            assert q[i, h].flat[np.argmin(s)] == 0 and q[i, h].flat[np.argmax(s)] == 255
            step = (float(hi[i, h]) - float(lo[i, h])) / 255.0
            assert np.abs(oi.decode_f64(q[i, h], lo[i, h], hi[i, h]) - s).max() <= 0.5 * step * (1 + 1e-5)


def test_pool_quantisation_of_mixed_row_counts():
    # blocks with different used-row counts: every (block, head) slab has the
    # range of its used rows only, and rows past them stay zero
    rng = np.random.default_rng(12)
    pool = rng.normal(size=(9, 2, 16, 8)).astype(np.float32)
    rows = [16, 1, 7, 16, 0, 7, 3, 16, 1]
    codes, params = oi.quantize_pool(pool, rows_used=rows)
    for b, n in enumerate(rows):
        for h in range(2):
            if n == 0:
                assert (codes[b, h] == 0).all() and (params[b, h] == 0).all()
                continue
            s = pool[b, h, :n]
            assert params[b, h, 0] == s.min() and params[b, h, 1] == s.max()
            assert (codes[b, h, n:] == 0).all()
            step = (float(s.max()) - float(s.min())) / 255.0
            dec = oi.decode_f64(codes[b, h, :n], *params[b, h])
            assert np.abs(dec - s).max() <= 0.5 * step * (1 + 1e-5) or step == 0
