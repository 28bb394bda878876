"""Pins of oracle.attention: invariants the pages state, special cases with a
closed form, a library routine on the contiguous special case, and brute
force against recomputation without a cache."""
import math

import numpy as np
import pytest
import torch

from oracle.attention import (contiguous_decode_attention, decode_one, gather_sequence,
                              paged_decode_attention, softmax_weights)
from oracle.block_pool import BlockPool, SequenceTable
from oracle.slots import append_rows, slot_mapping
from oracle.toy_model import ToyAttentionLayer


def _paged_from_contiguous(k_seqs, v_seqs, num_blocks, rng, bs=16, fill=np.nan):
    """Scatter contiguous per-sequence K/V [n, H, d] into a pool through a
    random physical layout; unused slots hold ``fill``."""
    n_heads, d = k_seqs[0].shape[1:]
    kc = np.full((num_blocks, n_heads, bs, d), fill)
    vc = np.full((num_blocks, n_heads, bs, d), fill)
    perm = rng.permutation(num_blocks)
    max_blocks = max(-(-len(k) // bs) for k in k_seqs) + 2
    tables = np.full((len(k_seqs), max_blocks), -1, dtype=np.int64)
    pos = 0
    for b, (k, v) in enumerate(zip(k_seqs, v_seqs)):
        nb = -(-len(k) // bs)
        tables[b, :nb] = perm[pos:pos + nb]
        pos += nb
        for j in range(len(k)):
            kc[tables[b, j // bs], :, j % bs] = k[j]
            vc[tables[b, j // bs], :, j % bs] = v[j]
    return kc, vc, tables


def _random_problem(rng, lens, hq, hkv, d):
    q = rng.standard_normal((len(lens), hq, d))
    ks = [rng.standard_normal((n, hkv, d)) for n in lens]
    vs = [rng.standard_normal((n, hkv, d)) for n in lens]
    return q, ks, vs


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2), (4, 1)])
def test_paged_equals_contiguous_bitwise(hq, hkv):
    # "KV cache capacity planning" section 3: paging does not change the numbers
    rng = np.random.default_rng(0)
    lens = [1, 15, 16, 17, 40, 100]
    q, ks, vs = _random_problem(rng, lens, hq, hkv, 32)
    kc, vc, tables = _paged_from_contiguous(ks, vs, 64, rng)
    out = paged_decode_attention(q, kc, vc, tables, lens, 0.17)
    for b in range(len(lens)):
        ref = contiguous_decode_attention(q[b], ks[b], vs[b], 0.17)
        assert np.array_equal(out[b], ref)


def test_physical_permutation_invariance_bitwise():
    # "Series 03" section 3.1: physical blocks need not be contiguous; any
    # placement of the same logical rows gives the same result
    rng = np.random.default_rng(1)
    lens = [33, 70, 5]
    q, ks, vs = _random_problem(rng, lens, 4, 2, 16)
    outs = []
    for seed in range(4):
        kc, vc, tables = _paged_from_contiguous(ks, vs, 32, np.random.default_rng(seed))
        outs.append(paged_decode_attention(q, kc, vc, tables, lens, 0.25))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_weights_sum_to_one():
    rng = np.random.default_rng(2)
    for n in [1, 2, 16, 1000]:
        p = softmax_weights(rng.standard_normal(64), rng.standard_normal((n, 64)) * 3, 1 / 8)
        assert abs(p.sum() - 1.0) < 1e-12 and np.all(p >= 0)


def test_constant_values_give_that_constant():
    rng = np.random.default_rng(3)
    lens = [7, 300]
    q, ks, _ = _random_problem(rng, lens, 2, 2, 8)
    vs = [np.full((n, 2, 8), 2.5) for n in lens]
    kc, vc, tables = _paged_from_contiguous(ks, vs, 32, rng)
    out = paged_decode_attention(q, kc, vc, tables, lens, 0.3)
    assert np.allclose(out, 2.5, rtol=0, atol=1e-13)


def test_zero_query_averages_values():
    rng = np.random.default_rng(4)
    lens = [9, 130]
    _, ks, vs = _random_problem(rng, lens, 2, 1, 8)
    q = np.zeros((2, 2, 8))
    kc, vc, tables = _paged_from_contiguous(ks, vs, 16, rng)
    out = paged_decode_attention(q, kc, vc, tables, lens, 0.3)
    for b in range(2):
        for h in range(2):
            assert np.allclose(out[b, h], vs[b][:, 0, :].mean(axis=0), atol=1e-14)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(5)
    q, ks, vs = _random_problem(rng, [1], 3, 3, 8)
    kc, vc, tables = _paged_from_contiguous(ks, vs, 4, rng)
    out = paged_decode_attention(q, kc, vc, tables, [1], 1.0)
    assert np.array_equal(out[0], vs[0][0])


def test_dominant_score_selects_its_value():
    rng = np.random.default_rng(6)
    n, d = 50, 16
    k = rng.standard_normal((n, 1, d)) * 0.01
    v = rng.standard_normal((n, 1, d))
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 1.0
    k[23, 0, 0] = 1000.0   # exp(1000) overflows float64 unless the max is subtracted
    kc, vc, tables = _paged_from_contiguous([k], [v], 8, rng)
    out = paged_decode_attention(q, kc, vc, tables, [n], 1.0)
    assert np.allclose(out[0, 0], v[23, 0], atol=1e-30 + 1e-12)


def test_gqa_group_mapping():
    # query head h reads KV head h // G (contiguous groups)
    rng = np.random.default_rng(7)
    lens = [20]
    q = rng.standard_normal((1, 8, 4))
    k = rng.standard_normal((20, 2, 4))
    v = np.zeros((20, 2, 4))
    v[:, 0, :] = 1.0
    v[:, 1, :] = -3.0
    kc, vc, tables = _paged_from_contiguous([k], [v], 4, rng)
    out = paged_decode_attention(q, kc, vc, tables, lens, 0.5)
    assert np.allclose(out[0, :4], 1.0) and np.allclose(out[0, 4:], -3.0)


def test_empty_context_and_unread_tail():
    rng = np.random.default_rng(8)
    q, ks, vs = _random_problem(rng, [18], 2, 1, 8)
    kc, vc, tables = _paged_from_contiguous(ks, vs, 8, rng)       # other slots NaN
    tables[0, 2:] = 10 ** 6                                       # never read
    out = paged_decode_attention(np.concatenate([q, q]), kc, vc,
                                 np.concatenate([tables, tables]), [18, 0], 0.5)
    assert np.all(np.isfinite(out[0])) and np.array_equal(out[1], np.zeros((2, 8)))
    assert np.array_equal(out[0, 1], decode_one(q, kc, vc, tables, [18], 0.5, 0, 1))


@pytest.mark.parametrize("hq,hkv,n", [(4, 4, 37), (8, 2, 300), (2, 1, 1)])
def test_contiguous_case_matches_library_sdpa(hq, hkv, n):
    # with contiguous K/V the definition reduces to scaled dot-product
    # attention with the default 1/sqrt(d) scale ("the memory notepad" section 二)
    rng = np.random.default_rng(9)
    d = 64
    q = rng.standard_normal((hq, d))
    k = rng.standard_normal((n, hkv, d))
    v = rng.standard_normal((n, hkv, d))
    ours = contiguous_decode_attention(q, k, v, 1 / math.sqrt(d))
    g = hq // hkv
    qt = torch.from_numpy(q)[:, None, :]                           # [H, 1, d]
    kt = torch.from_numpy(np.repeat(k, g, axis=1)).permute(1, 0, 2)  # [H, n, d]
    vt = torch.from_numpy(np.repeat(v, g, axis=1)).permute(1, 0, 2)
    lib = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[:, 0, :].numpy()
    assert np.allclose(ours, lib, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (4, 2)])
def test_cached_decode_equals_recomputation(hq, hkv):
    # "KV Cache, the memory notepad" sections 一 and 四: decoding with the cache
    # gives the same outputs as recomputing every K/V from scratch.  The cached
    # side here is the whole paged path: pool, block table, slot mapping,
    # append, paged attention.
    rng = np.random.default_rng(10)
    d_model, d, steps = 24, 8, 40
    layer = ToyAttentionLayer(rng.standard_normal((d_model, hq * d)) * 0.3,
                              rng.standard_normal((d_model, hkv * d)) * 0.3,
                              rng.standard_normal((d_model, hkv * d)) * 0.3, hq, hkv, d)
    hidden = rng.standard_normal((steps, d_model))
    pool = BlockPool(8)
    pool._free = [int(i) for i in rng.permutation(8)]
    seq = SequenceTable(pool)
    kc = np.full((8, hkv, 16, d), np.nan)
    vc = np.full((8, hkv, 16, d), np.nan)
    scale = 1 / math.sqrt(d)
    for t in range(steps):
        q_t, k_t, v_t = layer.project(hidden[t])
        pos = seq.append_tokens(1)
        slots = slot_mapping([seq.blocks], [0], pos)
        append_rows(kc, k_t[None], slots)
        append_rows(vc, v_t[None], slots)
        table = np.array([seq.blocks + [-1] * (8 - len(seq.blocks))])
        cached = paged_decode_attention(q_t[None], kc, vc, table, [seq.length], scale)[0]
        fresh = layer.recompute_step(hidden, t, scale)
        assert np.allclose(cached, fresh, rtol=1e-12, atol=1e-13)


def test_gather_follows_table():
    cache = np.arange(4 * 1 * 16 * 1).reshape(4, 1, 16, 1)
    got = gather_sequence(cache, [2, 0], 20, 0)[:, 0]
    assert got.tolist() == list(range(32, 48)) + [0, 1, 2, 3]
