"""Pins of the prefill oracle (oracle.prefill): causal extend attention over
the paged cache ("KV Cache, the memory notepad ..." sections 二-四; "Series
03 ..." sections 3.1 and 5.1)."""
import numpy as np
import pytest

from oracle import attention as oa
from oracle import prefill as op
from oracle import slots as osl


def _paged_from_contiguous(k_seqs, v_seqs, n_kv, d, rng, spare=3):
    """Scatter per-sequence contiguous K/V [n, H_kv, d] into a paged cache
    through random tables and the oracle's slot mapping + append."""
    nblk = [-(-len(k) // 16) for k in k_seqs]
    nb = sum(nblk) + spare
    perm = rng.permutation(nb)
    tables, pos = [], 0
    for n in nblk:
        tables.append(list(perm[pos:pos + n]) + [-1] * (max(nblk) - n))
        pos += n
    kc = np.full((nb, n_kv, 16, d), np.nan)
    vc = np.full((nb, n_kv, 16, d), np.nan)
    for b, (k, v) in enumerate(zip(k_seqs, v_seqs)):
        slots = osl.slot_mapping(tables, [b] * len(k), range(len(k)))
        osl.append_rows(kc, k, slots)
        osl.append_rows(vc, v, slots)
    return kc, vc, tables


def _case(rng, lens, news, n_q, n_kv, d=16):
    k_seqs = [rng.normal(size=(n, n_kv, d)) for n in lens]
    v_seqs = [rng.normal(size=(n, n_kv, d)) for n in lens]
    kc, vc, tables = _paged_from_contiguous(k_seqs, v_seqs, n_kv, d, rng)
    cu = np.concatenate([[0], np.cumsum(news)])
    q = rng.normal(size=(int(cu[-1]), n_q, d))
    return q, kc, vc, tables, np.array(lens), cu, k_seqs, v_seqs


@pytest.mark.parametrize("n_q,n_kv", [(4, 4), (8, 2), (6, 1)])
def test_each_row_equals_a_decode_step(n_q, n_kv):
    # prefilling n tokens gives what n decode steps give: row i equals decode
    # attention over the first (position + 1) tokens
    rng = np.random.default_rng(n_q * 10 + n_kv)
    lens, news = [37, 16, 90, 5], [37, 3, 50, 1]
    q, kc, vc, tables, ctx, cu, _, _ = _case(rng, lens, news, n_q, n_kv)
    out = op.paged_prefill_attention(q, kc, vc, tables, ctx, cu, 0.25)
    for t, (b, p) in enumerate(op.prefill_positions(ctx, cu)):
        dec = oa.paged_decode_attention(q[t][None], kc, vc, [tables[b]], [p + 1], 0.25)[0]
        assert np.array_equal(out[t], dec)


@pytest.mark.parametrize("prefix", [0, 21, 64])
@pytest.mark.parametrize("n_q,n_kv", [(4, 4), (8, 2)])
def test_against_torch_sdpa_with_a_causal_mask(prefix, n_q, n_kv):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(prefix + n_q)
    new, d, scale = 45, 16, 0.3
    q, kc, vc, tables, ctx, cu, k_seqs, v_seqs = _case(rng, [prefix + new], [new], n_q, n_kv, d)
    out = op.paged_prefill_attention(q, kc, vc, tables, ctx, cu, scale)
    group = n_q // n_kv
    qt = torch.from_numpy(q).permute(1, 0, 2)                                      # [Hq, new, d]
    kt = torch.from_numpy(k_seqs[0]).permute(1, 0, 2).repeat_interleave(group, 0)  # [Hq, n, d]
    vt = torch.from_numpy(v_seqs[0]).permute(1, 0, 2).repeat_interleave(group, 0)
    i = torch.arange(new)[:, None]
    j = torch.arange(prefix + new)[None, :]
    mask = j <= prefix + i                                                         # query i sits at prefix + i
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    assert np.allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_later_positions_do_not_leak():
    rng = np.random.default_rng(3)
    q, kc, vc, tables, ctx, cu, _, _ = _case(rng, [60], [60], 4, 2)
    out = op.paged_prefill_attention(q, kc, vc, tables, ctx, cu, 0.25)
    # change K and V of positions 30.. ; rows 0..29 must not move, row 30.. must
    kc2, vc2 = kc.copy(), vc.copy()
    for p in range(30, 60):
        blk, off = tables[0][p // 16], p % 16
        kc2[blk, :, off] += 1.0
        vc2[blk, :, off] -= 2.0
    out2 = op.paged_prefill_attention(q, kc2, vc2, tables, ctx, cu, 0.25)
    assert np.array_equal(out[:30], out2[:30])
    assert not np.allclose(out[30:], out2[30:])


def test_chunked_prefill_equals_one_shot():
    # "Series 03" section 5.1: a long prompt may be prefilled in chunks; the
    # rows come out the same as prefilling it at once
    rng = np.random.default_rng(11)
    n, n_kv, n_q, d = 70, 2, 4, 16
    k = rng.normal(size=(n, n_kv, d))
    v = rng.normal(size=(n, n_kv, d))
    q = rng.normal(size=(n, n_q, d))
    kc, vc, tables = _paged_from_contiguous([k], [v], n_kv, d, rng)
    one = op.paged_prefill_attention(q, kc, vc, tables, [n], [0, n], 0.2)
    # chunks of 16, 33 and 21 tokens: each chunk sees the tokens written so far
    kc2 = np.full_like(kc, np.nan)
    vc2 = np.full_like(vc, np.nan)
    rows, start = [], 0
    for c in (16, 33, 21):
        slots = osl.slot_mapping(tables, [0] * c, range(start, start + c))
        osl.append_rows(kc2, k[start:start + c], slots)
        osl.append_rows(vc2, v[start:start + c], slots)
        rows.append(op.paged_prefill_attention(q[start:start + c], kc2, vc2, tables, [start + c], [0, c], 0.2))
        start += c
    assert np.array_equal(np.concatenate(rows), one)


def test_too_many_new_tokens_is_an_error():
    with pytest.raises(ValueError):
        op.prefill_positions([3], [0, 4])
