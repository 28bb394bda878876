"""GPU parity of paged prefill / extend attention (tcgen05 kernel) against
the float64 oracle (oracle.prefill)."""
import numpy as np
import pytest
import torch

import pkv_workloads as wl
from oracle import numerics as on
from oracle import prefill as op

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

PKV_ERR_OOB = 4


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__ as g
    g.build()
    import paged_kv_cache_153_gb300 as m
    return m


def _run(pkv, pi, max_query_len=None):
    d = gu.dev()
    q = gu.bits_to_torch(pi.q, pi.dtype)
    kc, vc = gu.bits_to_torch(pi.k_pool, pi.dtype), gu.bits_to_torch(pi.v_pool, pi.dtype)
    out = torch.full_like(q, 7.0)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    pkv.pkv_paged_prefill_attention(
        q, kc, vc, torch.from_numpy(pi.block_tables).to(d), torch.from_numpy(pi.context_lens).to(d),
        torch.from_numpy(pi.cu_seqlens).to(d), out, scale=pi.scale,
        max_query_len=int(pi.new_lens.max()) if max_query_len is None else max_query_len, err_flag=err)
    torch.cuda.synchronize()
    return out, int(err.item())


def _oracle(pi, rows=None):
    return op.paged_prefill_attention(on.bits_to_f64(pi.q, pi.dtype), on.bits_to_f64(pi.k_pool, pi.dtype),
                                      on.bits_to_f64(pi.v_pool, pi.dtype), pi.block_tables, pi.context_lens,
                                      pi.cu_seqlens, pi.scale, rows=rows)


def _compare(out, ref, rows=None):
    g = out.float().cpu().numpy().astype(np.float64)
    rows = range(g.shape[0]) if rows is None else rows
    worst = 0.0
    for t in rows:
        diff = np.abs(g[t] - ref[t])
        lim = gu.ATOL + gu.RTOL * np.abs(ref[t])
        assert (diff <= lim).all(), (t, float(diff.max()))
        worst = max(worst, float(diff.max()))
    return worst


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (16, 2)])
def test_ragged_extend(pkv, dtype, hq, hkv):
    # cached / new mixes: one-token decode, short chunks, a whole prompt, tile
    # boundaries (128 keys, 128 / G tokens), a partial last block
    cached = [0, 5, 130, 0, 300, 16, 1]
    new = [1, 40, 7, 200, 129, 16, 250]
    pi = wl.prefill_inputs("extend", cached_lens=cached, new_lens=new, n_q_heads=hq, n_kv_heads=hkv,
                           head_dim=128, dtype=dtype, seed=hq * 10 + hkv)
    out, err = _run(pkv, pi)
    assert err == 0
    _compare(out, _oracle(pi))


def test_query_tiles_longer_than_needed(pkv):
    # max_query_len above every sequence's count: the extra tiles do nothing
    pi = wl.prefill_inputs("extra", cached_lens=[10, 0], new_lens=[3, 33], n_q_heads=8, n_kv_heads=2,
                           head_dim=128, dtype="bf16", seed=3)
    out, err = _run(pkv, pi, max_query_len=300)
    assert err == 0
    _compare(out, _oracle(pi))


def test_garbage_past_the_context_is_ignored(pkv):
    pi = wl.prefill_inputs("poison", cached_lens=[7, 100, 0], new_lens=[30, 21, 77], n_q_heads=16, n_kv_heads=4,
                           head_dim=128, dtype="bf16", seed=9)
    for b, n in enumerate(pi.context_lens):
        n = int(n)
        if n % 16:
            blk = int(pi.block_tables[b][(n - 1) // 16])
            pi.k_pool[blk, :, n % 16:, :] = 0x7FFF
            pi.v_pool[blk, :, n % 16:, :] = 0x7FFF
    out, err = _run(pkv, pi)
    assert err == 0 and bool(torch.isfinite(out).all())
    _compare(out, _oracle(pi))


def test_bad_block_id_is_flagged_not_faulted(pkv):
    pi = wl.prefill_inputs("oob", cached_lens=[20], new_lens=[12], n_q_heads=8, n_kv_heads=2, head_dim=128,
                           dtype="bf16", seed=4)
    pi.block_tables[0, 0] = pi.num_blocks + 5
    _, err = _run(pkv, pi)
    assert err == PKV_ERR_OOB


def test_rows_match_the_decode_kernel(pkv):
    # the last new token of each sequence is a decode step: the prefill kernel
    # and the decode kernel agree within the tolerance on it
    pi = wl.prefill_inputs("vs-decode", cached_lens=[64, 999], new_lens=[64, 1], n_q_heads=16, n_kv_heads=4,
                           head_dim=128, dtype="bf16", seed=12)
    out, err = _run(pkv, pi)
    assert err == 0
    ref = _oracle(pi)
    last = [int(c) - 1 for c in pi.cu_seqlens[1:]]
    _compare(out, ref, rows=last)


@pytest.mark.slow
def test_full_size_sampled(pkv):
    pi = wl.make_prefill()
    out, err = _run(pkv, pi)
    assert err == 0
    rng = np.random.default_rng(1)
    rows = sorted(set(rng.integers(0, pi.q.shape[0], 48).tolist()) |
                  {0, 127, 128, 2047, 2048, int(pi.q.shape[0]) - 1})
    _compare(out, _oracle(pi, rows=rows), rows=rows)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_cluster_pairs(pkv, dtype):
    # Query tiles run in pairs that share K/V loads.  At G = 4 (32 tokens per
    # tile): a pair whose tiles need 3 and 4 key tiles (positions 350..381 and
    # 382..413), a pair with one empty tile (33 new tokens: tiles 0 and 1 with
    # one token), a single tile padded with an empty partner (32 new tokens),
    # and a one-token decode row.
    pi = wl.prefill_inputs("pairs", cached_lens=[350, 0, 17, 4000], new_lens=[64, 33, 32, 1], n_q_heads=16,
                           n_kv_heads=4, head_dim=128, dtype=dtype, seed=21)
    out, err = _run(pkv, pi)
    assert err == 0
    _compare(out, _oracle(pi))


def test_sequences_without_new_tokens(pkv):
    # a sequence with no new tokens (equal cu_seqlens entries) has no rows and
    # no query tile; the others are unaffected
    pi = wl.prefill_inputs("zero-new", cached_lens=[30, 64, 5, 200], new_lens=[0, 17, 0, 90], n_q_heads=16,
                           n_kv_heads=4, head_dim=128, dtype="bf16", seed=33)
    out, err = _run(pkv, pi)
    assert err == 0
    _compare(out, _oracle(pi))
