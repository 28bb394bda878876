"""Copy-on-write on the GPU ("Series 03 ..." section 3.3): the block copy
kernel against the oracle's copy, bit for bit, and one decode step of a beam
search over shared prompt blocks -- the host pool's copy-on-write, the block
copies and the fused decode step -- against the oracle's fork /
prepare_write / copy / append / attention."""
import numpy as np
import pytest
import torch

import pkv_workloads as wl
from oracle import attention as oa
from oracle import numerics as on
from oracle import slots as osl
from oracle.block_pool import BlockPool, SequenceTable

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

PKV_ERR_OOB = 4


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__ as g
    g.build()
    import paged_kv_cache_153_gb300 as m
    return m


def _random_cache(rng, shape, kind):
    if kind == "e4m3":
        return rng.integers(0, 256, size=shape, dtype=np.uint8)
    return rng.integers(0, 2 ** 16, size=shape, dtype=np.uint16)


def _to_dev(a, kind):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if kind != "e4m3":
        t = t.view(gu.TORCH_16[kind])
    return t.to(gu.dev())


def _bits(t):
    return gu.torch_bits(t)


@pytest.mark.parametrize("kind,n_kv,d,nb,npairs", [("f16", 8, 128, 96, 40), ("bf16", 2, 64, 64, 31),
                                                   ("e4m3", 8, 128, 80, 33), ("e4m3", 1, 64, 20, 1)])
def test_copy_blocks_bit_exact(pkv, kind, n_kv, d, nb, npairs):
    rng = np.random.default_rng(nb + npairs)
    kc = _random_cache(rng, (nb, n_kv, 16, d), kind)
    vc = _random_cache(rng, (nb, n_kv, 16, d), kind)
    src, dst = wl.copy_pairs(nb, npairs, seed=nb)
    k_dev, v_dev = _to_dev(kc, kind), _to_dev(vc, kind)
    err = torch.zeros(1, dtype=torch.int32, device=gu.dev())
    pkv.pkv_copy_blocks(torch.from_numpy(src).to(gu.dev()), torch.from_numpy(dst).to(gu.dev()), k_dev, v_dev,
                        err_flag=err)
    torch.cuda.synchronize()
    pairs = list(zip(src.tolist(), dst.tolist()))
    osl.copy_blocks(kc, pairs)
    osl.copy_blocks(vc, pairs)
    assert int(err.item()) == 0
    assert np.array_equal(_bits(k_dev), kc) and np.array_equal(_bits(v_dev), vc)


def test_copy_blocks_out_of_range_pair_is_skipped_and_reported(pkv):
    rng = np.random.default_rng(5)
    nb = 24
    kc = _random_cache(rng, (nb, 2, 16, 64), "bf16")
    vc = _random_cache(rng, (nb, 2, 16, 64), "bf16")
    src = np.array([1, nb, 3, 5], dtype=np.int32)        # pair 1 reads past the pool
    dst = np.array([10, 11, -1, 12], dtype=np.int32)     # pair 2 writes before it
    k_dev, v_dev = _to_dev(kc, "bf16"), _to_dev(vc, "bf16")
    err = torch.zeros(1, dtype=torch.int32, device=gu.dev())
    pkv.pkv_copy_blocks(torch.from_numpy(src).to(gu.dev()), torch.from_numpy(dst).to(gu.dev()), k_dev, v_dev,
                        err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == PKV_ERR_OOB
    osl.copy_blocks(kc, [(1, 10), (5, 12)])
    osl.copy_blocks(vc, [(1, 10), (5, 12)])
    assert np.array_equal(_bits(k_dev), kc) and np.array_equal(_bits(v_dev), vc)


def test_copy_blocks_empty_is_a_no_op(pkv):
    kc = torch.zeros(4, 1, 16, 64, dtype=torch.float16, device=gu.dev())
    none = torch.empty(0, dtype=torch.int32, device=gu.dev())
    pkv.pkv_copy_blocks(none, none, kc, kc.clone())
    torch.cuda.synchronize()
    assert int(kc.abs().sum().item()) == 0


# ---------------------------------------------------------------------------
# one decode step of a beam search over shared prompts
# ---------------------------------------------------------------------------
def _c_state(pkv, bi):
    """Tables and copies from the library's host pool."""
    pool = pkv.BlockPool(bi.num_blocks)
    max_blocks = int(max(-(-(int(n) + 1) // 16) for n in bi.prompt_lens))
    tables = np.full((bi.batch, max_blocks), -1, dtype=np.int32)
    for p, n in enumerate(bi.prompt_lens):
        ids = [pool.alloc() for _ in range(-(-int(n) // 16))]
        for j in range(bi.beams):
            tables[p * bi.beams + j, :len(ids)] = ids
            if j:
                for i in ids:
                    pool.incref(i)
    lens = np.repeat(bi.prompt_lens.astype(np.int32) + 1, bi.beams)
    src, dst = pkv.pkv_prepare_append(pool, tables, lens)
    return pool, tables, lens, src, dst


def _oracle_state(bi):
    """The same step through the oracle: prompts, forks, one appended token
    per branch with copy-on-write."""
    pool = BlockPool(bi.num_blocks)
    prompts = []
    for n in bi.prompt_lens:
        s = SequenceTable(pool)
        s.append_tokens(int(n))
        prompts.append(s)
    seqs = []
    for s in prompts:
        seqs += [s] + [s.fork() for _ in range(bi.beams - 1)]
    pairs, slots = [], []
    for s in seqs:
        (pos,) = s.append_tokens(1)
        pr = s.prepare_write(pos)
        if pr is not None:
            pairs.append(pr)
        slots.append(osl.slot_of(s.blocks, pos))
    return pool, seqs, pairs, slots


def _run(pkv, bi, sample=None):
    pool, tables, lens, src, dst = _c_state(pkv, bi)
    opool, seqs, pairs, oslots = _oracle_state(bi)
    # host copy-on-write: identical tables, copies and pool state
    assert list(zip(src.tolist(), dst.tolist())) == pairs
    for b, s in enumerate(seqs):
        assert tables[b, :len(s.blocks)].tolist() == s.blocks
    assert pool.num_free == opool.num_free
    d = gu.dev()
    k_dev, v_dev = gu.bits_to_torch(bi.k_pool, bi.dtype), gu.bits_to_torch(bi.v_pool, bi.dtype)
    q = gu.bits_to_torch(bi.q, bi.dtype)
    k_new, v_new = gu.bits_to_torch(bi.k_new, bi.dtype), gu.bits_to_torch(bi.v_new, bi.dtype)
    t_dev, l_dev = torch.from_numpy(tables).to(d), torch.from_numpy(lens).to(d)
    out = torch.empty_like(q)
    slots = torch.empty(bi.batch, dtype=torch.int64, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    max_ctx = int(lens.max())
    ws = torch.empty(pkv.pkv_decode_workspace_bytes(bi.batch, bi.n_q_heads, bi.n_kv_heads, bi.head_dim,
                                                    tables.shape[1], max_ctx, 0), dtype=torch.uint8, device=d)
    pkv.pkv_copy_blocks(torch.from_numpy(src).to(d), torch.from_numpy(dst).to(d), k_dev, v_dev, err_flag=err)
    pkv.pkv_paged_decode_step(q, k_new, v_new, k_dev, v_dev, t_dev, l_dev, out, scale=bi.scale,
                              max_context_len=max_ctx, workspace=ws, slot_mapping_out=slots, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert slots.cpu().tolist() == oslots
    kp, vp = bi.k_pool.copy(), bi.v_pool.copy()
    osl.copy_blocks(kp, pairs)
    osl.copy_blocks(vp, pairs)
    osl.append_rows(kp, bi.k_new, oslots)
    osl.append_rows(vp, bi.v_new, oslots)
    assert np.array_equal(_bits(k_dev), kp) and np.array_equal(_bits(v_dev), vp)
    qf = on.bits_to_f64(bi.q, bi.dtype)
    kf, vf = on.bits_to_f64(kp, bi.dtype), on.bits_to_f64(vp, bi.dtype)
    group = bi.n_q_heads // bi.n_kv_heads
    if sample is None:
        sample = [(b, h) for b in range(bi.batch) for h in range(bi.n_q_heads)]
    ref = {}
    for b, h in sample:
        g = h // group
        n = int(lens[b])
        ref[(b, h)] = oa.attend(qf[b, h], oa.gather_sequence(kf, seqs[b].blocks, n, g),
                                oa.gather_sequence(vf, seqs[b].blocks, n, g), bi.scale)
    max_abs, max_rel, bad = gu.compare(out, ref)
    assert bad == 0, (max_abs, max_rel)
    return src.size


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_beam_step_small(pkv, seed):
    rng = np.random.default_rng(seed + 40)
    lens = rng.integers(1, 90, size=5)
    lens[0] = 32                       # a prompt that ends on a block boundary: no copy, a new block
    bi = wl.beam_inputs("beam-small", n_prompts=5, beams=4, n_q_heads=8, n_kv_heads=2, head_dim=64,
                        dtype="bf16", prompt_lens=lens, seed=seed)
    n_copies = _run(pkv, bi)
    assert n_copies == sum(bi.beams - 1 for n in lens if n % 16)


def test_beam_step_full_size_sampled(pkv):
    bi = wl.make_beam()
    rng = np.random.default_rng(9)
    sample = [(int(b), int(h)) for b, h in zip(rng.integers(0, bi.batch, 96), rng.integers(0, bi.n_q_heads, 96))]
    sample += [(b, 0) for b in range(bi.batch)]
    _run(pkv, bi, sample)
