"""INT8 per-block min-max cache on the GPU ("What a KV cache is ..." section
3.3): quantisation and the re-quantising append bit for bit against the
oracle (oracle.int8), decode attention against the float64 oracle fed the
same codes and scalars."""
import numpy as np
import pytest
import torch

import pkv_workloads as wl
from oracle import attention as oa
from oracle import int8 as oi
from oracle import numerics as on
from oracle import slots as osl

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

INT8_ATOL = 2e-2     # as for E4M3: attention of the same codes, GPU vs float64


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__ as g
    g.build()
    import paged_kv_cache_153_gb300 as m
    return m


def _quantize(pkv, w, rows_used=None):
    d = gu.dev()
    kc = torch.empty(w.k_pool.shape, dtype=torch.uint8, device=d)
    vc = torch.empty_like(kc)
    prm = torch.empty(w.num_blocks, w.n_kv_heads, 4, dtype=torch.float32, device=d)
    ru = None if rows_used is None else torch.from_numpy(np.asarray(rows_used, dtype=np.int32)).to(d)
    pkv.pkv_kv_quantize_int8(gu.bits_to_torch(w.k_pool, w.kv_dtype), gu.bits_to_torch(w.v_pool, w.kv_dtype), kc, vc,
                             prm, rows_used=ru)
    return kc, vc, prm


def _oracle_quantize(w, rows_used=None):
    kq, kp = oi.quantize_pool(wl.bits_to_f32(w.k_pool, w.kv_dtype), rows_used)
    vq, vp = oi.quantize_pool(wl.bits_to_f32(w.v_pool, w.kv_dtype), rows_used)
    return kq, vq, np.concatenate([kp, vp], axis=2)


@pytest.mark.parametrize("dtype,hkv,d", [("bf16", 4, 128), ("f16", 2, 64)])
def test_quantize_bit_exact(pkv, dtype, hkv, d):
    w = wl.build("q8", batch=3, n_q_heads=hkv, n_kv_heads=hkv, head_dim=d, dtype=dtype, kv_dtype=dtype,
                 context_lens=[40, 7, 100], seed=d + hkv)
    rows = np.random.default_rng(2).integers(0, 17, size=w.num_blocks)
    for ru in (None, rows):
        kc, vc, prm = _quantize(pkv, w, ru)
        torch.cuda.synchronize()
        kq, vq, op = _oracle_quantize(w, ru)
        assert np.array_equal(kc.cpu().numpy(), kq) and np.array_equal(vc.cpu().numpy(), vq)
        assert np.array_equal(prm.cpu().numpy(), op)


def test_append_requantises_bit_exact(pkv):
    w = wl.build("a8", batch=5, n_q_heads=8, n_kv_heads=2, head_dim=128, dtype="bf16", kv_dtype="bf16",
                 context_lens=[1, 16, 17, 30, 200], seed=5)
    # the pool holds the tokens before the step: rows < (ctx - 1) % 16 of each last block, all rows elsewhere
    rows = np.full(w.num_blocks, 16, dtype=np.int32)
    for b, n in enumerate(w.context_lens):
        rows[w.block_tables[b][(int(n) - 1) // 16]] = (int(n) - 1) % 16
    kc, vc, prm = _quantize(pkv, w, rows)
    kq, vq, op = _oracle_quantize(w, rows)
    slots = gu.oracle_slots(w)
    err = torch.zeros(1, dtype=torch.int32, device=gu.dev())
    pkv.pkv_kv_append_int8(gu.bits_to_torch(w.k_new, "bf16"), gu.bits_to_torch(w.v_new, "bf16"),
                           torch.from_numpy(slots).to(gu.dev()), kc, vc, prm, err_flag=err)
    torch.cuda.synchronize()
    kp, vp = op[:, :, :2].copy(), op[:, :, 2:].copy()
    kn, vn = wl.bits_to_f32(w.k_new, "bf16"), wl.bits_to_f32(w.v_new, "bf16")
    for t, s in enumerate(slots):
        for h in range(w.n_kv_heads):
            oi.append_row(kq, kp, int(s) // 16, h, int(s) % 16, kn[t, h])
            oi.append_row(vq, vp, int(s) // 16, h, int(s) % 16, vn[t, h])
    assert int(err.item()) == 0
    assert np.array_equal(kc.cpu().numpy(), kq) and np.array_equal(vc.cpu().numpy(), vq)
    assert np.array_equal(prm.cpu().numpy(), np.concatenate([kp, vp], axis=2))


def _oracle_attention(w, kq, vq, prm, pairs=None):
    q = on.bits_to_f64(w.q, w.dtype)
    kf = np.empty(kq.shape)
    vf = np.empty(vq.shape)
    for blk in range(w.num_blocks):
        for h in range(w.n_kv_heads):
            kf[blk, h] = oi.decode_f64(kq[blk, h], prm[blk, h, 0], prm[blk, h, 1])
            vf[blk, h] = oi.decode_f64(vq[blk, h], prm[blk, h, 2], prm[blk, h, 3])
    group = w.n_q_heads // w.n_kv_heads
    pairs = pairs or [(b, h) for b in range(w.batch) for h in range(w.n_q_heads)]
    ref = {}
    for b, h in pairs:
        n = int(w.context_lens[b])
        ref[(b, h)] = oa.attend(q[b, h], oa.gather_sequence(kf, w.block_tables[b], n, h // group),
                                oa.gather_sequence(vf, w.block_tables[b], n, h // group), w.scale)
    return ref


@pytest.mark.parametrize("hq,hkv,d,dtype", [(8, 8, 128, "f16"), (16, 4, 128, "bf16"), (8, 4, 64, "bf16"),
                                            (16, 2, 128, "bf16")])
@pytest.mark.parametrize("partition", [0, 32])
def test_attention(pkv, hq, hkv, d, dtype, partition):
    lens = [1, 15, 16, 17, 33, 100, 257, 1000]
    w = wl.build("att8", batch=len(lens), n_q_heads=hq, n_kv_heads=hkv, head_dim=d, dtype=dtype, kv_dtype=dtype,
                 context_lens=lens, seed=hq * 3 + d)
    kc, vc, prm = _quantize(pkv, w)
    q = gu.bits_to_torch(w.q, dtype)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=gu.dev())
    ws = torch.empty(pkv.pkv_decode_workspace_bytes(w.batch, hq, hkv, d, w.max_blocks_per_seq, max(lens), partition),
                     dtype=torch.uint8, device=gu.dev())
    pkv.pkv_paged_decode_attention_int8(q, kc, vc, prm, torch.from_numpy(w.block_tables).to(gu.dev()),
                                        torch.from_numpy(w.context_lens).to(gu.dev()), out, scale=w.scale,
                                        max_context_len=max(lens), workspace=ws, partition_tokens=partition,
                                        err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = _oracle_attention(w, kc.cpu().numpy(), vc.cpu().numpy(), prm.cpu().numpy())
    g = out.float().cpu().numpy().astype(np.float64)
    worst = max(float(np.abs(g[b, h] - r).max()) for (b, h), r in ref.items())
    assert worst <= INT8_ATOL, worst
