"""INT8 per-block min-max cache on the GPU ("What a KV cache is ..." section
3.3): quantisation and the re-quantising append bit for bit against the
oracle (oracle.int8); decode attention against the float64 oracle attending
over the oracle's own codes and scalars (after checking that the device holds
exactly those), within 2e-2 absolute as for the E4M3 cache."""
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


def _oracle_quantize(w, rows_used=None, chunk=2048):
    """Oracle codes and (k_min, k_max, v_min, v_max) of the 16-bit pools; the
    blocks are independent, so the pools are converted and quantised in
    chunks of blocks to bound host memory."""
    out = []
    for pool in (w.k_pool, w.v_pool):
        codes = np.empty(pool.shape, dtype=np.uint8)
        params = np.empty((pool.shape[0], pool.shape[1], 2), dtype=np.float32)
        for s in range(0, pool.shape[0], chunk):
            ru = None if rows_used is None else np.asarray(rows_used)[s:s + chunk]
            codes[s:s + chunk], params[s:s + chunk] = oi.quantize_pool(wl.bits_to_f32(pool[s:s + chunk], w.kv_dtype),
                                                                       ru)
        out.append((codes, params))
    (kq, kp), (vq, vp) = out
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
        _same_codes(kc, vc, prm, kq, vq, op)


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
    _same_codes(kc, vc, prm, kq, vq, np.concatenate([kp, vp], axis=2))


def _oracle_attention(w, kq, vq, prm, seqs=None):
    """float64 attention [B, Hq, d] over INT8 codes: each block of a sequence
    is decoded with its own (min, max) (NaN rows for sequences not in seqs)."""
    q = on.bits_to_f64(w.q, w.dtype)
    group = w.n_q_heads // w.n_kv_heads
    ref = np.full((w.batch, w.n_q_heads, w.head_dim), np.nan)
    for b in (range(w.batch) if seqs is None else seqs):
        n = int(w.context_lens[b])
        blocks = w.block_tables[b][:-(-n // 16)]
        for g in range(w.n_kv_heads):
            kf = np.stack([oi.decode_f64(kq[blk, g], prm[blk, g, 0], prm[blk, g, 1]) for blk in blocks]) \
                if n else np.zeros((0, 16, w.head_dim))
            vf = np.stack([oi.decode_f64(vq[blk, g], prm[blk, g, 2], prm[blk, g, 3]) for blk in blocks]) \
                if n else np.zeros((0, 16, w.head_dim))
            keys = kf.reshape(-1, w.head_dim)[:n]
            values = vf.reshape(-1, w.head_dim)[:n]
            for h in range(g * group, (g + 1) * group):
                ref[b, h] = oa.attend(q[b, h], keys, values, w.scale)
    return ref


# With head_dim 128 the library stores a V slab transposed, [128][16], with
# token r in column 4 ((r % 8) // 2) + 2 (r // 8) + r % 2 (its documented
# layout); the oracle's codes are [16][head_dim].
V_COLUMN_OF_TOKEN = np.array([4 * ((r % 8) // 2) + 2 * (r // 8) + r % 2 for r in range(16)])


def _v_rows(vc: np.ndarray) -> np.ndarray:
    """Device V codes in the oracle's [NB, H, 16, d] row layout."""
    if vc.shape[-1] != 128:
        return vc
    nb, h = vc.shape[:2]
    t = vc.reshape(nb, h, 128, 16)                 # [d][column]
    return np.ascontiguousarray(t[:, :, :, V_COLUMN_OF_TOKEN].transpose(0, 1, 3, 2))


def test_v_column_order_is_a_permutation():
    assert sorted(V_COLUMN_OF_TOKEN.tolist()) == list(range(16))
    assert V_COLUMN_OF_TOKEN.tolist()[:4] == [0, 1, 4, 5] and V_COLUMN_OF_TOKEN[8] == 2


def _same_codes(kc, vc, prm, kq, vq, op):
    assert np.array_equal(kc.cpu().numpy(), kq) and np.array_equal(_v_rows(vc.cpu().numpy()), vq)
    assert np.array_equal(prm.cpu().numpy(), op)


@pytest.mark.parametrize("hq,hkv,d,dtype", [(8, 8, 128, "f16"), (16, 4, 128, "bf16"), (8, 4, 64, "bf16"),
                                            (16, 2, 128, "bf16")])
@pytest.mark.parametrize("partition", [0, 32])
def test_attention(pkv, hq, hkv, d, dtype, partition):
    lens = [1, 15, 16, 17, 33, 100, 257, 1000]
    w = wl.build("att8", batch=len(lens), n_q_heads=hq, n_kv_heads=hkv, head_dim=d, dtype=dtype, kv_dtype=dtype,
                 context_lens=lens, seed=hq * 3 + d)
    kc, vc, prm = _quantize(pkv, w)
    kq, vq, op = _oracle_quantize(w)
    _same_codes(kc, vc, prm, kq, vq, op)          # the device holds the oracle's codes and scalars
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
    max_abs, _, n_bad, _ = gu.compare_all(out, _oracle_attention(w, kq, vq, op), INT8_ATOL, 0.0)
    assert n_bad == 0, max_abs


@pytest.mark.slow
def test_full_size_int8_step_every_output(pkv):
    """The INT8 step exactly as the benchmark runs it, on the Llama-3-8B-shaped
    GQA workload (batch 64, 32 query / 8 KV heads, d 128, bf16, contexts
    log-uniform in [128, 8192]): quantise the pool, then the fused step (slot
    mapping, re-quantising append and decode attention in one decode launch,
    then the combine; balanced split).  Codes, scalars and slots bit for bit;
    every output element."""
    w = wl.make("gqa8b")
    d = gu.dev()
    kc, vc, prm = _quantize(pkv, w)
    kq, vq, op = _oracle_quantize(w)
    _same_codes(kc, vc, prm, kq, vq, op)
    q, kn, vn = gu.bits_to_torch(w.q, "bf16"), gu.bits_to_torch(w.k_new, "bf16"), gu.bits_to_torch(w.v_new, "bf16")
    tables, lens = torch.from_numpy(w.block_tables).to(d), torch.from_numpy(w.context_lens).to(d)
    slots = torch.empty(w.batch, dtype=torch.int64, device=d)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    max_ctx = int(w.context_lens.max())
    ws = torch.empty(pkv.pkv_decode_workspace_bytes(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                                    w.max_blocks_per_seq, max_ctx, 0), dtype=torch.uint8, device=d)
    pkv.pkv_paged_decode_step_int8(q, kn, vn, kc, vc, prm, tables, lens, out, scale=w.scale, max_context_len=max_ctx,
                                   workspace=ws, slot_mapping_out=slots, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # oracle: the same append, row by row, on the oracle's codes
    ref_slots = gu.oracle_slots(w)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    kp, vp = op[:, :, :2].copy(), op[:, :, 2:].copy()
    knf, vnf = wl.bits_to_f32(w.k_new, "bf16"), wl.bits_to_f32(w.v_new, "bf16")
    for t, sl in enumerate(ref_slots):
        for h in range(w.n_kv_heads):
            oi.append_row(kq, kp, int(sl) // 16, h, int(sl) % 16, knf[t, h])
            oi.append_row(vq, vp, int(sl) // 16, h, int(sl) % 16, vnf[t, h])
    op = np.concatenate([kp, vp], axis=2)
    _same_codes(kc, vc, prm, kq, vq, op)
    max_abs, max_rel, n_bad, n = gu.compare_all(out, _oracle_attention(w, kq, vq, op), INT8_ATOL, 0.0)
    gu.record_parity("int8 (gqa8b shape)", split="balanced", max_abs=max_abs, max_rel=max_rel, elements=n,
                     bad=n_bad)
    assert n_bad == 0, f"{n_bad} of {n} elements beyond {INT8_ATOL} (max abs {max_abs:.3e})"


def _int8_case(pkv, w, rows_used):
    d = gu.dev()
    kc, vc, prm = _quantize(pkv, w, rows_used)
    tensors = dict(q=gu.bits_to_torch(w.q, w.dtype), kn=gu.bits_to_torch(w.k_new, w.dtype),
                   vn=gu.bits_to_torch(w.v_new, w.dtype), tables=torch.from_numpy(w.block_tables).to(d),
                   lens=torch.from_numpy(w.context_lens).to(d))
    return kc, vc, prm, tensors


def _rows_before_step(w):
    """Rows of each block that hold tokens before the step: the last block of
    each sequence holds (ctx - 1) % 16 rows, the others 16."""
    rows = np.full(w.num_blocks, 16, dtype=np.int32)
    for b, n in enumerate(w.context_lens):
        if int(n) > 0:
            rows[w.block_tables[b][(int(n) - 1) // 16]] = (int(n) - 1) % 16
    return rows


@pytest.mark.parametrize("hq,hkv,d,dtype,partition", [(32, 8, 128, "bf16", 0), (16, 16, 128, "f16", 0),
                                                      (16, 2, 128, "bf16", 32), (64, 8, 128, "bf16", 0),
                                                      (8, 4, 64, "bf16", 0), (8, 8, 64, "f16", 16)])
def test_fused_step_equals_the_three_calls(pkv, hq, hkv, d, dtype, partition):
    # pkv_paged_decode_step_int8 (the append with its slots from the table,
    # then the decode, which starts early and waits for it) gives the codes,
    # scalars, slots and outputs of slot mapping + pkv_kv_append_int8 +
    # pkv_paged_decode_attention_int8, bit for bit
    lens = [1, 2, 15, 16, 17, 33, 100, 257, 1000, 0]
    w = wl.build("int8fused", batch=len(lens), n_q_heads=hq, n_kv_heads=hkv, head_dim=d, dtype=dtype,
                 kv_dtype=dtype, context_lens=lens, seed=hq + 5 * hkv + d)
    rows = _rows_before_step(w)
    dev = gu.dev()
    ws = torch.empty(pkv.pkv_decode_workspace_bytes(w.batch, hq, hkv, d, w.max_blocks_per_seq, max(lens),
                                                    partition), dtype=torch.uint8, device=dev)
    # three calls
    kc1, vc1, prm1, t = _int8_case(pkv, w, rows)
    slots1 = torch.empty(w.batch, dtype=torch.int64, device=dev)
    out1 = torch.empty_like(t["q"])
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.pkv_slot_mapping(t["tables"], t["lens"], slots1, num_blocks=w.num_blocks, position_offset=-1, err_flag=err)
    pkv.pkv_kv_append_int8(t["kn"], t["vn"], slots1, kc1, vc1, prm1, err_flag=err)
    pkv.pkv_paged_decode_attention_int8(t["q"], kc1, vc1, prm1, t["tables"], t["lens"], out1, scale=w.scale,
                                        max_context_len=max(lens), workspace=ws, partition_tokens=partition,
                                        err_flag=err)
    # one fused call
    kc2, vc2, prm2, _ = _int8_case(pkv, w, rows)
    slots2 = torch.full((w.batch,), -7, dtype=torch.int64, device=dev)
    out2 = torch.empty_like(t["q"])
    pkv.pkv_paged_decode_step_int8(t["q"], t["kn"], t["vn"], kc2, vc2, prm2, t["tables"], t["lens"], out2,
                                   scale=w.scale, max_context_len=max(lens), workspace=ws,
                                   partition_tokens=partition, slot_mapping_out=slots2, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(slots1, slots2)
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2) and torch.equal(prm1, prm2)
    assert torch.equal(out1, out2)
    # and the outputs match the oracle attending over the oracle's appended codes
    kq, vq, op = _oracle_quantize(w, rows)
    kp, vp = op[:, :, :2].copy(), op[:, :, 2:].copy()
    knf, vnf = wl.bits_to_f32(w.k_new, dtype), wl.bits_to_f32(w.v_new, dtype)
    for b, sl in enumerate(gu.oracle_slots(w)):
        if sl < 0:
            continue
        for h in range(w.n_kv_heads):
            oi.append_row(kq, kp, int(sl) // 16, h, int(sl) % 16, knf[b, h])
            oi.append_row(vq, vp, int(sl) // 16, h, int(sl) % 16, vnf[b, h])
    op = np.concatenate([kp, vp], axis=2)
    _same_codes(kc2, vc2, prm2, kq, vq, op)
    max_abs, _, n_bad, _ = gu.compare_all(out2, _oracle_attention(w, kq, vq, op), INT8_ATOL, 0.0)
    assert n_bad == 0, max_abs


