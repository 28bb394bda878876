"""GPU parity of paged decode attention against the float64 oracle."""
import numpy as np
import pytest
import torch

import pkv_workloads as wl

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__ as g
    g.build()
    import paged_kv_cache_153_gb300 as m
    return m


def _check(case, ref, fp8=False, label=""):
    max_abs, max_rel, n_bad = gu.compare(case.out, ref, fp8=fp8)
    assert case.err_code() == 0, f"{label}: device error {case.err_code()}"
    assert n_bad == 0, f"{label}: {n_bad} elements out of tolerance (max abs {max_abs:.3e})"
    return max_abs


@pytest.mark.parametrize("partition", [0, 16, 64, 512])
def test_tiny_config_full(pkv, partition):
    w = wl.make("tiny")
    case = gu.GpuCase(w)
    case.step(partition_tokens=partition)
    kp, vp = gu.oracle_pools_after_append(w)
    _check(case, gu.oracle_decode(w, kp, vp), label=f"tiny P={partition}")


RAGGED = [1, 15, 16, 17, 33, 100, 257, 1000, 2049]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (16, 2)])
@pytest.mark.parametrize("partition", [0, 32])
def test_ragged_shapes(pkv, dtype, head_dim, hq, hkv, partition):
    w = wl.build("ragged", batch=len(RAGGED), n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim, dtype=dtype,
                 kv_dtype=dtype, context_lens=RAGGED, seed=head_dim * 100 + hq + hkv)
    case = gu.GpuCase(w)
    case.step(partition_tokens=partition)
    kp, vp = gu.oracle_pools_after_append(w)
    _check(case, gu.oracle_decode(w, kp, vp), label=f"{dtype} d{head_dim} {hq}/{hkv} P{partition}")


def test_empty_contexts(pkv):
    # context 0 gives zeros; the others are unaffected; all-empty is all zeros
    w = wl.build("empty", batch=4, n_q_heads=8, n_kv_heads=2, head_dim=128, dtype="bf16", kv_dtype="bf16",
                 context_lens=[0, 40, 0, 1], seed=5)
    case = gu.GpuCase(w)
    case.out.fill_(7.0)
    case.step(append=False)
    ref = gu.oracle_decode(w, w.k_pool, w.v_pool)
    _check(case, ref, label="empty")
    assert not case.out[0].any() and not case.out[2].any()
    case.lens.zero_()
    case.out.fill_(7.0)
    case.step(append=False)
    torch.cuda.synchronize()
    assert not case.out.any()


def test_physical_permutation_gives_identical_bits(pkv):
    # the same logical rows placed in other physical blocks must give the very
    # same output bits ("Series 03" 3.1: physical blocks need not be contiguous)
    w = wl.build("perm", batch=6, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16", kv_dtype="bf16",
                 context_lens=[5, 160, 161, 700, 1500, 3000], seed=9)
    a = gu.GpuCase(w)
    a.step(append=False)
    perm = np.random.default_rng(1).permutation(w.num_blocks)
    inv = np.argsort(perm)
    w2 = wl.build("perm", batch=6, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16", kv_dtype="bf16",
                  context_lens=[5, 160, 161, 700, 1500, 3000], seed=9)
    w2.k_pool = w.k_pool[inv]                         # new block i holds old block inv[i]
    w2.v_pool = w.v_pool[inv]
    t = w.block_tables.copy()
    t[t >= 0] = perm[t[t >= 0]]                      # old id j now lives at perm[j]
    w2.block_tables = t
    b = gu.GpuCase(w2)
    b.step(append=False)
    torch.cuda.synchronize()
    assert torch.equal(a.out, b.out)
    assert a.err_code() == 0 and b.err_code() == 0


def test_repeated_calls_are_deterministic(pkv):
    w = wl.make("tiny")
    case = gu.GpuCase(w)
    outs = []
    for _ in range(3):
        case.step(append=False)
        outs.append(case.out.clone())
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_constant_values(pkv):
    w = wl.build("const", batch=3, n_q_heads=16, n_kv_heads=4, head_dim=128, dtype="f16", kv_dtype="f16",
                 context_lens=[3, 77, 999], seed=2)
    w.v_pool[:] = np.float16(0.375).view(np.uint16)
    case = gu.GpuCase(w)
    case.step(append=False)
    torch.cuda.synchronize()
    assert torch.all(case.out == 0.375)


def test_out_of_range_block_id_is_flagged_not_faulted(pkv):
    w = wl.build("oob", batch=2, n_q_heads=8, n_kv_heads=2, head_dim=128, dtype="bf16", kv_dtype="bf16",
                 context_lens=[40, 40], seed=4)
    w.block_tables[1, 1] = w.num_blocks + 1000
    case = gu.GpuCase(w)
    case.step(append=False)
    assert case.err_code() == 4
    # sequence 0 does not depend on the bad entry
    ref = gu.oracle_decode(w, w.k_pool, w.v_pool, pairs=[(0, h) for h in range(8)])
    assert gu.compare(case.out, ref)[2] == 0


def test_context_past_table_is_flagged(pkv):
    w = wl.build("long", batch=1, n_q_heads=4, n_kv_heads=4, head_dim=64, dtype="f16", kv_dtype="f16",
                 context_lens=[64], seed=4)
    case = gu.GpuCase(w, max_context_len=64)
    case.lens.fill_(1000)                            # the table holds 4 blocks only
    case.step(append=False)
    assert case.err_code() == 4


# ---------------------------------------------------------------------------
# E4M3 cache
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("partition", [0, 512, 64])
def test_fp8_small(pkv, partition):
    w = wl.build("fp8small", batch=5, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
                 kv_dtype="e4m3", context_lens=[1, 17, 100, 513, 700], seed=21)
    kc, vc, kn, vn = gu.oracle_fp8_codes(w)
    case = gu.GpuCase(w, codes=(kc, vc))
    case.step(partition_tokens=partition)
    kp, vp = gu.oracle_pools_after_append(w)
    assert np.array_equal(case.k_cache.cpu().numpy(), kp)        # append bit-exact as well
    assert np.array_equal(case.v_cache.cpu().numpy(), vp)
    _check(case, gu.oracle_decode(w, kp, vp), fp8=True, label=f"fp8 P={partition}")


@pytest.mark.parametrize("hq,hkv,head_dim", [(16, 8, 128), (16, 16, 128), (64, 8, 128), (8, 4, 64), (8, 8, 64),
                                             (16, 2, 64)])
def test_fp8_shapes(pkv, hq, hkv, head_dim):
    # every group size on both head dims: the tensor-core consumer (128-byte
    # rows, G >= 2) and the CUDA-core consumer (G = 1 or 64-byte rows)
    w = wl.build("fp8shape", batch=4, n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim, dtype="f16",
                 kv_dtype="e4m3", context_lens=[1, 33, 250, 401], seed=hq * 7 + hkv + head_dim)
    kc, vc, kn, vn = gu.oracle_fp8_codes(w)
    case = gu.GpuCase(w, codes=(kc, vc))
    case.step(partition_tokens=0)
    kp, vp = gu.oracle_pools_after_append(w)
    _check(case, gu.oracle_decode(w, kp, vp), fp8=True, label=f"fp8 {hq}/{hkv} d{head_dim}")


# ---------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
# ---------------------------------------------------------------------------
def _sample_pairs(w, rng, n):
    pairs = {(0, 0), (w.batch - 1, w.n_q_heads - 1)}
    longest = int(np.argmax(w.context_lens))
    pairs.add((longest, int(rng.integers(w.n_q_heads))))
    while len(pairs) < n:
        pairs.add((int(rng.integers(w.batch)), int(rng.integers(w.n_q_heads))))
    return sorted(pairs)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mha7b", "gqa8b", "prefix"])
def test_full_size_sampled(pkv, name):
    w = wl.make(name)
    case = gu.GpuCase(w)
    case.step()
    torch.cuda.synchronize()
    kp, vp = gu.oracle_pools_after_append(w)
    pairs = _sample_pairs(w, np.random.default_rng(0), 24)
    _check(case, gu.oracle_decode(w, kp, vp, pairs), label=name)
    # partition split of the same call agrees too
    case.step(partition_tokens=512, append=False)
    _check(case, gu.oracle_decode(w, kp, vp, pairs), label=name + " P512")


@pytest.mark.slow
def test_full_size_fp8long_sampled(pkv):
    from oracle import e4m3 as oe
    from oracle import slots as osl
    w = wl.make("fp8long")
    d = gu.dev()
    # quantise the whole pool on the device (an append of every slot), then the step
    nb, H, bs, D = w.k_pool.shape
    placeholder = np.zeros((1, H, bs, D), np.uint8)
    case = gu.GpuCase(w, codes=(placeholder, placeholder))
    case.k_cache = torch.empty(nb, H, bs, D, dtype=torch.uint8, device=d)
    case.v_cache = torch.empty_like(case.k_cache)
    all_slots = torch.arange(nb * bs, dtype=torch.int64, device=d)
    k_rows = gu.bits_to_torch(w.k_pool, w.dtype).permute(0, 2, 1, 3).reshape(nb * bs, H, D).contiguous()
    v_rows = gu.bits_to_torch(w.v_pool, w.dtype).permute(0, 2, 1, 3).reshape(nb * bs, H, D).contiguous()
    pkv.pkv_kv_append_fp8(k_rows, v_rows, all_slots, case.k_cache, case.v_cache, case.k_scale, case.v_scale,
                          err_flag=case.err)
    del k_rows, v_rows
    kc = case.k_cache
    case.step()
    torch.cuda.synchronize()
    assert case.err_code() == 0
    # oracle: append the raw rows, then encode only the sampled sequences' rows
    slots = gu.oracle_slots(w)
    kp, vp = w.k_pool.copy(), w.v_pool.copy()
    osl.append_rows(kp, w.k_new, slots)
    osl.append_rows(vp, w.v_new, slots)
    from oracle import attention as oa
    from oracle import numerics as on
    group = w.n_q_heads // w.n_kv_heads
    short = [b for b in range(w.batch) if w.context_lens[b] == 2048][:2]
    long = [b for b in range(w.batch) if w.context_lens[b] == 65536][:1]
    got = case.out.float().cpu().numpy()
    kc_host = None
    for b in short + long:
        g = int(np.random.default_rng(b).integers(w.n_kv_heads))
        n = int(w.context_lens[b])
        kb = oe.encode(wl.bits_to_f32(oa.gather_sequence(kp, w.block_tables[b], n, g), w.dtype), w.k_scale[g])
        vb = oe.encode(wl.bits_to_f32(oa.gather_sequence(vp, w.block_tables[b], n, g), w.dtype), w.v_scale[g])
        # the device codes of those rows are the oracle's codes, bit for bit
        if kc_host is None:
            kc_host = kc.cpu().numpy()
        assert np.array_equal(oa.gather_sequence(kc_host, w.block_tables[b], n, g), kb)
        keys = oe.decode(kb) * float(w.k_scale[g])
        values = oe.decode(vb) * float(w.v_scale[g])
        q = on.bits_to_f64(w.q, w.dtype)
        for h in range(g * group, (g + 1) * group):
            ref = oa.attend(q[b, h], keys, values, w.scale)
            assert np.abs(got[b, h] - ref).max() <= gu.FP8_ATOL, (b, h)


def _poison_past_context(pool, w, pattern):
    """Rows of each sequence's last block that lie past its context (the new
    token's row is position ctx - 1, so rows >= ctx) get a NaN pattern."""
    for b, n in enumerate(w.context_lens):
        n = int(n)
        if n % 16:
            blk = int(w.block_tables[b][(n - 1) // 16])
            pool[blk, :, n % 16:, :] = pattern


@pytest.mark.parametrize("kind,hq,hkv,head_dim", [("f16", 8, 8, 128), ("bf16", 16, 4, 128), ("bf16", 8, 2, 64),
                                                  ("e4m3", 16, 4, 128), ("e4m3", 8, 8, 64)])
@pytest.mark.parametrize("partition", [0, 32])
def test_garbage_past_the_context_is_ignored(pkv, kind, hq, hkv, head_dim, partition):
    # The pages' block waste (the unused tail of a sequence's last block) may
    # hold anything; a NaN there must not reach the output.
    dtype = "bf16" if kind == "e4m3" else kind
    w = wl.build("poison", batch=len(RAGGED), n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim, dtype=dtype,
                 kv_dtype=kind, context_lens=RAGGED, seed=7 + hq + head_dim)
    if kind == "e4m3":
        kc, vc, kn, vn = gu.oracle_fp8_codes(w)
        _poison_past_context(kc, w, 0x7F)
        _poison_past_context(vc, w, 0x7F)
        case = gu.GpuCase(w, codes=(kc, vc))
        case.step(partition_tokens=partition)
        slots = gu.oracle_slots(w)
        gu.osl.append_rows(kc, kn, slots)
        gu.osl.append_rows(vc, vn, slots)
        _check(case, gu.oracle_decode(w, kc, vc), fp8=True, label=f"{kind} P{partition}")
    else:
        _poison_past_context(w.k_pool, w, 0x7FFF)
        _poison_past_context(w.v_pool, w, 0x7FFF)
        case = gu.GpuCase(w)
        case.step(partition_tokens=partition)
        kp, vp = gu.oracle_pools_after_append(w)
        _check(case, gu.oracle_decode(w, kp, vp), label=f"{kind} P{partition}")
    assert bool(torch.isfinite(case.out).all())


@pytest.mark.parametrize("hq,hkv", [(16, 4), (16, 2), (8, 4)])
def test_bf16_short_contexts(pkv, hq, hkv):
    # few keys: a single rounding of the softmax weights to bf16 would be
    # visible against the tolerance; the tensor-core path multiplies them exactly
    lens = list(range(2, 34)) * 2
    w = wl.build("short-bf16", batch=len(lens), n_q_heads=hq, n_kv_heads=hkv, head_dim=128, dtype="bf16",
                 kv_dtype="bf16", context_lens=lens, seed=hq + hkv)
    case = gu.GpuCase(w)
    case.step()
    kp, vp = gu.oracle_pools_after_append(w)
    _check(case, gu.oracle_decode(w, kp, vp), label=f"short bf16 {hq}/{hkv}")
