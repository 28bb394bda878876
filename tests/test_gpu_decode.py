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
# full-size workloads, in the launch configuration the benchmark times: every
# output element against the oracle
# ---------------------------------------------------------------------------
@pytest.mark.slow
@pytest.mark.parametrize("name", ["mha7b", "gqa8b", "prefix"])
def test_full_size_every_output(pkv, name):
    w = wl.make(name)
    case = gu.GpuCase(w)
    case.fused_step()                         # what bench.py times: the fused step, balanced split
    torch.cuda.synchronize()
    assert case.err_code() == 0
    kp, vp = gu.oracle_pools_after_append(w)
    # the fused append wrote exactly the oracle's rows into exactly the oracle's slots
    assert np.array_equal(case.slots.cpu().numpy(), gu.oracle_slots(w))
    assert np.array_equal(gu.torch_bits(case.k_cache), kp) and np.array_equal(gu.torch_bits(case.v_cache), vp)
    ref = gu.oracle_decode_all(w, kp, vp)
    max_abs, max_rel, n_bad, n = gu.compare_all(case.out, ref, gu.ATOL, gu.RTOL)
    gu.record_parity(name, split="balanced", max_abs=max_abs, max_rel=max_rel, elements=n, bad=n_bad)
    assert n_bad == 0, f"{name}: {n_bad} of {n} elements out of tolerance (max abs {max_abs:.3e})"
    # fixed 512-token partitions of the same call agree too
    case.step(partition_tokens=512, append=False)
    max_abs, max_rel, n_bad, n = gu.compare_all(case.out, ref, gu.ATOL, gu.RTOL)
    gu.record_parity(name, split="partitions of 512", max_abs=max_abs, max_rel=max_rel, elements=n, bad=n_bad)
    assert case.err_code() == 0 and n_bad == 0


@pytest.mark.slow
def test_full_size_fp8long_every_output(pkv):
    # the oracle's E4M3 codes of the whole pool go in; the fused step appends
    # (quantising the new rows) and attends with 512-token partitions, as the
    # benchmark runs it; every sequence, every query head is compared
    w = wl.make("fp8long")
    kc = gu.oracle_fp8_pool_codes(w, w.k_pool, w.k_scale)
    vc = gu.oracle_fp8_pool_codes(w, w.v_pool, w.v_scale)
    case = gu.GpuCase(w, codes=(kc, vc))
    case.fused_step()
    torch.cuda.synchronize()
    assert case.err_code() == 0
    slots = gu.oracle_slots(w)
    assert np.array_equal(case.slots.cpu().numpy(), slots)
    gu.osl.append_rows(kc, gu.oracle_fp8_pool_codes(w, w.k_new, w.k_scale), slots)
    gu.osl.append_rows(vc, gu.oracle_fp8_pool_codes(w, w.v_new, w.v_scale), slots)
    assert np.array_equal(case.k_cache.cpu().numpy(), kc) and np.array_equal(case.v_cache.cpu().numpy(), vc)
    ref = gu.oracle_decode_all(w, kc, vc)
    max_abs, max_rel, n_bad, n = gu.compare_all(case.out, ref, gu.FP8_ATOL, 0.0)
    gu.record_parity("fp8long", split="partitions of 512", max_abs=max_abs, max_rel=max_rel, elements=n, bad=n_bad)
    assert n_bad == 0, f"fp8long: {n_bad} of {n} elements beyond {gu.FP8_ATOL} (max abs {max_abs:.3e})"
    # the balanced split of the same cache agrees too
    case.step(partition_tokens=0, append=False)
    max_abs, max_rel, n_bad, n = gu.compare_all(case.out, ref, gu.FP8_ATOL, 0.0)
    gu.record_parity("fp8long", split="balanced", max_abs=max_abs, max_rel=max_rel, elements=n, bad=n_bad)
    assert case.err_code() == 0 and n_bad == 0


def test_fp8_code_table_is_the_oracle_encoder():
    # the table route gives the oracle's own codes (a few thousand values)
    w = wl.build("fp8tab", batch=2, n_q_heads=8, n_kv_heads=2, head_dim=64, dtype="bf16", kv_dtype="e4m3",
                 context_lens=[20, 40], seed=3)
    kc, vc, kn, vn = gu.oracle_fp8_codes(w)
    assert np.array_equal(gu.oracle_fp8_pool_codes(w, w.k_pool, w.k_scale), kc)
    assert np.array_equal(gu.oracle_fp8_pool_codes(w, w.v_new, w.v_scale), vn)


@pytest.mark.slow
def test_full_size_tiny_every_output(pkv):
    w = wl.make("tiny")
    case = gu.GpuCase(w)
    case.fused_step()
    kp, vp = gu.oracle_pools_after_append(w)
    max_abs, max_rel, n_bad, n = gu.compare_all(case.out, gu.oracle_decode_all(w, kp, vp), gu.ATOL, gu.RTOL)
    gu.record_parity("tiny", split="balanced", max_abs=max_abs, max_rel=max_rel, elements=n, bad=n_bad)
    assert case.err_code() == 0 and n_bad == 0


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


@pytest.mark.parametrize("name,partition", [("gqa8b", 0), ("fp8long", 512), ("mha7b", 0)])
def test_workspace_contents_do_not_change_the_result(pkv, name, partition):
    # the workspace needs no initialisation: whatever an earlier call or a
    # fill left in it, every call gives the same bits
    w = wl.make(name)
    if w.fp8:
        case = gu.GpuCase(w, codes=(gu.oracle_fp8_pool_codes(w, w.k_pool, w.k_scale),
                                    gu.oracle_fp8_pool_codes(w, w.v_pool, w.v_scale)))
    else:
        case = gu.GpuCase(w)
    ws = case.workspace(partition)
    outs = []
    for fill in (0xFF, None, None, 0x00, None):
        if fill is not None:
            ws.fill_(fill)
        case.step(partition_tokens=partition, append=False)
        outs.append(case.out.clone())
    torch.cuda.synchronize()
    assert case.err_code() == 0
    assert all(torch.equal(outs[0], o) for o in outs[1:])
