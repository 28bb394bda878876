"""The fused decode step (pkv_paged_decode_step[_fp8]: slot mapping, append and
attention in one decode launch) against the three separate calls, bit for bit:
outputs, cache contents and slots.  The separate calls are checked against
the oracle elsewhere; one case here is checked against the oracle directly."""
import numpy as np
import pytest
import torch

import pkv_workloads as wl

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

LENS = [1, 15, 16, 17, 48, 100, 257, 1000]    # new token in row 0, 14, 15, 0, 15, 3, 0, 7


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__ as g
    g.build()
    import paged_kv_cache_153_gb300 as m
    return m


def _fused(pkv, case, partition):
    w = case.w
    ws = case.workspace(partition)
    slots = torch.full((w.batch,), -7, dtype=torch.int64, device=gu.dev())
    if case.fp8:
        pkv.pkv_paged_decode_step_fp8(case.q, case.k_new, case.v_new, case.k_cache, case.v_cache, case.k_scale,
                                      case.v_scale, case.tables, case.lens, case.out, scale=w.scale,
                                      max_context_len=case.max_ctx, workspace=ws, partition_tokens=partition,
                                      slot_mapping_out=slots, err_flag=case.err)
    else:
        pkv.pkv_paged_decode_step(case.q, case.k_new, case.v_new, case.k_cache, case.v_cache, case.tables, case.lens,
                                  case.out, scale=w.scale, max_context_len=case.max_ctx, workspace=ws,
                                  partition_tokens=partition, slot_mapping_out=slots, err_flag=case.err)
    return slots


def _same(pkv, w, partition, codes=None):
    sep, fus = gu.GpuCase(w, codes=codes), gu.GpuCase(w, codes=codes)
    sep.step(partition_tokens=partition)
    slots = _fused(pkv, fus, partition)
    torch.cuda.synchronize()
    assert sep.err_code() == 0 and fus.err_code() == 0
    assert torch.equal(slots, sep.slots)
    assert torch.equal(fus.k_cache, sep.k_cache) and torch.equal(fus.v_cache, sep.v_cache)
    assert torch.equal(fus.out, sep.out)
    return fus


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv,head_dim", [(8, 8, 128), (32, 8, 128), (16, 8, 64), (16, 16, 64), (16, 2, 128)])
@pytest.mark.parametrize("partition", [0, 64])
def test_fused_step_equals_separate_calls(pkv, dtype, hq, hkv, head_dim, partition):
    w = wl.build("fused", batch=len(LENS), n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim, dtype=dtype,
                 kv_dtype=dtype, context_lens=LENS, seed=hq + 3 * hkv + head_dim)
    _same(pkv, w, partition)


def test_fused_step_matches_oracle_and_empty_context(pkv):
    w = wl.build("fused0", batch=4, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16", kv_dtype="bf16",
                 context_lens=[0, 33, 1, 4096], seed=77)
    fus = _same(pkv, w, 0)
    kp, vp = gu.oracle_pools_after_append(w)
    assert gu.compare(fus.out, gu.oracle_decode(w, kp, vp))[2] == 0
    assert not fus.out[0].any()


def test_fused_step_shared_prefix(pkv):
    _same(pkv, wl.make("prefix"), 0)


@pytest.mark.parametrize("hq,hkv,head_dim", [(32, 8, 128), (8, 8, 64), (16, 4, 64)])
def test_fused_step_fp8(pkv, hq, hkv, head_dim):
    w = wl.build("fusedfp8", batch=5, n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim, dtype="bf16", kv_dtype="e4m3",
                 context_lens=[1, 16, 31, 200, 513], seed=hq + hkv + head_dim)
    kc, vc, _, _ = gu.oracle_fp8_codes(w)
    _same(pkv, w, 0, codes=(kc, vc))
    _same(pkv, w, 64, codes=(kc, vc))
