"""The allocation-free decode entry point (pkv_paged_decode_attention_noalloc).

Some callers cannot allocate device memory: a plugin or C host program whose
host application owns every allocation and offers no allocator, or a
latency-critical loop where cudaMalloc / cudaFree would synchronise the
device.  For them the library keeps its decode scratch in one fixed device
array instead of a caller workspace.  This test calls that entry point through
the C ABI twice in a row (the second call on a different batch, so it runs on
the scratch the first call left behind), with the balanced split and with
fixed 512-token partitions, and checks that each output has the very bits of
the workspace-taking entry point (the same kernels on the same grid) and is
within the parity tolerance of the oracle.
It sits in its own file, collected last, and passes alone or after the others.
"""
import ctypes as C

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


def _call_noalloc(pkv, case, out, partition_tokens=0):
    w = case.w
    return pkv.lib.pkv_paged_decode_attention_noalloc(
        case.q.data_ptr(), case.k_cache.data_ptr(), case.v_cache.data_ptr(), case.tables.data_ptr(),
        case.lens.data_ptr(), w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, 16, w.max_blocks_per_seq,
        w.num_blocks, case.max_ctx, C.c_float(w.scale), out.data_ptr(), 1 if w.dtype == "bf16" else 0,
        partition_tokens, case.err.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _two_calls(pkv, workloads, partition_tokens):
    for w in workloads:
        case = gu.GpuCase(w)
        case.step(partition_tokens=partition_tokens, append=False)   # existing entry point, caller workspace
        torch.cuda.synchronize()
        ref = case.out.clone()
        out = torch.full_like(case.q, float("nan"))
        assert _call_noalloc(pkv, case, out, partition_tokens) == 0, pkv.pkv_last_error()
        torch.cuda.synchronize()
        assert case.err_code() == 0
        # same kernels on the same grid: the very same bits
        assert torch.equal(out, ref)
        # and both agree with the oracle
        assert gu.compare(out, gu.oracle_decode(w, w.k_pool, w.v_pool))[2] == 0


def test_noalloc_matches_workspace_entry_point_on_two_calls(pkv):
    first = wl.build("noalloc_a", batch=9, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
                     kv_dtype="bf16", context_lens=[1, 16, 17, 300, 1024, 2049, 4000, 77, 5000], seed=61)
    second = wl.build("noalloc_b", batch=5, n_q_heads=16, n_kv_heads=16, head_dim=64, dtype="f16",
                      kv_dtype="f16", context_lens=[3000, 5, 0, 640, 129], seed=62)
    _two_calls(pkv, (first, second), 0)


def test_noalloc_fixed_partitions_on_two_calls(pkv):
    # the fixed-partition split indexes its partial slots differently from the
    # balanced one; a scaled-down long/short mix (512-token partitions) fits in
    # the scratch, and the second call runs over what the first left behind
    first = wl.build("noalloc_p", batch=12, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
                     kv_dtype="bf16", context_lens=[2048] * 10 + [16384, 9000], seed=63)
    second = wl.build("noalloc_q", batch=6, n_q_heads=8, n_kv_heads=8, head_dim=128, dtype="f16",
                      kv_dtype="f16", context_lens=[700, 1, 4096, 513, 0, 2000], seed=65)
    assert pkv.pkv_decode_workspace_bytes(12, 32, 8, 128, first.max_blocks_per_seq, 16384, 512) \
        <= pkv.PKV_NOALLOC_SCRATCH_BYTES
    _two_calls(pkv, (first, second), 512)


def test_noalloc_argument_errors_match_the_workspace_entry_point(pkv):
    # batch 0 with a bad group is rejected like the workspace entry point does
    dummy = C.c_void_p(256)
    st = pkv.lib.pkv_paged_decode_attention_noalloc(dummy, dummy, dummy, dummy, dummy, 0, 6, 2, 128, 16, 4, 8, 64,
                                                    C.c_float(0.1), dummy, 0, 0, None, None)
    ref = pkv.lib.pkv_paged_decode_attention(dummy, dummy, dummy, dummy, dummy, 0, 6, 2, 128, 16, 4, 8, 64,
                                             C.c_float(0.1), dummy, 0, 0, dummy, 1 << 20, None, None)
    assert st == ref == 2


def test_noalloc_refuses_work_larger_than_its_scratch(pkv):
    # the partial slots are bounded by the resident thread blocks, but the
    # per-sequence prefixes grow with the batch: 2.5 million sequences need
    # more than the 16 MiB scratch, and the call is refused before any launch
    # (before q or the tables are read)
    w = wl.build("noalloc_big", batch=64, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
                 kv_dtype="bf16", context_lens=[16] * 64, seed=64)
    case = gu.GpuCase(w)
    big = 2_500_000
    assert pkv.pkv_decode_workspace_bytes(big, 32, 8, 128, 4096, 1 << 16, 16) > 16 * 1024 * 1024
    out = torch.empty_like(case.q)
    st = pkv.lib.pkv_paged_decode_attention_noalloc(
        case.q.data_ptr(), case.k_cache.data_ptr(), case.v_cache.data_ptr(), case.tables.data_ptr(),
        case.lens.data_ptr(), big, 32, 8, 128, 16, 4096, w.num_blocks, 1 << 16, C.c_float(w.scale),
        out.data_ptr(), 1, 16, case.err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 6 and "scratch" in pkv.pkv_last_error()
