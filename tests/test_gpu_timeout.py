"""The bounded waits of the decode kernel, made to run out on purpose.

Every pipeline wait of the decode kernel is limited (1 s by default).  The
environment variable PKV_WAIT_LIMIT_NS shortens that limit for the test: with
a limit of 1 ns, waits give up before their copies land.  The kernel then
records PKV_ERR_TIMEOUT, stops issuing copies, waits (with the full limit)
for the copies already in flight and returns -- no trap, no fault, no endless
wait -- and the same context computes the next call correctly."""
import time

import numpy as np
import pytest
import torch

import pkv_workloads as wl

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

PKV_ERR_TIMEOUT = 7


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__ as g
    g.build()
    import paged_kv_cache_153_gb300 as m
    return m


@pytest.mark.parametrize("hq,hkv,dtype", [(32, 8, "bf16"), (16, 16, "f16")])
def test_expired_waits_report_timeout_and_the_kernel_returns(pkv, monkeypatch, hq, hkv, dtype):
    # tensor-core (G = 4) and CUDA-core (G = 1) consumers; long contexts give
    # every thread block many waits
    w = wl.build("timeout", batch=8, n_q_heads=hq, n_kv_heads=hkv, head_dim=128, dtype=dtype, kv_dtype=dtype,
                 context_lens=[4096, 3000, 2048, 5000, 1, 700, 4096, 2500], seed=hq + hkv)
    case = gu.GpuCase(w)
    torch.cuda.synchronize()
    monkeypatch.setenv("PKV_WAIT_LIMIT_NS", "1")
    t0 = time.perf_counter()
    case.fused_step()
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    monkeypatch.delenv("PKV_WAIT_LIMIT_NS")
    assert case.err_code() == PKV_ERR_TIMEOUT
    assert elapsed < 10.0                       # the launch ended on its own
    # the context is intact: the next call is exact again
    case.err.zero_()
    case.step(append=False)
    torch.cuda.synchronize()
    assert case.err_code() == 0
    kp, vp = gu.oracle_pools_after_append(w)
    max_abs, _, n_bad, _ = gu.compare_all(case.out, gu.oracle_decode_all(w, kp, vp), gu.ATOL, gu.RTOL)
    assert n_bad == 0, max_abs
