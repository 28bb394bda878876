"""The whole decode step from host buffers (pkv_decode_step_host) gives the
same bits as the device-resident path, and matches the oracle."""
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


def test_host_step_matches_device_step(pkv):
    w = wl.build("e2e", batch=7, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16", kv_dtype="bf16",
                 context_lens=[1, 16, 17, 200, 640, 1111, 4000], seed=33)
    ref_case = gu.GpuCase(w)
    ref_case.step()
    host_case = gu.GpuCase(w)
    d = gu.dev()
    pin = lambda a, dt=None: (torch.from_numpy(np.ascontiguousarray(a)).view(dt) if dt else
                              torch.from_numpy(np.ascontiguousarray(a))).pin_memory()
    h_q = pin(w.q, torch.bfloat16)
    h_k = pin(w.k_new, torch.bfloat16)
    h_v = pin(w.v_new, torch.bfloat16)
    h_t = pin(w.block_tables)
    h_l = pin(w.context_lens)
    h_out = torch.empty(h_q.shape, dtype=torch.bfloat16).pin_memory()
    d_q, d_k, d_v = torch.empty_like(h_q, device=d), torch.empty_like(h_k, device=d), torch.empty_like(h_v, device=d)
    d_t, d_l = torch.empty_like(h_t, device=d), torch.empty_like(h_l, device=d)
    d_s = torch.empty(w.batch, dtype=torch.int64, device=d)
    d_o = torch.empty_like(h_q, device=d)
    pkv.pkv_decode_step_host(h_q, h_k, h_v, h_t, h_l, h_out, d_q, d_k, d_v, d_t, d_l, d_s, d_o,
                             host_case.k_cache, host_case.v_cache, scale=w.scale,
                             max_context_len=int(w.context_lens.max()), workspace=host_case.workspace(0),
                             err_flag=host_case.err)
    torch.cuda.synchronize()
    assert host_case.err_code() == 0 and ref_case.err_code() == 0
    assert torch.equal(h_out, ref_case.out.cpu())
    kp, vp = gu.oracle_pools_after_append(w)
    assert gu.compare(h_out, gu.oracle_decode(w, kp, vp))[2] == 0
