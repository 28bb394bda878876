"""The model-wide cache [num_blocks, num_layers, H_kv, 16, d] on the GPU: the
per-layer fused step and the captured whole-step graph against the oracle
(oracle.attention.layer_view + paged decode per layer)."""
import numpy as np
import pytest
import torch

import pkv_workloads as wl
from oracle import attention as oa
from oracle import numerics as on
from oracle import slots as osl

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__ as g
    g.build()
    import paged_kv_cache_153_gb300 as m
    return m


def _device(li):
    w, d = li.base, gu.dev()
    t = {k: gu.bits_to_torch(getattr(li, k), w.kv_dtype) for k in ("k_pool", "v_pool", "k_new", "v_new")}
    t["q"] = gu.bits_to_torch(li.q, w.dtype)
    t["tables"] = torch.from_numpy(w.block_tables).to(d)
    t["lens"] = torch.from_numpy(w.context_lens).to(d)
    t["out"] = torch.zeros_like(t["q"])
    t["slots"] = torch.empty(w.batch, dtype=torch.int64, device=d)
    t["err"] = torch.zeros(1, dtype=torch.int32, device=d)
    return t


def _oracle(li):
    """Per layer: append the layer's new rows, then paged decode attention on
    that layer's view of the model-wide cache."""
    w = li.base
    slots = osl.slot_mapping(w.block_tables, range(w.batch), w.context_lens.astype(np.int64) - 1)
    kp, vp = li.k_pool.copy(), li.v_pool.copy()
    outs = []
    for l in range(li.n_layers):
        kl, vl = oa.layer_view(kp, l), oa.layer_view(vp, l)
        osl.append_rows(kl, li.k_new[l], slots)
        osl.append_rows(vl, li.v_new[l], slots)
        outs.append(oa.paged_decode_attention(on.bits_to_f64(li.q[l], w.dtype), on.bits_to_f64(kl, w.kv_dtype),
                                              on.bits_to_f64(vl, w.kv_dtype), w.block_tables, w.context_lens,
                                              w.scale))
    return np.stack(outs), kp, vp, slots


def _check(li, t, ref):
    outs, kp, vp, slots = ref
    g = t["out"].float().cpu().numpy().astype(np.float64)
    lim = gu.ATOL + gu.RTOL * np.abs(outs)
    assert (np.abs(g - outs) <= lim).all(), float(np.abs(g - outs).max())
    assert np.array_equal(gu.torch_bits(t["k_pool"]), kp) and np.array_equal(gu.torch_bits(t["v_pool"]), vp)
    assert t["slots"].cpu().numpy().tolist() == slots.tolist()
    assert int(t["err"].item()) == 0


def _ws(pkv, w):
    n = pkv.pkv_decode_workspace_bytes(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.max_blocks_per_seq,
                                       int(w.context_lens.max()), 0)
    return torch.empty(n, dtype=torch.uint8, device=gu.dev())


@pytest.mark.parametrize("hq,hkv,head_dim,dtype", [(4, 4, 64, "f16"), (16, 4, 128, "bf16")])
def test_layer_steps(pkv, hq, hkv, head_dim, dtype):
    base = wl.build("layers", batch=6, n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim, dtype=dtype,
                    kv_dtype=dtype, context_lens=[1, 16, 17, 100, 257, 40], seed=hq + head_dim)
    li = wl.layers_inputs(base, 5, seed=3)
    t = _device(li)
    ws = _ws(pkv, base)
    for l in range(li.n_layers):
        pkv.pkv_paged_decode_step_layer(t["q"][l], t["k_new"][l], t["v_new"][l], t["k_pool"], t["v_pool"],
                                        t["tables"], t["lens"], t["out"][l], layer=l, scale=base.scale,
                                        max_context_len=int(base.context_lens.max()), workspace=ws,
                                        slot_mapping_out=t["slots"], err_flag=t["err"])
    torch.cuda.synchronize()
    _check(li, t, _oracle(li))


def test_step_graph_equals_layer_calls(pkv):
    li = wl.make_layers()
    base = li.base
    ref = _oracle(li)
    t = _device(li)
    ws = _ws(pkv, base)
    graph = pkv.StepGraph(t["q"], t["k_new"], t["v_new"], t["k_pool"], t["v_pool"], t["tables"], t["lens"], t["out"],
                          scale=base.scale, max_context_len=int(base.context_lens.max()), workspace=ws,
                          slot_mapping_out=t["slots"], err_flag=t["err"])
    graph.launch()
    torch.cuda.synchronize()
    _check(li, t, ref)
    first = t["out"].clone()
    # replays are idempotent (the same slots are rewritten) and bitwise stable
    for _ in range(3):
        graph.launch()
    torch.cuda.synchronize()
    assert torch.equal(first, t["out"])
    # the graph reads the buffers' current contents: new queries give new outputs
    t["q"].mul_(-1.0)
    graph.launch()
    torch.cuda.synchronize()
    assert not torch.equal(first, t["out"])
    del graph


def test_bad_layer_is_rejected(pkv):
    base = wl.make("tiny")
    li = wl.layers_inputs(base, 2, seed=1)
    t = _device(li)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_paged_decode_step_layer(t["q"][0], t["k_new"][0], t["v_new"][0], t["k_pool"], t["v_pool"],
                                        t["tables"], t["lens"], t["out"][0], layer=2, scale=base.scale,
                                        max_context_len=256, workspace=_ws(pkv, base))
