"""GPU parity of slot mapping and append (bit-exact against the oracle)."""
import numpy as np
import pytest
import torch

import pkv_workloads as wl
from oracle import e4m3 as oe
from oracle import slots as osl

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__ as g
    g.build()
    import paged_kv_cache_153_gb300 as m
    return m


@pytest.mark.parametrize("name", ["tiny", "gqa8b", "prefix"])
def test_decode_slots_and_append_bit_exact(pkv, name):
    w = wl.make(name)
    case = gu.GpuCase(w)
    pkv.pkv_slot_mapping(case.tables, case.lens, case.slots, num_blocks=w.num_blocks, position_offset=-1,
                         err_flag=case.err)
    pkv.pkv_kv_append(case.k_new, case.v_new, case.slots, case.k_cache, case.v_cache, err_flag=case.err)
    assert case.err_code() == 0
    assert np.array_equal(case.slots.cpu().numpy(), gu.oracle_slots(w))
    kp, vp = gu.oracle_pools_after_append(w)
    assert np.array_equal(gu.torch_bits(case.k_cache), kp)
    assert np.array_equal(gu.torch_bits(case.v_cache), vp)


def test_general_slot_mapping(pkv):
    rng = np.random.default_rng(3)
    tables = rng.permutation(64).astype(np.int32).reshape(4, 16)
    seq = np.repeat(np.arange(4), 50).astype(np.int32)
    pos = np.tile(np.arange(-2, 48), 4).astype(np.int32)          # includes padding (-2, -1)
    d = gu.dev()
    out = torch.empty(len(pos), dtype=torch.int64, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    pkv.pkv_slot_mapping(torch.from_numpy(tables).to(d), torch.from_numpy(pos).to(d), out, num_blocks=64,
                         seq_idx=torch.from_numpy(seq).to(d), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(out.cpu().numpy(), osl.slot_mapping(tables, seq, pos))


def test_slot_mapping_flags_bad_entries(pkv):
    d = gu.dev()
    tables = torch.tensor([[3, 99, -1, 5]], dtype=torch.int32, device=d)   # 99 >= num_blocks, -1 unset
    pos = torch.tensor([0, 17, 40, 70], dtype=torch.int32, device=d)      # 70 is past the table
    seq = torch.zeros(4, dtype=torch.int32, device=d)
    out = torch.empty(4, dtype=torch.int64, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    pkv.pkv_slot_mapping(tables, pos, out, num_blocks=8, seq_idx=seq, err_flag=err)
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [48, -1, -1, -1]
    assert int(err.item()) == 4


def test_append_skips_negative_and_flags_oob(pkv):
    d = gu.dev()
    cache_k = torch.zeros(4, 2, 16, 64, dtype=torch.float16, device=d)
    cache_v = torch.zeros_like(cache_k)
    k_new = torch.randn(3, 2, 64, dtype=torch.float16, device=d)
    v_new = torch.randn(3, 2, 64, dtype=torch.float16, device=d)
    slots = torch.tensor([-1, 5, 64], dtype=torch.int64, device=d)        # skip, write, out of range
    err = torch.zeros(1, dtype=torch.int32, device=d)
    pkv.pkv_kv_append(k_new, v_new, slots, cache_k, cache_v, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 4
    assert torch.equal(cache_k[0, :, 5], k_new[1]) and torch.equal(cache_v[0, :, 5], v_new[1])
    mask = torch.ones_like(cache_k, dtype=torch.bool)
    mask[0, :, 5] = False
    assert not cache_k[mask].any() and not cache_v[mask].any()


def _fp8_append_case(pkv, k_rows_f32, v_rows_f32, k_scale, v_scale, in_dtype):
    """Quantise rows [T, H, D] into an empty cache through the C ABI; return the
    device codes and the oracle codes of the same rows."""
    d = gu.dev()
    T, H, D = k_rows_f32.shape
    kb, vb = wl.f32_to_bits(k_rows_f32, in_dtype), wl.f32_to_bits(v_rows_f32, in_dtype)
    nb = -(-T // 16)
    kc = torch.zeros(nb, H, 16, D, dtype=torch.uint8, device=d)
    vc = torch.zeros_like(kc)
    slots = torch.arange(T, dtype=torch.int64, device=d)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    ks = torch.tensor(k_scale, dtype=torch.float32, device=d)
    vs = torch.tensor(v_scale, dtype=torch.float32, device=d)
    pkv.pkv_kv_append_fp8(gu.bits_to_torch(kb, in_dtype), gu.bits_to_torch(vb, in_dtype), slots, kc, vc, ks, vs,
                          err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got_k = kc.cpu().numpy().transpose(0, 2, 1, 3).reshape(nb * 16, H, D)[:T]
    got_v = vc.cpu().numpy().transpose(0, 2, 1, 3).reshape(nb * 16, H, D)[:T]
    ref_k = np.stack([oe.encode(wl.bits_to_f32(kb[:, h], in_dtype), k_scale[h]) for h in range(H)], axis=1)
    ref_v = np.stack([oe.encode(wl.bits_to_f32(vb[:, h], in_dtype), v_scale[h]) for h in range(H)], axis=1)
    return got_k, ref_k, got_v, ref_v


@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
def test_fp8_append_random_rows_bit_exact(pkv, in_dtype):
    rng = np.random.default_rng(11)
    k = rng.standard_normal((300, 8, 128)).astype(np.float32)
    v = rng.standard_normal((300, 8, 128)).astype(np.float32) * 3
    ks = (np.abs(k).max(axis=(0, 2)) / 448).astype(np.float32)
    vs = (np.abs(v).max(axis=(0, 2)) / 448 * 0.5).astype(np.float32)     # half scale -> saturation too
    gk, rk, gv, rv = _fp8_append_case(pkv, k, v, ks, vs, in_dtype)
    assert np.array_equal(gk, rk)
    assert np.array_equal(gv, rv)


def test_fp8_append_special_values(pkv):
    # exact E4M3 values, midpoints between neighbours (ties to even), the
    # saturation boundary and signed zeros, with scale 1
    vals = oe.decode(np.arange(0x7F))
    mids = (vals[:-1] + vals[1:]) / 2
    special = np.array([0.0, -0.0, 448.0, 450.0, 464.0, 480.0, 1024.0, -16384.0, 2.0 ** -10, 3 * 2.0 ** -10,
                        -2.0 ** -12])
    x = np.concatenate([vals, -vals, mids, -mids, special]).astype(np.float32)
    # bf16 holds every E4M3 value and midpoint exactly
    assert np.array_equal(wl.bits_to_f32(wl.f32_to_bits(x, "bf16"), "bf16"), x)
    n = len(x)
    T = -(-n // 64)
    pad = np.zeros(T * 64, dtype=np.float32)
    pad[:n] = x
    rows = pad.reshape(T, 1, 64)
    gk, rk, gv, rv = _fp8_append_case(pkv, rows, -rows, np.ones(1, np.float32), np.ones(1, np.float32), "bf16")
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)
