"""E5M2 KV cache on the GPU ("KV cache capacity planning ..." section 4: the
second FP8 format, wider exponent range and lower precision; section 5:
dequantised before the arithmetic).  The append is bit for bit the oracle's
encoder (oracle.e5m2); attention is within 2e-2 absolute of the float64
oracle fed the same codes and scales, as for E4M3."""
import numpy as np
import pytest
import torch

import pkv_workloads as wl
from oracle import e5m2 as o5

from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__ as g
    g.build()
    import paged_kv_cache_153_gb300 as m
    return m


def _append_case(pkv, k_rows_f32, v_rows_f32, k_scale, v_scale, in_dtype):
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
    pkv.pkv_kv_append_e5m2(gu.bits_to_torch(kb, in_dtype), gu.bits_to_torch(vb, in_dtype), slots, kc, vc, ks, vs,
                           err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got_k = kc.cpu().numpy().transpose(0, 2, 1, 3).reshape(nb * 16, H, D)[:T]
    got_v = vc.cpu().numpy().transpose(0, 2, 1, 3).reshape(nb * 16, H, D)[:T]
    with np.errstate(over="ignore"):
        ref_k = np.stack([o5.encode(wl.bits_to_f32(kb[:, h], in_dtype), k_scale[h]) for h in range(H)], axis=1)
        ref_v = np.stack([o5.encode(wl.bits_to_f32(vb[:, h], in_dtype), v_scale[h]) for h in range(H)], axis=1)
    return got_k, ref_k, got_v, ref_v


@pytest.mark.parametrize("in_dtype", ["bf16", "f16"])
def test_append_random_rows_bit_exact(pkv, in_dtype):
    rng = np.random.default_rng(12)
    k = rng.standard_normal((300, 8, 128)).astype(np.float32)
    v = rng.standard_normal((300, 8, 128)).astype(np.float32) * 3
    ks = (np.abs(k).max(axis=(0, 2)) / 57344).astype(np.float32)
    vs = (np.abs(v).max(axis=(0, 2)) / 57344 * 0.5).astype(np.float32)   # half scale -> saturation too
    gk, rk, gv, rv = _append_case(pkv, k, v, ks, vs, in_dtype)
    assert np.array_equal(gk, rk)
    assert np.array_equal(gv, rv)


def test_append_special_values(pkv):
    # every finite E5M2 value, the midpoints between neighbours (ties to
    # even), the saturation boundary, infinities, subnormal ties and signed
    # zeros, with scale 1
    vals = o5.decode(np.arange(0x7C))
    mids = (vals[:-1] + vals[1:]) / 2
    special = np.array([0.0, -0.0, 57344.0, 61440.0, 65536.0, 2.0 ** 20, -2.0 ** 25, np.inf, -np.inf, 2.0 ** -17,
                        3 * 2.0 ** -17, -2.0 ** -20])
    x = np.concatenate([vals, -vals, mids, -mids, special]).astype(np.float32)
    # bf16 holds every E5M2 value and midpoint exactly
    assert np.array_equal(wl.bits_to_f32(wl.f32_to_bits(x, "bf16"), "bf16"), x)
    n = len(x)
    T = -(-n // 64)
    pad = np.zeros(T * 64, dtype=np.float32)
    pad[:n] = x
    rows = pad.reshape(T, 1, 64)
    gk, rk, gv, rv = _append_case(pkv, rows, -rows, np.ones(1, np.float32), np.ones(1, np.float32), "bf16")
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


def _check(case, ref, label):
    max_abs, _, n_bad, _ = gu.compare_all(case.out, ref, gu.FP8_ATOL, 0.0)
    assert case.err_code() == 0, f"{label}: device error {case.err_code()}"
    assert n_bad == 0, f"{label}: {n_bad} elements beyond {gu.FP8_ATOL} (max abs {max_abs:.3e})"


@pytest.mark.parametrize("hq,hkv,head_dim", [(32, 8, 128), (16, 16, 128), (64, 8, 128), (16, 8, 128), (8, 4, 64),
                                             (8, 8, 64), (16, 2, 64)])
@pytest.mark.parametrize("partition", [0, 64])
def test_attention_shapes(pkv, hq, hkv, head_dim, partition):
    # every group size on both head dims: the tensor-core consumer (128-byte
    # rows, G >= 2) and the CUDA-core consumer (G = 1 or 64-byte rows)
    w = wl.build("e5m2shape", batch=6, n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim, dtype="bf16",
                 kv_dtype="e5m2", context_lens=[1, 16, 33, 250, 401, 1100], seed=hq * 7 + hkv + head_dim)
    kc, vc, _, _ = gu.oracle_fp8_codes(w)
    case = gu.GpuCase(w, codes=(kc, vc))
    case.step(partition_tokens=partition)
    kp, vp = gu.oracle_pools_after_append(w)
    assert np.array_equal(case.k_cache.cpu().numpy(), kp) and np.array_equal(case.v_cache.cpu().numpy(), vp)
    _check(case, gu.oracle_decode_all(w, kp, vp), f"e5m2 {hq}/{hkv} d{head_dim} P{partition}")


@pytest.mark.parametrize("hq,hkv,head_dim", [(32, 8, 128), (8, 8, 64), (16, 4, 64)])
def test_fused_step_equals_separate_calls(pkv, hq, hkv, head_dim):
    w = wl.build("e5m2fused", batch=5, n_q_heads=hq, n_kv_heads=hkv, head_dim=head_dim, dtype="bf16",
                 kv_dtype="e5m2", context_lens=[1, 16, 31, 200, 513], seed=hq + hkv + head_dim)
    kc, vc, _, _ = gu.oracle_fp8_codes(w)
    for partition in (0, 64):
        sep, fus = gu.GpuCase(w, codes=(kc.copy(), vc.copy())), gu.GpuCase(w, codes=(kc.copy(), vc.copy()))
        sep.step(partition_tokens=partition)
        fus.fused_step(partition_tokens=partition)
        torch.cuda.synchronize()
        assert sep.err_code() == 0 and fus.err_code() == 0
        assert torch.equal(fus.slots, sep.slots)
        assert torch.equal(fus.k_cache, sep.k_cache) and torch.equal(fus.v_cache, sep.v_cache)
        assert torch.equal(fus.out, sep.out)


def test_garbage_past_the_context_is_ignored(pkv):
    # NaN codes in the unused tail of each last block must not reach the output
    lens = [1, 15, 16, 17, 33, 100, 257]
    for hq, hkv, d in ((16, 4, 128), (8, 8, 64)):
        w = wl.build("e5m2poison", batch=len(lens), n_q_heads=hq, n_kv_heads=hkv, head_dim=d, dtype="bf16",
                     kv_dtype="e5m2", context_lens=lens, seed=hq + d)
        kc, vc, kn, vn = gu.oracle_fp8_codes(w)
        for b, n in enumerate(lens):
            if n % 16:
                blk = int(w.block_tables[b][(n - 1) // 16])
                kc[blk, :, n % 16:, :] = 0x7F
                vc[blk, :, n % 16:, :] = 0x7F
        case = gu.GpuCase(w, codes=(kc, vc))
        case.step(partition_tokens=0)
        slots = gu.oracle_slots(w)
        gu.osl.append_rows(kc, kn, slots)
        gu.osl.append_rows(vc, vn, slots)
        _check(case, gu.oracle_decode_all(w, kc, vc), f"e5m2 poison {hq}/{hkv}")
        assert bool(torch.isfinite(case.out).all())


@pytest.mark.slow
def test_full_size_long_mix_every_output(pkv):
    # the long-context mix (29 x 2048 + 3 x 65536 tokens, 32/8 heads, d 128, q
    # bf16) with an E5M2 cache: the fused step with 512-token partitions, as
    # the benchmark runs the E4M3 configuration; every output element
    w = wl.make("fp8long", fp8="e5m2")
    kc = gu.oracle_fp8_pool_codes(w, w.k_pool, w.k_scale)
    vc = gu.oracle_fp8_pool_codes(w, w.v_pool, w.v_scale)
    case = gu.GpuCase(w, codes=(kc, vc))
    case.fused_step()
    torch.cuda.synchronize()
    assert case.err_code() == 0
    slots = gu.oracle_slots(w)
    gu.osl.append_rows(kc, gu.oracle_fp8_pool_codes(w, w.k_new, w.k_scale), slots)
    gu.osl.append_rows(vc, gu.oracle_fp8_pool_codes(w, w.v_new, w.v_scale), slots)
    assert np.array_equal(case.k_cache.cpu().numpy(), kc) and np.array_equal(case.v_cache.cpu().numpy(), vc)
    ref = gu.oracle_decode_all(w, kc, vc)
    max_abs, max_rel, n_bad, n = gu.compare_all(case.out, ref, gu.FP8_ATOL, 0.0)
    gu.record_parity("fp8long_e5m2", split="partitions of 512", max_abs=max_abs, max_rel=max_rel, elements=n,
                     bad=n_bad)
    assert n_bad == 0, f"{n_bad} of {n} elements beyond {gu.FP8_ATOL} (max abs {max_abs:.3e})"
