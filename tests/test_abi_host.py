"""CPU-only checks of the C ABI: every declared symbol is exported, argument
validation that returns before any CUDA call, and the host block pool against
the oracle's pool."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from oracle.block_pool import BlockPool as OraclePool, PoolExhausted, blocks_needed

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__ as g
    g.build()
    import paged_kv_cache_153_gb300 as m
    return m


# each header and the library that exports what it declares
HEADER_LIBRARIES = {"pkv.h": "libpkv.so", "pkv_prefill.h": "libpkv_prefill.so"}


def declared_symbols(header=None):
    names = set()
    for fname in os.listdir(os.path.join(ROOT, "include")):
        if fname.endswith(".h") and (header is None or fname == header):
            text = open(os.path.join(ROOT, "include", fname)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text))
    return names


def test_every_header_has_a_library():
    headers = {f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")}
    assert headers == set(HEADER_LIBRARIES)


@pytest.mark.parametrize("header", sorted(HEADER_LIBRARIES))
def test_every_declared_symbol_is_exported(pkv, header):
    names = declared_symbols(header)
    if header == "pkv.h":
        assert {"pkv_kv_append", "pkv_paged_decode_attention", "pkv_paged_decode_attention_fp8"} <= names
    else:
        assert names == {"pkv_paged_prefill_attention"}
    lib = C.CDLL(os.path.join(os.path.dirname(pkv.library_path), HEADER_LIBRARIES[header]))
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing


def test_decode_library_holds_no_prefill_kernel(pkv):
    # a decode-only process never loads the clustered prefill kernel
    lib = C.CDLL(pkv.library_path)
    assert not hasattr(lib, "pkv_paged_prefill_attention")


def test_status_strings(pkv):
    assert pkv.pkv_status_string(0) == "ok"
    assert "workspace" in pkv.pkv_status_string(6)
    assert pkv.pkv_version() >= 100


def test_validation_before_any_cuda_call(pkv):
    lib = pkv.lib
    dummy = C.c_void_p(16)
    # group 3 is not built
    st = lib.pkv_paged_decode_attention(dummy, dummy, dummy, dummy, dummy, 2, 6, 2, 128, 16, 4, 8, 64,
                                        0.1, dummy, 0, 0, dummy, 1 << 20, None, None)
    assert st == 2
    # H_q not a multiple of H_kv
    st = lib.pkv_paged_decode_attention(dummy, dummy, dummy, dummy, dummy, 2, 5, 2, 128, 16, 4, 8, 64,
                                        0.1, dummy, 0, 0, dummy, 1 << 20, None, None)
    assert st == 1
    # block size other than 16, head_dim 96
    assert lib.pkv_kv_append(dummy, dummy, dummy, 1, dummy, dummy, 4, 2, 128, 32, 0, None, None) == 2
    assert lib.pkv_kv_append(dummy, dummy, dummy, 1, dummy, dummy, 4, 2, 96, 16, 0, None, None) == 2
    # partition not a multiple of the block size
    st = lib.pkv_paged_decode_attention(dummy, dummy, dummy, dummy, dummy, 2, 4, 2, 128, 16, 4, 8, 64,
                                        0.1, dummy, 0, 24, dummy, 1 << 20, None, None)
    assert st == 1
    # empty work is a no-op
    assert lib.pkv_kv_append(None, None, None, 0, None, None, 4, 2, 128, 16, 0, None, None) == 0
    # null pointers with work
    assert lib.pkv_kv_append(None, dummy, dummy, 1, dummy, dummy, 4, 2, 128, 16, 0, None, None) == 1


@pytest.mark.parametrize("seed", range(4))
def test_host_pool_matches_oracle_pool(pkv, seed):
    rng = np.random.default_rng(seed)
    n = 37
    ours, ref = pkv.BlockPool(n), OraclePool(n)
    held = []
    for _ in range(600):
        op = rng.integers(3)
        if op == 0:
            try:
                b = ref.alloc()
            except PoolExhausted:
                with pytest.raises(pkv.PkvError) as ei:
                    ours.alloc()
                assert ei.value.status == 3
                continue
            assert ours.alloc() == b
            held.append(b)
        elif op == 1 and held:
            b = held[rng.integers(len(held))]
            ref.incref(b)
            ours.incref(b)
            held.append(b)
        elif op == 2 and held:
            b = held.pop(rng.integers(len(held)))
            ref.decref(b)
            ours.decref(b)
        assert ours.num_free == ref.num_free
    for b in range(n):
        assert ours.refcount(b) == ref.refcount(b)
    with pytest.raises(pkv.PkvError):
        ours.incref(n + 5)


def test_blocks_needed(pkv):
    for t in [0, 1, 15, 16, 17, 1200, 65536]:
        assert pkv.pkv_blocks_needed(t) == blocks_needed(t)


def test_int8_step_validates_everything_before_its_first_launch(pkv):
    # the INT8 step launches the re-quantising append before the decode, so
    # every argument the decode would refuse is refused before the append
    # writes the cache (no CUDA call is needed to see these)
    lib = pkv.lib
    a = C.c_void_p(4096)          # 16-byte aligned stand-in pointers
    odd = C.c_void_p(4096 + 8)

    def step(q=a, kc=a, vc=a, prm=a, out=a, ws=a, hq=32, hkv=8, part=0):
        return lib.pkv_paged_decode_step_int8(q, a, a, kc, vc, prm, a, a, 4, hq, hkv, 128, 16, 8, 64, 128, 0.1,
                                              out, 1, part, None, ws, 1 << 24, None, None)
    assert step(kc=odd) == 1 and step(vc=odd) == 1 and step(prm=odd) == 1
    assert step(q=None) == 1 and step(out=None) == 1 and step(ws=None) == 1
    assert step(q=odd) == 1 and step(out=odd) == 1 and step(ws=odd) == 1
    assert step(hq=30) == 1            # H_q not a multiple of H_kv
    assert step(part=24) == 1          # partition not a multiple of the block size
    assert step(hq=24) == 2            # group 3 is not built
    # the plain INT8 append wants aligned caches as well
    assert lib.pkv_kv_append_int8(a, a, a, 1, odd, a, a, 64, 8, 128, 16, 1, None, None) == 1
