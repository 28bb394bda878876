"""Python binding of libpkv.so, the sm_103a paged KV-cache decode library.

Argument marshalling only: every function here extracts device pointers,
sizes and the current CUDA stream from torch tensors and calls the C entry
point of the same name (declared in include/pkv.h).  All arithmetic runs in
the library's CUDA kernels; there is no CPU fallback.  Importing this module
fails loudly when the library has not been built (``__graft_entry__.build()``
or ``python -m paged_kv_cache_153_gb300._build``).

Tensors: 16-bit data is passed as torch.float16 / torch.bfloat16 (or any
2-byte dtype, tagged with ``dtype``), E4M3 caches as torch.uint8, tables and
lengths as torch.int32, slot mappings as torch.int64.
"""
from __future__ import annotations

import ctypes as C
import os

__all__ = [
    "PKV_F16", "PKV_BF16", "PkvError", "lib", "library_path",
    "pkv_slot_mapping", "pkv_kv_append", "pkv_kv_append_fp8", "pkv_decode_workspace_bytes",
    "pkv_paged_decode_attention", "pkv_paged_decode_attention_fp8", "pkv_decode_step_host",
    "pkv_paged_decode_attention_noalloc", "pkv_paged_decode_step", "pkv_paged_decode_step_fp8",
    "BlockPool", "pkv_blocks_needed", "pkv_version", "pkv_status_string", "pkv_last_error",
    "pkv_copy_blocks", "pkv_prepare_append", "pkv_paged_prefill_attention", "pkv_paged_decode_step_layer",
    "StepGraph", "pkv_kv_quantize_int8", "pkv_kv_append_int8", "pkv_paged_decode_attention_int8",
    "pkv_kv_append_e5m2", "pkv_paged_decode_attention_e5m2", "pkv_paged_decode_step_e5m2",
    "pkv_paged_decode_step_int8",
]

PKV_F16 = 0
PKV_BF16 = 1
PKV_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024   # as in pkv.h
_DIR = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_DIR, "libpkv.so")

if not os.path.exists(library_path):
    raise ImportError(f"{library_path} is missing: build it with __graft_entry__.build() "
                      "(the CUDA path has no fallback)")
lib = C.CDLL(library_path)

# The prefill kernel lives in a library of its own (pkv_prefill.h), loaded on
# first use, so that a process that only decodes never loads it.
prefill_library_path = os.path.join(_DIR, "libpkv_prefill.so")
_prefill_lib = None


def prefill_lib():
    global _prefill_lib
    if _prefill_lib is None:
        if not os.path.exists(prefill_library_path):
            raise ImportError(f"{prefill_library_path} is missing: build it with __graft_entry__.build()")
        pl = C.CDLL(prefill_library_path)
        pl.pkv_paged_prefill_attention.restype = C.c_int
        pl.pkv_paged_prefill_attention.argtypes = _PREFILL_SIG
        _prefill_lib = pl
    return _prefill_lib

_p, _i, _i64, _sz, _f = C.c_void_p, C.c_int, C.c_int64, C.c_size_t, C.c_float
_SIGS = {
    "pkv_version": (_i, []),
    "pkv_status_string": (C.c_char_p, [_i]),
    "pkv_last_error": (C.c_char_p, []),
    "pkv_slot_mapping": (_i, [_p, _i, _i64, _p, _p, C.c_int32, _i64, _i, _p, _p, _p]),
    "pkv_kv_append": (_i, [_p, _p, _p, _i64, _p, _p, _i64, _i, _i, _i, _i, _p, _p]),
    "pkv_kv_append_fp8": (_i, [_p, _p, _p, _i64, _p, _p, _i64, _p, _p, _i, _i, _i, _i, _p, _p]),
    "pkv_kv_append_e5m2": (_i, [_p, _p, _p, _i64, _p, _p, _i64, _p, _p, _i, _i, _i, _i, _p, _p]),
    "pkv_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "pkv_paged_decode_attention": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _f, _p, _i, _i,
                                        _p, _sz, _p, _p]),
    "pkv_paged_decode_attention_fp8": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _f,
                                            _p, _i, _i, _p, _sz, _p, _p]),
    "pkv_paged_decode_attention_e5m2": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _f,
                                             _p, _i, _i, _p, _sz, _p, _p]),
    "pkv_paged_decode_step": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _f, _p, _i, _i, _p,
                                   _p, _sz, _p, _p]),
    "pkv_paged_decode_step_fp8": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _f, _p,
                                       _i, _i, _p, _p, _sz, _p, _p]),
    "pkv_paged_decode_step_e5m2": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _f,
                                        _p, _i, _i, _p, _p, _sz, _p, _p]),
    "pkv_paged_decode_attention_noalloc": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _f, _p, _i,
                                                _i, _p, _p]),
    "pkv_decode_step_host": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i,
                                  _i, _i, _i64, _i, _f, _i, _i, _p, _sz, _p, _p]),
    "pkv_pool_create": (_p, [_i64, _i]),
    "pkv_pool_destroy": (None, [_p]),
    "pkv_pool_alloc": (_i, [_p, C.POINTER(C.c_int32)]),
    "pkv_pool_incref": (_i, [_p, C.c_int32]),
    "pkv_pool_decref": (_i, [_p, C.c_int32]),
    "pkv_pool_num_free": (_i64, [_p]),
    "pkv_pool_refcount": (C.c_int32, [_p, C.c_int32]),
    "pkv_blocks_needed": (_i64, [_i64, _i]),
    "pkv_pool_cow": (_i, [_p, C.c_int32, C.POINTER(C.c_int32)]),
    "pkv_prepare_append": (_i, [_p, _p, _i, _i, _p, _p, _p, C.POINTER(C.c_int32)]),
    "pkv_copy_blocks": (_i, [_p, _p, _i64, _p, _p, _i64, _i, _i, _i, _i, _p, _p]),
    "pkv_paged_decode_step_layer": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _i, _i, _f,
                                         _p, _i, _i, _p, _p, _sz, _p, _p]),
    "pkv_step_graph_create": (_i, [C.POINTER(_p), _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i,
                                   _i, _f, _p, _i, _i, _p, _p, _sz, _p]),
    "pkv_step_graph_launch": (_i, [_p, _p]),
    "pkv_step_graph_destroy": (None, [_p]),
    "pkv_kv_quantize_int8": (_i, [_p, _p, _p, _p, _p, _p, _i64, _i, _i, _i, _i, _p, _p]),
    "pkv_kv_append_int8": (_i, [_p, _p, _p, _i64, _p, _p, _p, _i64, _i, _i, _i, _i, _p, _p]),
    "pkv_paged_decode_attention_int8": (_i, [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _f, _p, _i,
                                             _i, _p, _sz, _p, _p]),
    "pkv_paged_decode_step_int8": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _f, _p, _i,
                                        _i, _p, _p, _sz, _p, _p]),
}
_PREFILL_SIG = [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i64, _i, _f, _p, _i, _p, _p]
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        detail = f": {pkv_last_error()}" if status == 5 else ""
        super().__init__(f"{fn}: {pkv_status_string(status)} (status {status}){detail}")
        self.status = status


def pkv_version() -> int:
    return lib.pkv_version()


def pkv_status_string(status: int) -> str:
    return lib.pkv_status_string(status).decode()


def pkv_last_error() -> str:
    return lib.pkv_last_error().decode()


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise PkvError(fn, status)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _dtype_code(t, dtype) -> int:
    if dtype is not None:
        return dtype
    import torch
    if t.dtype == torch.float16:
        return PKV_F16
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"cannot infer the 16-bit kind of {t.dtype}; pass dtype=PKV_F16/PKV_BF16")


def pkv_slot_mapping(block_tables, positions, slot_mapping, *, num_blocks: int, seq_idx=None,
                     position_offset: int = 0, block_size: int = 16, err_flag=None, stream=None) -> None:
    n = positions.numel()
    _check("pkv_slot_mapping", lib.pkv_slot_mapping(
        _ptr(block_tables), block_tables.shape[1], num_blocks, _ptr(seq_idx), _ptr(positions),
        position_offset, n, block_size, _ptr(slot_mapping), _ptr(err_flag), _stream(stream)))


def pkv_kv_append(k_new, v_new, slot_mapping, k_cache, v_cache, *, dtype=None, err_flag=None,
                  stream=None) -> None:
    nb, hkv, bs, d = k_cache.shape
    _check("pkv_kv_append", lib.pkv_kv_append(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), slot_mapping.numel(), _ptr(k_cache), _ptr(v_cache),
        nb, hkv, d, bs, _dtype_code(k_new, dtype), _ptr(err_flag), _stream(stream)))


def _append_fp8(fn, k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, in_dtype, err_flag, stream):
    nb, hkv, bs, d = k_cache.shape
    _check(fn, getattr(lib, fn)(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), slot_mapping.numel(), _ptr(k_cache), _ptr(v_cache),
        nb, _ptr(k_scale), _ptr(v_scale), hkv, d, bs, _dtype_code(k_new, in_dtype), _ptr(err_flag),
        _stream(stream)))


def pkv_kv_append_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, *, in_dtype=None,
                      err_flag=None, stream=None) -> None:
    """E4M3 append: uint8 caches [NB, Hkv, 16, D], fp32 per-head scales."""
    _append_fp8("pkv_kv_append_fp8", k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, in_dtype,
                err_flag, stream)


def pkv_kv_append_e5m2(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, *, in_dtype=None,
                       err_flag=None, stream=None) -> None:
    """E5M2 append: uint8 caches [NB, Hkv, 16, D], fp32 per-head scales."""
    _append_fp8("pkv_kv_append_e5m2", k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, in_dtype,
                err_flag, stream)


def pkv_decode_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                               max_blocks_per_seq: int, max_context_len: int,
                               partition_tokens: int = 0) -> int:
    n = lib.pkv_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                       max_context_len, partition_tokens)
    if n == 0 and batch > 0:
        raise PkvError("pkv_decode_workspace_bytes", 1)
    return n


def pkv_paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, out, *, scale: float,
                               max_context_len: int, workspace, partition_tokens: int = 0, dtype=None,
                               err_flag=None, stream=None) -> None:
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_paged_decode_attention", lib.pkv_paged_decode_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), b, hq, hkv, d, bs,
        block_tables.shape[1], nb, max_context_len, scale, _ptr(out), _dtype_code(q, dtype), partition_tokens,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err_flag), _stream(stream)))


def _decode_fp8(fn, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, out, scale,
                max_context_len, workspace, partition_tokens, q_dtype, err_flag, stream):
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check(fn, getattr(lib, fn)(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
        _ptr(context_lens), b, hq, hkv, d, bs, block_tables.shape[1], nb, max_context_len, scale, _ptr(out),
        _dtype_code(q, q_dtype), partition_tokens, _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(err_flag), _stream(stream)))


def pkv_paged_decode_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, out, *,
                                   scale: float, max_context_len: int, workspace, partition_tokens: int = 0,
                                   q_dtype=None, err_flag=None, stream=None) -> None:
    _decode_fp8("pkv_paged_decode_attention_fp8", q, k_cache, v_cache, k_scale, v_scale, block_tables,
                context_lens, out, scale, max_context_len, workspace, partition_tokens, q_dtype, err_flag, stream)


def pkv_paged_decode_attention_e5m2(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, out, *,
                                    scale: float, max_context_len: int, workspace, partition_tokens: int = 0,
                                    q_dtype=None, err_flag=None, stream=None) -> None:
    _decode_fp8("pkv_paged_decode_attention_e5m2", q, k_cache, v_cache, k_scale, v_scale, block_tables,
                context_lens, out, scale, max_context_len, workspace, partition_tokens, q_dtype, err_flag, stream)


def pkv_paged_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, *, scale: float,
                          max_context_len: int, workspace, partition_tokens: int = 0, slot_mapping_out=None,
                          dtype=None, err_flag=None, stream=None) -> None:
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_paged_decode_step", lib.pkv_paged_decode_step(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), b,
        hq, hkv, d, bs, block_tables.shape[1], nb, max_context_len, scale, _ptr(out), _dtype_code(q, dtype),
        partition_tokens, _ptr(slot_mapping_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(err_flag), _stream(stream)))


def _step_fp8(fn, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, out, scale,
              max_context_len, workspace, partition_tokens, slot_mapping_out, q_dtype, err_flag, stream):
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check(fn, getattr(lib, fn)(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
        _ptr(block_tables), _ptr(context_lens), b, hq, hkv, d, bs, block_tables.shape[1], nb, max_context_len, scale,
        _ptr(out), _dtype_code(q, q_dtype), partition_tokens, _ptr(slot_mapping_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err_flag), _stream(stream)))


def pkv_paged_decode_step_fp8(q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                              out, *, scale: float, max_context_len: int, workspace, partition_tokens: int = 0,
                              slot_mapping_out=None, q_dtype=None, err_flag=None, stream=None) -> None:
    _step_fp8("pkv_paged_decode_step_fp8", q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables,
              context_lens, out, scale, max_context_len, workspace, partition_tokens, slot_mapping_out, q_dtype,
              err_flag, stream)


def pkv_paged_decode_step_e5m2(q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                               out, *, scale: float, max_context_len: int, workspace, partition_tokens: int = 0,
                               slot_mapping_out=None, q_dtype=None, err_flag=None, stream=None) -> None:
    _step_fp8("pkv_paged_decode_step_e5m2", q, k_new, v_new, k_cache, v_cache, k_scale, v_scale, block_tables,
              context_lens, out, scale, max_context_len, workspace, partition_tokens, slot_mapping_out, q_dtype,
              err_flag, stream)


def pkv_paged_decode_attention_noalloc(q, k_cache, v_cache, block_tables, context_lens, out, *, scale: float,
                                       max_context_len: int, partition_tokens: int = 0, dtype=None,
                                       err_flag=None, stream=None) -> None:
    """Decode attention with the library's fixed device scratch instead of a
    caller workspace (for callers that cannot allocate)."""
    b, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_paged_decode_attention_noalloc", lib.pkv_paged_decode_attention_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), b, hq, hkv, d, bs,
        block_tables.shape[1], nb, max_context_len, scale, _ptr(out), _dtype_code(q, dtype), partition_tokens,
        _ptr(err_flag), _stream(stream)))


def pkv_decode_step_host(h_q, h_k_new, h_v_new, h_block_tables, h_context_lens, h_out, d_q, d_k_new, d_v_new,
                         d_block_tables, d_context_lens, d_slots, d_out, k_cache, v_cache, *, scale: float,
                         max_context_len: int, workspace, partition_tokens: int = 0, dtype=None,
                         err_flag=None, stream=None) -> None:
    b, hq, d = h_q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_decode_step_host", lib.pkv_decode_step_host(
        _ptr(h_q), _ptr(h_k_new), _ptr(h_v_new), _ptr(h_block_tables), _ptr(h_context_lens), _ptr(h_out),
        _ptr(d_q), _ptr(d_k_new), _ptr(d_v_new), _ptr(d_block_tables), _ptr(d_context_lens), _ptr(d_slots),
        _ptr(d_out), _ptr(k_cache), _ptr(v_cache), b, hq, hkv, d, bs, h_block_tables.shape[1], nb,
        max_context_len, scale, _dtype_code(h_q, dtype), partition_tokens, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err_flag), _stream(stream)))


def pkv_copy_blocks(src_blocks, dst_blocks, k_cache, v_cache, *, err_flag=None, stream=None) -> None:
    """Copy-on-write block copy on the device: block dst_blocks[i] of both
    caches takes block src_blocks[i] (int32 device tensors of equal length)."""
    nb, hkv, bs, d = k_cache.shape
    _check("pkv_copy_blocks", lib.pkv_copy_blocks(
        _ptr(src_blocks), _ptr(dst_blocks), src_blocks.numel(), _ptr(k_cache), _ptr(v_cache), nb, hkv, d, bs,
        k_cache.element_size(), _ptr(err_flag), _stream(stream)))


def pkv_prepare_append(pool: "BlockPool", block_tables, context_lens):
    """Host side of one decode step over shared blocks (pkv_prepare_append):
    updates the int32 host array block_tables [batch, max_blocks] in place and
    returns the copy pairs (src, dst) as two int32 numpy arrays."""
    import numpy as np
    assert block_tables.dtype == np.int32 and block_tables.flags["C_CONTIGUOUS"]
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    batch, max_blocks = block_tables.shape
    src = np.empty(max(batch, 1), dtype=np.int32)
    dst = np.empty(max(batch, 1), dtype=np.int32)
    n = C.c_int32(0)
    _check("pkv_prepare_append", lib.pkv_prepare_append(
        pool._h, block_tables.ctypes.data, batch, max_blocks, lens.ctypes.data, src.ctypes.data,
        dst.ctypes.data, C.byref(n)))
    return src[:n.value].copy(), dst[:n.value].copy()


def pkv_paged_prefill_attention(q, k_cache, v_cache, block_tables, context_lens, cu_seqlens, out, *, scale: float,
                                max_query_len: int, dtype=None, err_flag=None, stream=None) -> None:
    """Causal extend attention of the new tokens q [T, Hq, D] over the paged
    cache (which already holds their K/V)."""
    nb, hkv, bs, d = k_cache.shape
    _check("pkv_paged_prefill_attention", prefill_lib().pkv_paged_prefill_attention(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), _ptr(cu_seqlens),
        context_lens.numel(), q.shape[1], hkv, d, bs, block_tables.shape[1], nb, max_query_len, scale, _ptr(out),
        _dtype_code(q, dtype), _ptr(err_flag), _stream(stream)))


def pkv_paged_decode_step_layer(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, *, layer: int,
                                scale: float, max_context_len: int, workspace, partition_tokens: int = 0,
                                slot_mapping_out=None, dtype=None, err_flag=None, stream=None) -> None:
    """The fused decode step on layer ``layer`` of a layer-major cache
    [NB, L, Hkv, 16, D]."""
    nb, n_layers, hkv, bs, d = k_cache.shape
    _check("pkv_paged_decode_step_layer", lib.pkv_paged_decode_step_layer(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        q.shape[0], q.shape[1], hkv, d, bs, block_tables.shape[1], nb, n_layers, layer, max_context_len, scale,
        _ptr(out), _dtype_code(q, dtype), partition_tokens, _ptr(slot_mapping_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err_flag), _stream(stream)))


class StepGraph:
    """One decode step over every layer of a layer-major cache, captured into
    a CUDA graph by the library (pkv_step_graph_*): q, out [L, B, Hq, D];
    k_new, v_new [L, B, Hkv, D]; caches [NB, L, Hkv, 16, D].  The tensors must
    outlive the graph; ``launch`` replays the step with their current data."""

    def __init__(self, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, *, scale: float,
                 max_context_len: int, workspace, partition_tokens: int = 0, slot_mapping_out=None, dtype=None,
                 err_flag=None):
        nb, n_layers, hkv, bs, d = k_cache.shape
        h = _p()
        self._keep = (q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, workspace,
                      slot_mapping_out, err_flag)
        _check("pkv_step_graph_create", lib.pkv_step_graph_create(
            C.byref(h), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            _ptr(context_lens), q.shape[1], q.shape[2], hkv, d, bs, block_tables.shape[1], nb, n_layers,
            max_context_len, scale, _ptr(out), _dtype_code(q, dtype), partition_tokens, _ptr(slot_mapping_out),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err_flag)))
        self._h = h

    def launch(self, stream=None) -> None:
        _check("pkv_step_graph_launch", lib.pkv_step_graph_launch(self._h, _stream(stream)))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib.pkv_step_graph_destroy(h)
            self._h = None


def pkv_kv_quantize_int8(k_src, v_src, k_cache, v_cache, slab_params, *, rows_used=None, dtype=None,
                         err_flag=None, stream=None) -> None:
    """INT8 codes and per-(block, head) (k_min, k_max, v_min, v_max) of 16-bit pools."""
    nb, hkv, bs, d = k_cache.shape
    _check("pkv_kv_quantize_int8", lib.pkv_kv_quantize_int8(
        _ptr(k_src), _ptr(v_src), _ptr(k_cache), _ptr(v_cache), _ptr(slab_params), _ptr(rows_used), nb, hkv, d, bs,
        _dtype_code(k_src, dtype), _ptr(err_flag), _stream(stream)))


def pkv_kv_append_int8(k_new, v_new, slot_mapping, k_cache, v_cache, slab_params, *, dtype=None, err_flag=None,
                       stream=None) -> None:
    nb, hkv, bs, d = k_cache.shape
    _check("pkv_kv_append_int8", lib.pkv_kv_append_int8(
        _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), slot_mapping.numel(), _ptr(k_cache), _ptr(v_cache),
        _ptr(slab_params), nb, hkv, d, bs, _dtype_code(k_new, dtype), _ptr(err_flag), _stream(stream)))


def pkv_paged_decode_attention_int8(q, k_cache, v_cache, slab_params, block_tables, context_lens, out, *,
                                    scale: float, max_context_len: int, workspace, partition_tokens: int = 0,
                                    q_dtype=None, err_flag=None, stream=None) -> None:
    nb, hkv, bs, d = k_cache.shape
    _check("pkv_paged_decode_attention_int8", lib.pkv_paged_decode_attention_int8(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(slab_params), _ptr(block_tables), _ptr(context_lens),
        q.shape[0], q.shape[1], hkv, d, bs, block_tables.shape[1], nb, max_context_len, scale, _ptr(out),
        _dtype_code(q, q_dtype), partition_tokens, _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(err_flag), _stream(stream)))


def pkv_paged_decode_step_int8(q, k_new, v_new, k_cache, v_cache, slab_params, block_tables, context_lens, out, *,
                               scale: float, max_context_len: int, workspace, partition_tokens: int = 0,
                               slot_mapping_out=None, q_dtype=None, err_flag=None, stream=None) -> None:
    """The INT8 decode step in one decode launch (head_dim 128): the new rows
    are appended with re-quantisation of their blocks, then attention."""
    nb, hkv, bs, d = k_cache.shape
    _check("pkv_paged_decode_step_int8", lib.pkv_paged_decode_step_int8(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slab_params), _ptr(block_tables),
        _ptr(context_lens), q.shape[0], q.shape[1], hkv, d, bs, block_tables.shape[1], nb, max_context_len, scale,
        _ptr(out), _dtype_code(q, q_dtype), partition_tokens, _ptr(slot_mapping_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(err_flag), _stream(stream)))


def pkv_blocks_needed(num_tokens: int, block_size: int = 16) -> int:
    return lib.pkv_blocks_needed(num_tokens, block_size)


class BlockPool:
    """The C-ABI host block pool (pkv_pool_*)."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        self._h = lib.pkv_pool_create(num_blocks, block_size)
        if not self._h:
            raise PkvError("pkv_pool_create", 1)
        self.num_blocks, self.block_size = num_blocks, block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib.pkv_pool_destroy(h)
            self._h = None

    def alloc(self) -> int:
        out = C.c_int32(-1)
        _check("pkv_pool_alloc", lib.pkv_pool_alloc(self._h, C.byref(out)))
        return out.value

    def incref(self, block_id: int) -> None:
        _check("pkv_pool_incref", lib.pkv_pool_incref(self._h, block_id))

    def decref(self, block_id: int) -> None:
        _check("pkv_pool_decref", lib.pkv_pool_decref(self._h, block_id))

    @property
    def num_free(self) -> int:
        return lib.pkv_pool_num_free(self._h)

    def refcount(self, block_id: int) -> int:
        return lib.pkv_pool_refcount(self._h, block_id)

    def cow(self, block_id: int) -> int:
        out = C.c_int32(-1)
        _check("pkv_pool_cow", lib.pkv_pool_cow(self._h, block_id, C.byref(out)))
        return out.value
