"""Decode attention over a paged KV cache, in float64 (oracle; test infrastructure only).

Sources:

* "KV Cache, the memory notepad ..." section 二: Attention(Q, K, V) =
  softmax(Q K^T / sqrt(d)) V; section 三: at a decode step the new token's
  query attends over every cached K/V of its sequence (the history plus the
  token itself, whose K/V were just appended); section 四: the softmax
  subtracts the row maximum before exponentiating.
* "KV Cache: principle and memory share (kp-013)" section 图示: decode step t
  computes attention(Q_t x KV[0..t-1]).
* "Series 03: why the KV cache eats memory ..." section 3.1: the sequence's
  K/V rows are found through its block table; physical blocks may be anywhere.
* "KV Cache, the memory notepad ..." section 六 (GQA): several query heads
  share one KV head.  Reading: query head h uses KV head h // G with
  G = H_q / H_kv (contiguous groups).
* "KV cache capacity planning ..." section 3: paging changes how memory is
  allocated, not the numbers: paged and contiguous attention agree.

Definition computed for every sequence b and query head h (g = h // G,
n = context_lens[b]):
    K_j = k_cache[table[b][j // bs], g, j % bs, :],  V_j likewise, j < n
    s_j = scale * <q[b, h], K_j>
    p_j = exp(s_j - max_i s_i) / sum_i exp(s_i - max_i s_i)
    out[b, h] = sum_j p_j V_j
An empty context (n = 0) gives out = 0 (a reading; the pages do not say).
Table entries past ceil(n / bs) are never read.
"""
from __future__ import annotations

import numpy as np


def gather_sequence(cache: np.ndarray, table_row, n: int, kv_head: int) -> np.ndarray:
    """Rows 0..n-1 of one sequence for one KV head: [n, head_dim].  Row j is
    read from physical block table_row[j // bs] at offset j % bs."""
    block_size = cache.shape[2]
    j = np.arange(n)
    blocks = np.asarray(table_row)[j // block_size]
    return cache[blocks, kv_head, j % block_size, :]


def softmax_weights(q_vec: np.ndarray, keys: np.ndarray, scale: float) -> np.ndarray:
    """p_j = softmax_j(scale * <q, K_j>) with the maximum subtracted first."""
    s = scale * (keys @ q_vec)
    e = np.exp(s - s.max())
    return e / e.sum()


def attend(q_vec: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """sum_j p_j V_j for one query vector; zeros when there are no keys."""
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1], dtype=np.float64)
    return softmax_weights(q_vec, keys, scale) @ values


def decode_one(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
               block_tables, context_lens, scale: float, b: int, h: int) -> np.ndarray:
    """out[b, h] alone (used to check sampled outputs of large workloads)."""
    group = q.shape[1] // k_cache.shape[1]
    g = h // group
    n = int(context_lens[b])
    keys = gather_sequence(k_cache, block_tables[b], n, g)
    values = gather_sequence(v_cache, block_tables[b], n, g)
    return attend(q[b, h], keys, values, scale)


def paged_decode_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                           block_tables, context_lens, scale: float) -> np.ndarray:
    """out [B, H_q, d] in float64.  q is [B, H_q, d]; the caches are
    [num_blocks, H_kv, block_size, d] holding exact float64 values."""
    batch, n_q_heads, head_dim = q.shape
    n_kv_heads = k_cache.shape[1]
    if n_q_heads % n_kv_heads:
        raise ValueError("H_q must be a multiple of H_kv")
    group = n_q_heads // n_kv_heads
    out = np.zeros((batch, n_q_heads, head_dim), dtype=np.float64)
    for b in range(batch):
        n = int(context_lens[b])
        for g in range(n_kv_heads):
            keys = gather_sequence(k_cache, block_tables[b], n, g)
            values = gather_sequence(v_cache, block_tables[b], n, g)
            for h in range(g * group, (g + 1) * group):
                out[b, h] = attend(q[b, h], keys, values, scale)
    return out


def contiguous_decode_attention(q: np.ndarray, k_seq: np.ndarray, v_seq: np.ndarray,
                                scale: float) -> np.ndarray:
    """The same attention for ONE sequence whose K/V are stored contiguously
    as [n, H_kv, d] (the no-cache comparator); q is [H_q, d]."""
    n_q_heads = q.shape[0]
    n_kv_heads = k_seq.shape[1]
    group = n_q_heads // n_kv_heads
    out = np.zeros(q.shape, dtype=np.float64)
    for h in range(n_q_heads):
        g = h // group
        out[h] = attend(q[h], k_seq[:, g, :], v_seq[:, g, :], scale)
    return out


def dequantize_cache(codes_values: np.ndarray, head_scales) -> np.ndarray:
    """FP8 cache of decoded code values [NB, H_kv, bs, d] times the per-head
    scale ("KV cache capacity planning ..." section 5: dequantise, then
    compute).  The caller decodes the codes with ``oracle.e4m3.decode``."""
    scales = np.asarray(head_scales, dtype=np.float64).reshape(1, -1, 1, 1)
    return codes_values * scales


def layer_view(cache: np.ndarray, layer: int) -> np.ndarray:
    """Layer ``layer`` of a model-wide cache [num_blocks, num_layers, H_kv,
    block_size, d] ("What a KV cache is ..." section 2.2: one preallocated
    cache laid out as (num_blocks, num_layers, num_kv_heads, block_size,
    head_dim), so one block id covers a token range in every layer): the
    [num_blocks, H_kv, block_size, d] cache that layer's attention reads."""
    return cache[:, layer]
