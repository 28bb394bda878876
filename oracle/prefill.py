"""Paged prefill / extend attention, in float64 (oracle; test infrastructure only).

Sources:

* "KV Cache, the memory notepad ..." section 三: prefill runs the whole prompt
  through the model at once and writes every prompt token's K/V into the
  cache; decode then adds one token per step.  Section 二: Attention(Q, K, V)
  = softmax(Q K^T / sqrt(d)) V; section 四: the softmax subtracts the row
  maximum.
* "What a KV cache is ..." section 3.2: a prompt is prefilled into the
  preallocated cache, then generation appends token by token.
* "Series 03: why the KV cache eats memory ..." section 5.1: with chunked
  prefill a long prompt is cut into chunks processed one after another, so a
  chunk's queries also see the chunks already in the cache.  Section 3.1:
  K/V rows are found through the block table.
* "KV Cache, the memory notepad ..." section 六 (GQA): query head h uses KV
  head h // G.

Reading (the pages print no mask; section 四's toy attends with the last
query only): token t of a sequence attends to the positions up to and
including its own -- the causal reading, under which prefilling n tokens
gives exactly what n decode steps would give.  The new tokens of sequence b
are its last n_b positions: with ctx_b = context_lens[b] (the length after
the new tokens were appended) and n_b = cu_seqlens[b+1] - cu_seqlens[b],
token i (0 <= i < n_b) sits at position p = ctx_b - n_b + i and

    out[cu_seqlens[b] + i, h] = sum_{j <= p} softmax_j(scale <q, K_j>) V_j,

K_j, V_j read from the paged cache of KV head h // G.
"""
from __future__ import annotations

import numpy as np

from oracle import attention as oa


def prefill_positions(context_lens, cu_seqlens):
    """(sequence, position) of every new token, in the order of cu_seqlens."""
    out = []
    for b in range(len(context_lens)):
        n = int(cu_seqlens[b + 1]) - int(cu_seqlens[b])
        start = int(context_lens[b]) - n
        if start < 0:
            raise ValueError("a sequence has more new tokens than context")
        out += [(b, start + i) for i in range(n)]
    return out


def paged_prefill_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, block_tables,
                            context_lens, cu_seqlens, scale: float, rows=None) -> np.ndarray:
    """out [T, H_q, d] in float64 for q [T, H_q, d] (T = cu_seqlens[-1]); the
    caches are [num_blocks, H_kv, block_size, d] of exact float64 values and
    already hold the new tokens' K/V.  ``rows``: compute only these token
    indices (the others stay zero)."""
    n_tokens, n_q_heads, head_dim = q.shape
    n_kv_heads = k_cache.shape[1]
    if n_q_heads % n_kv_heads:
        raise ValueError("H_q must be a multiple of H_kv")
    group = n_q_heads // n_kv_heads
    pos = prefill_positions(context_lens, cu_seqlens)
    if len(pos) != n_tokens:
        raise ValueError("q holds a different number of tokens than cu_seqlens")
    out = np.zeros((n_tokens, n_q_heads, head_dim), dtype=np.float64)
    for t in (range(n_tokens) if rows is None else rows):
        b, p = pos[t]
        for g in range(n_kv_heads):
            keys = oa.gather_sequence(k_cache, block_tables[b], p + 1, g)
            values = oa.gather_sequence(v_cache, block_tables[b], p + 1, g)
            for h in range(g * group, (g + 1) * group):
                out[t, h] = oa.attend(q[t, h], keys, values, scale)
    return out
