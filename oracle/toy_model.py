"""A tiny attention layer that recomputes every K/V from the hidden states
(oracle; test infrastructure only).

Sources:

* "KV Cache, the memory notepad ..." section 一: without a cache every new
  token recomputes the Keys and Values of the whole prefix (O(n^2) work);
  section 四: a toy layer with random projection matrices W_q, W_k, W_v whose
  output is the same with and without the cache.
* "KV Cache: principle and memory share (kp-013)" section 核心概念: the history's
  K/V depend only on the history, which is why caching them is exact.

This module only holds the no-cache side: projections and a from-scratch
recomputation of decode step t.  The cached side (slot mapping, append, paged
decode attention) is assembled from the other oracle modules by the tests.
"""
from __future__ import annotations

import numpy as np

from .attention import attend


class ToyAttentionLayer:
    """Projections x -> q [H_q, d], k [H_kv, d], v [H_kv, d]."""

    def __init__(self, w_q: np.ndarray, w_k: np.ndarray, w_v: np.ndarray,
                 n_q_heads: int, n_kv_heads: int, head_dim: int) -> None:
        self.w_q, self.w_k, self.w_v = w_q, w_k, w_v
        self.n_q_heads, self.n_kv_heads, self.head_dim = n_q_heads, n_kv_heads, head_dim

    def project(self, x: np.ndarray):
        q = (x @ self.w_q).reshape(self.n_q_heads, self.head_dim)
        k = (x @ self.w_k).reshape(self.n_kv_heads, self.head_dim)
        v = (x @ self.w_v).reshape(self.n_kv_heads, self.head_dim)
        return q, k, v

    def recompute_step(self, hidden: np.ndarray, t: int, scale: float) -> np.ndarray:
        """Output [H_q, d] of decode step t computed with no cache: K and V
        of tokens 0..t are projected again from ``hidden`` and token t's
        query attends over all t + 1 of them."""
        q_t, _, _ = self.project(hidden[t])
        keys = np.stack([self.project(hidden[j])[1] for j in range(t + 1)])    # [t+1, H_kv, d]
        values = np.stack([self.project(hidden[j])[2] for j in range(t + 1)])
        group = self.n_q_heads // self.n_kv_heads
        out = np.zeros((self.n_q_heads, self.head_dim))
        for h in range(self.n_q_heads):
            out[h] = attend(q_t[h], keys[:, h // group, :], values[:, h // group, :], scale)
        return out
