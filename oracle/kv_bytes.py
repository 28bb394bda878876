"""Closed-form KV-cache byte counts (oracle; test infrastructure only).

The size of a KV cache follows from counting: for every cached token, every
layer stores one Key row and one Value row for each KV head, each row holding
``head_dim`` elements.  Sources:

* "Series 03: why the KV cache eats memory ..." section 1.2: bytes per token
  = 2 (K and V) x layers x KV heads x head_dim x bytes per element.
* "KV cache capacity planning ..." section 1: the same product times the
  number of cached tokens; section 2: a budget calculator that rejects
  non-positive shapes and keeps a safety margin of the budget.
* "KV Cache: principle and memory share (kp-013)" section 公式与模型:
  Bytes = 2 x L x H_kv x d_head x N_ctx x B_batch x B_dtype.
* "Series 03 ..." section 4.2: a GiB budget divided by bytes per token gives a
  token capacity (truncated to an integer).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

GIB = 1024 ** 3


def per_token_kv_bytes(layers: int, kv_heads: int, head_dim: int,
                       bytes_per_element: float) -> float:
    """Bytes one token occupies across all layers: 2 * L * H_kv * d * bytes."""
    return 2 * layers * kv_heads * head_dim * bytes_per_element


def kv_cache_bytes(layers: int, kv_heads: int, head_dim: int,
                   bytes_per_element: float, n_ctx: int, batch: int = 1) -> float:
    """kp-013 formula: per-token bytes times context length times batch."""
    return per_token_kv_bytes(layers, kv_heads, head_dim, bytes_per_element) * n_ctx * batch


@dataclass(frozen=True)
class KVShape:
    """Model shape the budget depends on; every field must be positive
    ("KV cache capacity planning ..." section 2 rejects a non-positive field
    with ValueError)."""

    layers: int
    kv_heads: int
    head_dim: int
    bytes_per_element: float

    def __post_init__(self) -> None:
        for name in ("layers", "kv_heads", "head_dim", "bytes_per_element"):
            if not getattr(self, name) > 0:
                raise ValueError(f"KVShape.{name} must be > 0")


def kv_bytes(shape: KVShape, tokens: int, sequences: int = 1) -> int:
    """Bytes for ``sequences`` sequences of ``tokens`` cached tokens each.
    Negative counts are rejected with ValueError (same section)."""
    if tokens < 0 or sequences < 0:
        raise ValueError("token and sequence counts must be >= 0")
    per_tok = per_token_kv_bytes(shape.layers, shape.kv_heads, shape.head_dim,
                                 shape.bytes_per_element)
    return int(per_tok * tokens * sequences)


def max_sequences(budget_gib: float, shape: KVShape, tokens_per_sequence: int,
                  safety_ratio: float = 0.85) -> int:
    """How many equal-length sequences fit into ``budget_gib`` GiB once only
    ``safety_ratio`` of it is counted as usable (same section).  The budget
    must be positive and the ratio strictly between 0 and 1."""
    if not budget_gib > 0 or not (0 < safety_ratio < 1):
        raise ValueError("budget must be > 0 and 0 < safety_ratio < 1")
    usable = budget_gib * GIB * safety_ratio
    per_seq = kv_bytes(shape, tokens_per_sequence)
    return math.floor(usable / per_seq)


def budget_tokens(budget_gib: float, bytes_per_token: float) -> int:
    """Token capacity of a GiB budget ("Series 03 ..." section 4.2)."""
    return int(budget_gib * GIB / bytes_per_token)
