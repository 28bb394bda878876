"""Pins of oracle.kv_bytes against the byte counts the pages print."""
import json
import os

import pytest

from oracle import kv_bytes as kb
from tests.conftest import GOLDEN

with open(os.path.join(GOLDEN, "kv_bytes_examples.json")) as f:
    EX = json.load(f)


@pytest.mark.parametrize("e", EX["per_token"], ids=lambda e: e["cite"][:40])
def test_per_token_bytes(e):
    got = kb.per_token_kv_bytes(e["layers"], e["kv_heads"], e["head_dim"], e["bytes_per_element"])
    assert got == e["bytes"]


@pytest.mark.parametrize("e", EX["totals"], ids=lambda e: e["cite"][:40])
def test_total_bytes(e):
    shape = kb.KVShape(e["layers"], e["kv_heads"], e["head_dim"], e["bytes_per_element"])
    assert kb.kv_bytes(shape, e["tokens"], e["sequences"]) == e["bytes"]
    assert kb.kv_cache_bytes(e["layers"], e["kv_heads"], e["head_dim"], e["bytes_per_element"],
                             e["tokens"], e["sequences"]) == e["bytes"]


@pytest.mark.parametrize("e", EX["budget"], ids=lambda e: e["cite"][:40])
def test_budget_example(e):
    tokens = kb.budget_tokens(e["budget_gib"], e["bytes_per_token"])
    assert tokens == e["tokens"]
    assert tokens // e["tokens_per_request"] == e["requests"]


@pytest.mark.parametrize("e", EX["layout"], ids=lambda e: e["cite"][:40])
def test_block_buffer_bytes(e):
    # one K block over all layers of the "(num_blocks, num_layers, kv_heads, bs, d)" layout
    per_token_k = kb.per_token_kv_bytes(e["layers"], e["kv_heads"], e["head_dim"],
                                        e["bytes_per_element"]) / 2
    assert per_token_k * e["block_size"] == e["k_bytes_per_block"]
    assert round(e["k_bytes_per_block"] / 1e6, 1) == 4.2


def test_kp013_rounded_figures():
    # kp-013 公式与模型: a 4096-token request is about 2.1 GB and GQA with 8 KV
    # heads takes 0.125 MB per token
    per_tok = kb.per_token_kv_bytes(32, 32, 128, 2)
    assert round(per_tok * 4096 / 1e9, 1) == 2.1
    assert kb.per_token_kv_bytes(32, 8, 128, 2) / 2 ** 20 == 0.125


def test_calculator_rejects_bad_input():
    # "KV cache capacity planning" section 2: non-positive shape fields and
    # negative counts are ValueErrors; the tiny shape fits at least one sequence
    tiny = kb.KVShape(2, 2, 4, 2)
    assert kb.max_sequences(1, tiny, 10) > 0
    for bad in [(0, 2, 4, 2), (2, 0, 4, 2), (2, 2, -4, 2), (2, 2, 4, 0)]:
        with pytest.raises(ValueError):
            kb.KVShape(*bad)
    with pytest.raises(ValueError):
        kb.kv_bytes(tiny, -1)
    with pytest.raises(ValueError):
        kb.kv_bytes(tiny, 1, -1)
    with pytest.raises(ValueError):
        kb.max_sequences(0, tiny, 10)
    with pytest.raises(ValueError):
        kb.max_sequences(1, tiny, 10, safety_ratio=1.0)


def test_fp8_halves_the_bytes():
    # "KV cache capacity planning" section 2: one byte per element for FP8
    assert kb.per_token_kv_bytes(32, 8, 128, 1) * 2 == kb.per_token_kv_bytes(32, 8, 128, 2)
