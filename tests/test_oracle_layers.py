"""Pins of the model-wide (layer-major) cache layout of "What a KV cache is
..." section 2.2: (num_blocks, num_layers, num_kv_heads, block_size,
head_dim)."""
import numpy as np

from oracle import attention as oa
from oracle import kv_bytes as kb


def test_layer_view_is_each_layers_cache():
    rng = np.random.default_rng(0)
    per_layer = [rng.normal(size=(6, 2, 16, 8)) for _ in range(3)]
    model = np.stack(per_layer, axis=1)                       # [NB, L, H, 16, d]
    for l, c in enumerate(per_layer):
        assert np.array_equal(oa.layer_view(model, l), c)
    # attention through a layer view equals attention on that layer's own cache
    q = rng.normal(size=(2, 4, 8))
    tables, lens = [[3, 1], [0, 5]], [20, 31]
    for l, c in enumerate(per_layer):
        a = oa.paged_decode_attention(q, oa.layer_view(model, l), oa.layer_view(model, l), tables, lens, 0.3)
        assert np.array_equal(a, oa.paged_decode_attention(q, c, c, tables, lens, 0.3))


def test_bytes_per_token_of_the_layout_match_the_closed_form():
    # one token of every layer: a block of the model-wide cache over 16 tokens,
    # K and V, equals 16 x the closed-form per-token bytes 2 L H_kv d bytes
    # (524,288 B for 32 layers x 32 heads x 128 in fp16)
    n_layers, h_kv, d = 32, 32, 128
    block = np.zeros((1, n_layers, h_kv, 16, d), dtype=np.float16)
    per_token = 2 * block.nbytes // 16
    assert per_token == kb.per_token_kv_bytes(n_layers, h_kv, d, 2) == 524288
