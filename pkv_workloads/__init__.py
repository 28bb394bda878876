"""Seeded synthetic inputs for paged decode attention.

This module is shared by the oracle-side tests and the CUDA-side tests and
bench; it holds none of the method's arithmetic (no slot mapping, no append,
no attention, no FP8 encoding).  It only draws random numbers and lays them
out: query vectors, the K/V pool contents, the new tokens' K/V rows, context
lengths and block tables.  Values are drawn with numpy's PCG64 from a seed.

Workloads (shapes from the pages' models: Llama-2-7B-like 32 x 32 x 128 MHA,
Llama-3-8B-like 32 query / 8 KV heads with head_dim 128; the length mix of the
last one follows the 90 % short / 10 % long bucket example of the capacity
planning article):

  tiny        batch 4, 4 query = 4 KV heads, d 64, fp16, context U{1..256},
              pool 128 blocks, tables from one random permutation of the pool.
  mha7b       batch 16, 32 = 32 heads, d 128, fp16, every context 4096,
              pool 4096 blocks, tables = a random permutation cut in 16 rows.
  gqa8b       batch 64, 32 query / 8 KV heads, d 128, bf16, context
              log-uniform in [128, 8192], pool = needed blocks + 10 % free.
  prefix      gqa8b shape, batch 16: one 2048-token prefix (128 shared physical
              blocks) referenced by every table, then a private suffix
              U{16..512}.
  fp8long     32 query / 8 KV heads, d 128, q bf16, KV stored as E4M3 with
              per-KV-head scales; batch 32: 29 contexts of 2048 and 3 of 65536
              (positions drawn from the seed); partitions of 512 tokens.

Model-wide cache inputs (``layers_inputs``, ``make_layers``): random pools of
shape [num_blocks, num_layers, H_kv, 16, d] and per-layer queries / new rows
over one workload's tables.

Prefill inputs (``prefill_inputs``, ``make_prefill``): sequences with a
cached prefix and new tokens after it, random queries and pool, tables from a
random permutation of the pool.

Copy-on-write inputs (``beam_inputs``, ``make_beam``, ``copy_pairs``): random
pools, queries and new rows for a beam search over shared prompts, and random
disjoint block pairs for block copies; the tables and copies themselves come
from the block pool under test.

Conventions of every workload:
  * ``context_lens[b]`` counts the tokens attended AFTER the step's append; the
    pool already holds positions 0..ctx-2 and the step appends position ctx-1
    (its rows are ``k_new[b]`` / ``v_new[b]``).
  * The whole pool, including slots no table uses and slots past a sequence's
    end, holds N(0, 1) data, so a kernel that reads past the end is caught.
  * 16-bit data is stored as uint16 bit patterns (fp16 or bf16, rounded to
    nearest-even from float32 draws).
  * For an FP8 cache ("e4m3" or "e5m2") the pool and new rows hold the 16-bit
    data before quantisation and ``k_scale``/``v_scale`` are per-KV-head
    calibration scales: absmax over that head's data divided by the format's
    largest finite value (448 for E4M3, 57344 for E5M2), i.e. the
    absmax-calibrated per-head scale the FP8 roll-out advice asks for; they are
    inputs of the method, not part of it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16

CONFIG_NAMES = ("tiny", "mha7b", "gqa8b", "prefix", "fp8long")

# largest finite value of each FP8 storage format (the calibration divisor)
FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}
CONFIG_SEEDS = {name: 1000 + i for i, name in enumerate(CONFIG_NAMES)}


@dataclass
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str                  # q / out / new-row dtype: "f16" | "bf16"
    kv_dtype: str               # cache dtype: "f16" | "bf16" | "e4m3" | "e5m2"
    scale: float                # softmax scale 1/sqrt(head_dim)
    num_blocks: int
    context_lens: np.ndarray    # int32 [B]
    block_tables: np.ndarray    # int32 [B, max_blocks_per_seq], -1 padded
    q: np.ndarray               # uint16 [B, Hq, d]
    k_pool: np.ndarray          # uint16 [NB, Hkv, bs, d]  (pre-quantisation for FP8)
    v_pool: np.ndarray
    k_new: np.ndarray           # uint16 [B, Hkv, d]
    v_new: np.ndarray
    k_scale: np.ndarray | None = None   # float32 [Hkv] (FP8 only)
    v_scale: np.ndarray | None = None
    partition_tokens: int = 0   # 0 = let the planner choose
    block_size: int = BLOCK_SIZE
    meta: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def fp8(self) -> bool:
        return self.kv_dtype in FP8_MAX

    @property
    def kv_elt_bytes(self) -> int:
        return 1 if self.fp8 else 2

    @property
    def q_elt_bytes(self) -> int:
        return 2

    def algorithmic_bytes(self) -> int:
        """KV bytes read (every attended token, every KV head, K and V) plus
        q read plus out written.  Block tables and lengths are excluded."""
        kv = int(self.context_lens.astype(np.int64).sum()) * self.n_kv_heads * self.head_dim \
            * 2 * self.kv_elt_bytes
        qo = 2 * self.batch * self.n_q_heads * self.head_dim * self.q_elt_bytes
        return kv + qo


# ----------------------------------------------------------------------------
# random draws
# ----------------------------------------------------------------------------
def f32_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 draws to fp16 / bf16 (nearest-even) and return the bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32)
        rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        return rounded.astype(np.uint16)
    raise ValueError(dtype)


def _normal_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0, 1) draws rounded to ``dtype``, generated in chunks of the flat
    array so that no full-size float32 temporary is needed."""
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    chunk = 1 << 22
    buf = np.empty(chunk, dtype=np.float32)
    for s in range(0, flat.size, chunk):
        n = min(chunk, flat.size - s)
        rng.standard_normal(out=buf[:n], dtype=np.float32)
        flat[s:s + n] = f32_to_bits(buf[:n], dtype)
    return out


def _bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _absmax_over_head(pool_bits: np.ndarray, new_bits: np.ndarray, dtype: str) -> np.ndarray:
    """Per-KV-head absmax of the data (pool [NB, H, bs, d] and new rows
    [B, H, d]), computed one head at a time to bound memory."""
    n_heads = pool_bits.shape[1]
    out = np.empty(n_heads, dtype=np.float32)
    for g in range(n_heads):
        a = np.abs(_bits_to_f32(np.ascontiguousarray(pool_bits[:, g]), dtype)).max()
        b = np.abs(_bits_to_f32(np.ascontiguousarray(new_bits[:, g]), dtype)).max()
        out[g] = max(a, b)
    return out


def _tables_from_ids(ids: np.ndarray, blocks_per_seq, max_blocks: int) -> np.ndarray:
    tables = np.full((len(blocks_per_seq), max(1, max_blocks)), -1, dtype=np.int32)
    pos = 0
    for b, nb in enumerate(blocks_per_seq):
        tables[b, :nb] = ids[pos:pos + nb]
        pos += nb
    return tables


def _nblocks(n: int) -> int:
    return -(-int(n) // BLOCK_SIZE)


# ----------------------------------------------------------------------------
# generic builder
# ----------------------------------------------------------------------------
def build(name: str, *, batch: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
          dtype: str, kv_dtype: str, context_lens, seed: int,
          num_blocks: int | None = None, free_fraction: float = 0.10,
          shared_prefix_blocks: int = 0, partition_tokens: int = 0,
          scale: float | None = None) -> Workload:
    """Lay out a workload: contexts as given, physical ids drawn as one random
    permutation of the pool (disjoint between sequences, except for the
    ``shared_prefix_blocks`` blocks that every table starts with)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    ctx = np.asarray(context_lens, dtype=np.int32)
    if shared_prefix_blocks:
        private = [max(0, _nblocks(c) - shared_prefix_blocks) for c in ctx]
        needed = shared_prefix_blocks + sum(private)
    else:
        private = [_nblocks(c) for c in ctx]
        needed = sum(private)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(needed * (1.0 + free_fraction)))
    if needed > num_blocks:
        raise ValueError("pool too small for the contexts")
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = max([_nblocks(c) for c in ctx] + [1])
    if shared_prefix_blocks:
        prefix_ids = perm[:shared_prefix_blocks]
        rest = perm[shared_prefix_blocks:]
        tables = np.full((batch, max_blocks), -1, dtype=np.int32)
        pos = 0
        for b in range(batch):
            tables[b, :shared_prefix_blocks] = prefix_ids
            nb = private[b]
            tables[b, shared_prefix_blocks:shared_prefix_blocks + nb] = rest[pos:pos + nb]
            pos += nb
    else:
        tables = _tables_from_ids(perm, private, max_blocks)

    raw_dtype = dtype if kv_dtype in FP8_MAX else kv_dtype
    q = _normal_bits(rng, (batch, n_q_heads, head_dim), dtype)
    k_pool = _normal_bits(rng, (num_blocks, n_kv_heads, BLOCK_SIZE, head_dim), raw_dtype)
    v_pool = _normal_bits(rng, (num_blocks, n_kv_heads, BLOCK_SIZE, head_dim), raw_dtype)
    k_new = _normal_bits(rng, (batch, n_kv_heads, head_dim), raw_dtype)
    v_new = _normal_bits(rng, (batch, n_kv_heads, head_dim), raw_dtype)
    k_scale = v_scale = None
    if kv_dtype in FP8_MAX:
        top = np.float32(FP8_MAX[kv_dtype])
        k_scale = (_absmax_over_head(k_pool, k_new, raw_dtype) / top).astype(np.float32)
        v_scale = (_absmax_over_head(v_pool, v_new, raw_dtype) / top).astype(np.float32)
    return Workload(
        name=name, batch=batch, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads,
        head_dim=head_dim, dtype=dtype, kv_dtype=kv_dtype,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(head_dim)),
        num_blocks=int(num_blocks), context_lens=ctx, block_tables=tables, q=q,
        k_pool=k_pool, v_pool=v_pool, k_new=k_new, v_new=v_new,
        k_scale=k_scale, v_scale=v_scale, partition_tokens=partition_tokens,
        meta={"seed": seed, "shared_prefix_blocks": shared_prefix_blocks})


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------
def make(name: str, seed: int | None = None, fp8: str = "e4m3") -> Workload:
    """The named workload; ``fp8`` picks the storage format of fp8long's cache
    ("e4m3", the configuration's own, or "e5m2"), with the same data."""
    seed = CONFIG_SEEDS[name] if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed + 7919))   # length draws
    if name == "tiny":
        ctx = rng.integers(1, 256, size=4, endpoint=True)
        return build(name, batch=4, n_q_heads=4, n_kv_heads=4, head_dim=64, dtype="f16",
                     kv_dtype="f16", context_lens=ctx, seed=seed, num_blocks=128)
    if name == "mha7b":
        return build(name, batch=16, n_q_heads=32, n_kv_heads=32, head_dim=128, dtype="f16",
                     kv_dtype="f16", context_lens=[4096] * 16, seed=seed, num_blocks=4096)
    if name == "gqa8b":
        u = rng.uniform(math.log(128), math.log(8192), size=64)
        ctx = np.clip(np.floor(np.exp(u)), 128, 8192).astype(np.int32)
        return build(name, batch=64, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
                     kv_dtype="bf16", context_lens=ctx, seed=seed)
    if name == "prefix":
        suffix = rng.integers(16, 512, size=16, endpoint=True)
        ctx = 2048 + suffix
        return build(name, batch=16, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
                     kv_dtype="bf16", context_lens=ctx, seed=seed, shared_prefix_blocks=128)
    if name == "fp8long":
        ctx = np.full(32, 2048, dtype=np.int32)
        ctx[rng.choice(32, size=3, replace=False)] = 65536
        if fp8 not in FP8_MAX:
            raise KeyError(fp8)
        return build(name if fp8 == "e4m3" else f"{name}_{fp8}", batch=32, n_q_heads=32, n_kv_heads=8,
                     head_dim=128, dtype="bf16", kv_dtype=fp8, context_lens=ctx, seed=seed, partition_tokens=512)
    raise KeyError(name)


# ----------------------------------------------------------------------------
# copy-on-write inputs
# ----------------------------------------------------------------------------
@dataclass
class BeamInputs:
    """Random data for one decode step of a beam search over shared prompts.

    ``n_prompts`` prompts of ``prompt_lens[p]`` tokens; each is followed by
    ``beams`` branches that share its blocks, and sequence b = p * beams + j
    is branch j of prompt p.  Every branch appends one token at position
    prompt_lens[p] in this step (its context after the append is
    prompt_lens[p] + 1).  The block tables are NOT laid out here: the caller's
    block pool takes the prompt blocks (prompt 0 first) and the branches share
    them, so the tables and the copies follow from the pool under test."""
    name: str
    n_prompts: int
    beams: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str
    scale: float
    num_blocks: int
    prompt_lens: np.ndarray        # [n_prompts] int32
    q: np.ndarray                  # [B, Hq, d] 16-bit bits, B = n_prompts * beams
    k_pool: np.ndarray             # [NB, Hkv, 16, d] 16-bit bits (every block random)
    v_pool: np.ndarray
    k_new: np.ndarray              # [B, Hkv, d]
    v_new: np.ndarray
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return self.n_prompts * self.beams


def beam_inputs(name: str, *, n_prompts: int, beams: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                dtype: str, prompt_lens, seed: int, spare_blocks: int | None = None) -> BeamInputs:
    """Pool = the prompts' blocks + ``spare_blocks`` (default: two per branch)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(prompt_lens, dtype=np.int32)
    batch = n_prompts * beams
    spare = 2 * batch if spare_blocks is None else spare_blocks
    num_blocks = int(sum(_nblocks(n) for n in lens) + spare)
    return BeamInputs(
        name=name, n_prompts=n_prompts, beams=beams, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads,
        head_dim=head_dim, dtype=dtype, scale=1.0 / math.sqrt(head_dim), num_blocks=num_blocks,
        prompt_lens=lens,
        q=_normal_bits(rng, (batch, n_q_heads, head_dim), dtype),
        k_pool=_normal_bits(rng, (num_blocks, n_kv_heads, BLOCK_SIZE, head_dim), dtype),
        v_pool=_normal_bits(rng, (num_blocks, n_kv_heads, BLOCK_SIZE, head_dim), dtype),
        k_new=_normal_bits(rng, (batch, n_kv_heads, head_dim), dtype),
        v_new=_normal_bits(rng, (batch, n_kv_heads, head_dim), dtype),
        meta={"seed": seed})


def make_beam(seed: int = 1100) -> BeamInputs:
    """8 prompts x 8 branches (64 sequences), Llama-3-8B-like heads (32 query /
    8 KV, d 128, bf16), prompt lengths U{1000..3000}."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    lens = rng.integers(1000, 3000, size=8, endpoint=True)
    return beam_inputs("beam", n_prompts=8, beams=8, n_q_heads=32, n_kv_heads=8, head_dim=128, dtype="bf16",
                       prompt_lens=lens, seed=seed)


def copy_pairs(num_blocks: int, n_pairs: int, seed: int):
    """``n_pairs`` (src, dst) block pairs with distinct sources, distinct
    destinations and no destination among the sources, drawn as one random
    permutation of the pool (int32 arrays)."""
    if 2 * n_pairs > num_blocks:
        raise ValueError("the pool holds fewer than 2 * n_pairs blocks")
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(num_blocks).astype(np.int32)
    return perm[:n_pairs].copy(), perm[n_pairs:2 * n_pairs].copy()


# ----------------------------------------------------------------------------
# prefill / extend inputs
# ----------------------------------------------------------------------------
@dataclass
class PrefillInputs:
    """Random data for one prefill (extend) call: sequence b has
    ``cached_lens[b]`` tokens already in the cache and ``new_lens[b]`` new
    tokens after them (their K/V rows are already in the pool too, as after
    the append); q holds the new tokens' queries, packed by cu_seqlens."""
    name: str
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    dtype: str
    scale: float
    num_blocks: int
    cached_lens: np.ndarray        # [B] int32
    new_lens: np.ndarray           # [B] int32
    context_lens: np.ndarray       # [B] int32 = cached + new
    cu_seqlens: np.ndarray         # [B + 1] int32
    block_tables: np.ndarray       # [B, max_blocks] int32, -1 padded
    q: np.ndarray                  # [T, Hq, d] 16-bit bits
    k_pool: np.ndarray             # [NB, Hkv, 16, d] 16-bit bits
    v_pool: np.ndarray
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.new_lens)

    @property
    def max_blocks_per_seq(self) -> int:
        return self.block_tables.shape[1]

    def flops(self) -> int:
        """Causal extend attention: 4 d flops per (query token, query head,
        attended key) -- 2 d for q.K, 2 d for p.V."""
        n = 0
        for c, m in zip(self.cached_lens, self.new_lens):
            c, m = int(c), int(m)
            n += m * c + m * (m + 1) // 2          # sum over new tokens of (position + 1)
        return 4 * self.head_dim * self.n_q_heads * n


def prefill_inputs(name: str, *, cached_lens, new_lens, n_q_heads: int, n_kv_heads: int, head_dim: int,
                   dtype: str, seed: int, free_fraction: float = 0.05) -> PrefillInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    cached = np.asarray(cached_lens, dtype=np.int32)
    new = np.asarray(new_lens, dtype=np.int32)
    ctx = cached + new
    blocks = [_nblocks(c) for c in ctx]
    num_blocks = max(1, math.ceil(sum(blocks) * (1.0 + free_fraction)))
    perm = rng.permutation(num_blocks).astype(np.int32)
    tables = _tables_from_ids(perm, blocks, max(blocks + [1]))
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    return PrefillInputs(
        name=name, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim=head_dim, dtype=dtype,
        scale=1.0 / math.sqrt(head_dim), num_blocks=int(num_blocks), cached_lens=cached, new_lens=new,
        context_lens=ctx.astype(np.int32), cu_seqlens=cu, block_tables=tables,
        q=_normal_bits(rng, (int(cu[-1]), n_q_heads, head_dim), dtype),
        k_pool=_normal_bits(rng, (num_blocks, n_kv_heads, BLOCK_SIZE, head_dim), dtype),
        v_pool=_normal_bits(rng, (num_blocks, n_kv_heads, BLOCK_SIZE, head_dim), dtype),
        meta={"seed": seed})


def make_prefill(seed: int = 1300) -> PrefillInputs:
    """Chunked prefill of 4 sequences: 2048 tokens cached, 2048 new tokens
    each; Llama-3-8B-like heads (32 query / 8 KV, d 128, bf16)."""
    return prefill_inputs("prefill", cached_lens=[2048] * 4, new_lens=[2048] * 4, n_q_heads=32, n_kv_heads=8,
                          head_dim=128, dtype="bf16", seed=seed)


# ----------------------------------------------------------------------------
# model-wide (layer-major) cache inputs
# ----------------------------------------------------------------------------
@dataclass
class LayerInputs:
    """One decode step of an ``n_layers``-layer model over a cache laid out
    [num_blocks, n_layers, H_kv, 16, d]: ``base`` carries the shapes, tables,
    lengths and scale shared by all layers; every layer has its own pool
    slice, queries and new rows."""
    base: Workload
    n_layers: int
    k_pool: np.ndarray             # [NB, L, Hkv, 16, d] 16-bit bits
    v_pool: np.ndarray
    q: np.ndarray                  # [L, B, Hq, d]
    k_new: np.ndarray              # [L, B, Hkv, d]
    v_new: np.ndarray


def layers_inputs(base: Workload, n_layers: int, seed: int) -> LayerInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    w = base
    nb, L = w.num_blocks, n_layers
    return LayerInputs(
        base=w, n_layers=L,
        k_pool=_normal_bits(rng, (nb, L, w.n_kv_heads, BLOCK_SIZE, w.head_dim), w.kv_dtype),
        v_pool=_normal_bits(rng, (nb, L, w.n_kv_heads, BLOCK_SIZE, w.head_dim), w.kv_dtype),
        q=_normal_bits(rng, (L, w.batch, w.n_q_heads, w.head_dim), w.dtype),
        k_new=_normal_bits(rng, (L, w.batch, w.n_kv_heads, w.head_dim), w.kv_dtype),
        v_new=_normal_bits(rng, (L, w.batch, w.n_kv_heads, w.head_dim), w.kv_dtype))


def make_layers(seed: int = 1400) -> LayerInputs:
    """The tiny workload's shape (batch 4, 4 = 4 heads, d 64, fp16, contexts
    U{1..256}) through 32 layers: a step whose calls are launch-bound."""
    return layers_inputs(make("tiny"), 32, seed)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    """float32 view of stored 16-bit data (for host-side plumbing only)."""
    return _bits_to_f32(np.asarray(bits, dtype=np.uint16), dtype)
