"""Helpers for the GPU parity tests: move a seeded workload to the device,
run the CUDA path through the C ABI, and build the oracle's expectation.

Nothing here computes the method on the GPU side except through libpkv.so;
the expectations come only from ``oracle``.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import pkv_workloads as wl
from oracle import attention as oa
from oracle import e4m3 as oe
from oracle import e5m2 as o5
from oracle import numerics as on
from oracle import slots as osl

ATOL, RTOL = 2e-3, 1e-2          # fp16 / bf16 attention: |gpu - ref| <= ATOL + RTOL |ref|
FP8_ATOL = 2e-2                  # FP8 attention: |gpu - ref| <= FP8_ATOL (same codes on both sides)

FP8_ORACLE = {"e4m3": oe, "e5m2": o5}   # the oracle module of each FP8 storage format

TORCH_16 = {"f16": torch.float16, "bf16": torch.bfloat16}


def dev():
    return torch.device("cuda:0")


def bits_to_torch(bits: np.ndarray, dtype: str, device=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits)).view(TORCH_16[dtype])
    return t.to(device or dev())


def torch_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.uint16).numpy() if t.dtype != torch.uint8 else t.cpu().numpy()


class GpuCase:
    """Device copies of a workload plus the buffers one decode step needs."""

    def __init__(self, w: wl.Workload, *, codes=None, max_context_len=None):
        d = dev()
        self.w = w
        self.fp8 = w.fp8
        self.fmt = w.kv_dtype
        if self.fp8:
            kc, vc = codes
            self.k_cache = torch.from_numpy(kc).to(d)
            self.v_cache = torch.from_numpy(vc).to(d)
            self.k_scale = torch.from_numpy(w.k_scale).to(d)
            self.v_scale = torch.from_numpy(w.v_scale).to(d)
        else:
            self.k_cache = bits_to_torch(w.k_pool, w.kv_dtype)
            self.v_cache = bits_to_torch(w.v_pool, w.kv_dtype)
        self.q = bits_to_torch(w.q, w.dtype)
        self.k_new = bits_to_torch(w.k_new, w.dtype if self.fp8 else w.kv_dtype)
        self.v_new = bits_to_torch(w.v_new, w.dtype if self.fp8 else w.kv_dtype)
        self.tables = torch.from_numpy(w.block_tables).to(d)
        self.lens = torch.from_numpy(w.context_lens).to(d)
        self.slots = torch.empty(w.batch, dtype=torch.int64, device=d)
        self.out = torch.empty_like(self.q)
        self.err = torch.zeros(1, dtype=torch.int32, device=d)
        self.max_ctx = int(max_context_len if max_context_len is not None else max(1, w.context_lens.max()))
        self.ws = None

    def workspace(self, partition_tokens):
        import paged_kv_cache_153_gb300 as pkv
        w = self.w
        n = pkv.pkv_decode_workspace_bytes(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                           w.max_blocks_per_seq, self.max_ctx, partition_tokens)
        if self.ws is None or self.ws.numel() < n:
            self.ws = torch.empty(n, dtype=torch.uint8, device=dev())
        return self.ws

    def step(self, partition_tokens=None, append=True, stream=None):
        """slot mapping + append + decode attention, all through the C ABI."""
        import paged_kv_cache_153_gb300 as pkv
        w = self.w
        pt = w.partition_tokens if partition_tokens is None else partition_tokens
        ws = self.workspace(pt)
        if append:
            pkv.pkv_slot_mapping(self.tables, self.lens, self.slots, num_blocks=w.num_blocks,
                                 position_offset=-1, err_flag=self.err, stream=stream)
            if self.fp8:
                append = pkv.pkv_kv_append_fp8 if self.fmt == "e4m3" else pkv.pkv_kv_append_e5m2
                append(self.k_new, self.v_new, self.slots, self.k_cache, self.v_cache, self.k_scale, self.v_scale,
                       err_flag=self.err, stream=stream)
            else:
                pkv.pkv_kv_append(self.k_new, self.v_new, self.slots, self.k_cache, self.v_cache,
                                  err_flag=self.err, stream=stream)
        if self.fp8:
            attend = pkv.pkv_paged_decode_attention_fp8 if self.fmt == "e4m3" else pkv.pkv_paged_decode_attention_e5m2
            attend(self.q, self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.tables, self.lens, self.out,
                   scale=w.scale, max_context_len=self.max_ctx, workspace=ws, partition_tokens=pt,
                   err_flag=self.err, stream=stream)
        else:
            pkv.pkv_paged_decode_attention(self.q, self.k_cache, self.v_cache, self.tables, self.lens,
                                           self.out, scale=w.scale, max_context_len=self.max_ctx,
                                           workspace=ws, partition_tokens=pt, err_flag=self.err,
                                           stream=stream)
        return self.out

    def fused_step(self, partition_tokens=None, stream=None):
        """The call the benchmark times: pkv_paged_decode_step[_fp8] (slot
        mapping, append and attention in the decode launch, then the combine)."""
        import paged_kv_cache_153_gb300 as pkv
        w = self.w
        pt = w.partition_tokens if partition_tokens is None else partition_tokens
        ws = self.workspace(pt)
        if self.fp8:
            fused = pkv.pkv_paged_decode_step_fp8 if self.fmt == "e4m3" else pkv.pkv_paged_decode_step_e5m2
            fused(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.tables,
                  self.lens, self.out, scale=w.scale, max_context_len=self.max_ctx, workspace=ws, partition_tokens=pt,
                  slot_mapping_out=self.slots, err_flag=self.err, stream=stream)
        else:
            pkv.pkv_paged_decode_step(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache, self.tables,
                                      self.lens, self.out, scale=w.scale, max_context_len=self.max_ctx,
                                      workspace=ws, partition_tokens=pt, slot_mapping_out=self.slots,
                                      err_flag=self.err, stream=stream)
        return self.out

    def err_code(self) -> int:
        torch.cuda.synchronize()
        return int(self.err.item())


# ---------------------------------------------------------------------------
# oracle side
# ---------------------------------------------------------------------------
def oracle_slots(w: wl.Workload) -> np.ndarray:
    return osl.slot_mapping(w.block_tables, range(w.batch), w.context_lens.astype(np.int64) - 1)


def oracle_pools_after_append(w: wl.Workload):
    """Bit patterns (16-bit) or E4M3 codes of the pools after the step's append."""
    slots = oracle_slots(w)
    if w.fp8:
        kc, vc, kn, vn = oracle_fp8_codes(w)
        osl.append_rows(kc, kn, slots)
        osl.append_rows(vc, vn, slots)
        return kc, vc
    kp, vp = w.k_pool.copy(), w.v_pool.copy()
    osl.append_rows(kp, w.k_new, slots)
    osl.append_rows(vp, w.v_new, slots)
    return kp, vp


def oracle_fp8_codes(w: wl.Workload):
    """Oracle FP8 codes (the workload's format) of the whole pool (before the
    append) and of the new rows, per KV head with that head's scale."""
    enc = FP8_ORACLE[w.kv_dtype].encode
    kc = np.empty(w.k_pool.shape, dtype=np.uint8)
    vc = np.empty(w.v_pool.shape, dtype=np.uint8)
    kn = np.empty(w.k_new.shape, dtype=np.uint8)
    vn = np.empty(w.v_new.shape, dtype=np.uint8)
    for g in range(w.n_kv_heads):
        kc[:, g] = enc(wl.bits_to_f32(w.k_pool[:, g], w.dtype), w.k_scale[g])
        vc[:, g] = enc(wl.bits_to_f32(w.v_pool[:, g], w.dtype), w.v_scale[g])
        kn[:, g] = enc(wl.bits_to_f32(w.k_new[:, g], w.dtype), w.k_scale[g])
        vn[:, g] = enc(wl.bits_to_f32(w.v_new[:, g], w.dtype), w.v_scale[g])
    return kc, vc, kn, vn


def fp8_codes_by_table(bits: np.ndarray, dtype: str, scale, fmt: str = "e4m3") -> np.ndarray:
    """The oracle's FP8 codes (format ``fmt``) of 16-bit data ``bits`` with one
    scale: the oracle's encoder is applied to every one of the 65,536 bit
    patterns once and the data are looked up in that table (the code of a
    value depends only on its bits and the scale)."""
    with np.errstate(over="ignore", invalid="ignore"):
        table = FP8_ORACLE[fmt].encode(wl.bits_to_f32(np.arange(1 << 16, dtype=np.uint16), dtype), scale)
    return table[np.asarray(bits, dtype=np.uint16)]


def oracle_fp8_pool_codes(w: wl.Workload, pool: np.ndarray, scales) -> np.ndarray:
    """Oracle FP8 codes (the workload's format) of a whole pool [NB, H, 16, d]
    (or rows [T, H, d]), per KV head with that head's scale, through the
    per-head code table."""
    out = np.empty(pool.shape, dtype=np.uint8)
    for g in range(w.n_kv_heads):
        out[:, g] = fp8_codes_by_table(pool[:, g], w.dtype, scales[g], w.kv_dtype)
    return out


def oracle_decode_all(w: wl.Workload, kp, vp, seqs=None):
    """float64 expectation [B, Hq, d] (rows of sequences not in ``seqs`` are
    NaN), gathering each (sequence, KV head) once."""
    q = on.bits_to_f64(w.q, w.dtype)
    group = w.n_q_heads // w.n_kv_heads
    ref = np.full((w.batch, w.n_q_heads, w.head_dim), np.nan)
    for b in (range(w.batch) if seqs is None else seqs):
        n = int(w.context_lens[b])
        for g in range(w.n_kv_heads):
            kb = oa.gather_sequence(kp, w.block_tables[b], n, g)
            vb = oa.gather_sequence(vp, w.block_tables[b], n, g)
            if w.fp8:
                keys = FP8_ORACLE[w.kv_dtype].decode(kb) * float(w.k_scale[g])
                values = FP8_ORACLE[w.kv_dtype].decode(vb) * float(w.v_scale[g])
            else:
                keys = on.bits_to_f64(kb, w.kv_dtype)
                values = on.bits_to_f64(vb, w.kv_dtype)
            for h in range(g * group, (g + 1) * group):
                ref[b, h] = oa.attend(q[b, h], keys, values, w.scale)
    return ref


def compare_all(got: torch.Tensor, ref: np.ndarray, atol: float, rtol: float):
    """Elementwise |got - ref| <= atol + rtol |ref| over the rows of ``ref``
    that are not NaN; returns (max_abs, max_rel, n_bad, n_checked)."""
    g = got.float().cpu().numpy().astype(np.float64)
    sel = ~np.isnan(ref)
    diff = np.abs(g[sel] - ref[sel])
    lim = atol + rtol * np.abs(ref[sel])
    rel = diff / np.maximum(np.abs(ref[sel]), 1e-30)
    return float(diff.max()), float(rel.max()), int((diff > lim).sum()) + int(np.isnan(g[sel]).sum()), int(sel.sum())


def record_parity(label: str, **fields) -> None:
    """Print a parity record and append it, as one JSON line, to the file
    named by PKV_PARITY_LOG (if set)."""
    rec = {"case": label, **fields}
    print("parity", json.dumps(rec))
    path = os.environ.get("PKV_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def oracle_decode(w: wl.Workload, kp, vp, pairs=None):
    """float64 expectation for (b, h) pairs (all pairs when None); kp/vp are
    16-bit bit patterns or (for E4M3) codes of the pools after the append."""
    q = on.bits_to_f64(w.q, w.dtype)
    group = w.n_q_heads // w.n_kv_heads
    if pairs is None:
        pairs = [(b, h) for b in range(w.batch) for h in range(w.n_q_heads)]
    out = {}
    for b, h in pairs:
        g = h // group
        n = int(w.context_lens[b])
        kb = oa.gather_sequence(kp, w.block_tables[b], n, g)
        vb = oa.gather_sequence(vp, w.block_tables[b], n, g)
        if w.fp8:
            keys = FP8_ORACLE[w.kv_dtype].decode(kb) * float(w.k_scale[g])
            values = FP8_ORACLE[w.kv_dtype].decode(vb) * float(w.v_scale[g])
        else:
            keys = on.bits_to_f64(kb, w.kv_dtype)
            values = on.bits_to_f64(vb, w.kv_dtype)
        out[(b, h)] = oa.attend(q[b, h], keys, values, w.scale)
    return out


def compare(got: torch.Tensor, ref: dict, fp8: bool = False):
    """Elementwise tolerance check; returns (max_abs, max_rel, n_bad)."""
    g = got.float().cpu().numpy().astype(np.float64)
    max_abs = max_rel = 0.0
    n_bad = 0
    for (b, h), r in ref.items():
        diff = np.abs(g[b, h] - r)
        lim = FP8_ATOL if fp8 else ATOL + RTOL * np.abs(r)
        n_bad += int((diff > lim).sum())
        max_abs = max(max_abs, float(diff.max()))
        max_rel = max(max_rel, float((diff / np.maximum(np.abs(r), 1e-30)).max()))
    return max_abs, max_rel, n_bad
