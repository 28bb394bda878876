"""Benchmark of one paged decode step on GB300: slot mapping, KV append and
paged decode attention (split + combine), all through the libpkv C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mha7b]
    python bench.py --impl reference ...      # the float64 oracle on host cores

Prints one JSON line (rank 0).  The headline workload is the Llama-2-7B-shaped
MHA decode: batch 16, 32 query = 32 KV heads, head_dim 128, fp16, block 16,
every context 4096 tokens, block tables drawn as a random permutation of a
4096-block pool.  Its KV cache (1.07 GB read per step) is larger than L2, so
no flush is needed between steps.  A default run (no --workload) also times
the other large decode configurations in the same process -- the
Llama-3-8B-shaped GQA decode, the shared-prefix batch and the long-context
E4M3 mix -- and reports each under "configs" with its own roofline and CPU
baseline.  Under torchrun every rank runs its own replica of the headline
workload (no data-path collective); the timing is the maximum over ranks and
``value`` is the tokens of all ranks divided by it.

The CPU baseline is the float64 oracle on a bounded sample of each workload,
timed on every host core (a process pool forked before any CUDA call, one
sequence per task) and on one core.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

# the oracle's numpy/BLAS work is timed on one host thread
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import pkv_workloads as wl  # noqa: E402

METRIC = "decode-attn tokens/s and achieved HBM GB/s (% of GB300 roofline), 1 GPU"
UNIT = "tokens/s"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "decode_traffic.json")


_T0 = time.perf_counter()


def log(msg: str) -> None:
    """Progress on stderr (the JSON result is the only line on stdout)."""
    print(f"[bench {time.perf_counter() - _T0:7.1f}s] {msg}", file=sys.stderr, flush=True)


def describe(w: wl.Workload) -> dict:
    ctx = w.context_lens
    return {
        "workload": f"{w.name}: paged decode step, batch {w.batch}, {w.n_q_heads} query / {w.n_kv_heads} KV "
                    f"heads, head_dim {w.head_dim}, {w.kv_dtype} KV cache, block 16, contexts "
                    f"{int(ctx.min())}..{int(ctx.max())} (mean {float(ctx.mean()):.0f})",
        "batch": w.batch, "num_q_heads": w.n_q_heads, "num_kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
        "kv_dtype": w.kv_dtype, "block_size": 16, "num_blocks": w.num_blocks,
        "context_tokens_total": int(ctx.sum()), "partition_tokens": w.partition_tokens,
        "step": "pkv_paged_decode_step: slot mapping + append + paged decode attention in one decode launch, + combine",
        "l2": f"inputs larger than L2: {w.algorithmic_bytes() / 1e9:.3f} GB of KV + q + out per step, no flush",
    }


# the sources each timed kernel is built from: a committed DRAM-traffic figure
# stays valid while the code of these files (comments and layout aside) is unchanged
_COMMON_SOURCES = ("pkv_common.cuh", "host_util.h")
_DECODE_SOURCES = ("api.cu", "decode.cuh", "decode_launch.cuh", "decode_f16.cu", "decode_bf16.cu",
                   "decode_e4m3.cu", "decode_e5m2.cu", "decode_int8.cu")
KERNEL_SOURCES = {
    "decode": _COMMON_SOURCES + _DECODE_SOURCES,
    "int8": _COMMON_SOURCES + _DECODE_SOURCES + ("append.cu", "append_int8.cu"),
    "cow": _COMMON_SOURCES + ("append.cu",),
    "prefill": _COMMON_SOURCES + ("prefill.cu",),
}


def code_only(src: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed to
    one space (string and character literals kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":                       # a literal: copy up to its closing quote
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):         # a line comment
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):         # a block comment
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_digest(family: str = "decode") -> str:
    """Hash of the code (not the comments) of the sources a workload's kernels
    are built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_153_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[family]):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def source_family(workload: str) -> str:
    return workload if workload in KERNEL_SOURCES else "decode"


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def ncu_traffic(workload: str):
    """DRAM bytes per timed call from a committed ncu summary, if it was taken
    on the current source of the kernels the workload runs (else None)."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("source_digest") != kernel_source_digest(source_family(workload)):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# replicas: every rank runs its own copy of the workload; no data crosses ranks
# ---------------------------------------------------------------------------
def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's time (the job ends when its last replica ends)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest time."""
    return world * units_per_rank / seconds


# ---------------------------------------------------------------------------
# oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_step(w: wl.Workload, seqs) -> int:
    """One decode step of the float64 oracle for sequences ``seqs``: slot
    mapping, append, attention for all their query heads.  Returns tokens."""
    from oracle import attention as oa
    from oracle import e4m3, e5m2
    from oracle import numerics as on
    from oracle import slots as osl
    seqs = list(seqs)
    slots = osl.slot_mapping(w.block_tables, seqs, w.context_lens[seqs].astype(np.int64) - 1)
    fp8 = w.fp8
    oe = {"e4m3": e4m3, "e5m2": e5m2}.get(w.kv_dtype)
    osl.append_rows(w.k_pool, w.k_new[seqs], slots)
    osl.append_rows(w.v_pool, w.v_new[seqs], slots)
    q = on.bits_to_f64(w.q[seqs], w.dtype)
    group = w.n_q_heads // w.n_kv_heads
    for i, b in enumerate(seqs):
        n = int(w.context_lens[b])
        for g in range(w.n_kv_heads):
            kb = oa.gather_sequence(w.k_pool, w.block_tables[b], n, g)
            vb = oa.gather_sequence(w.v_pool, w.block_tables[b], n, g)
            if fp8:
                keys = oe.decode(oe.encode(wl.bits_to_f32(kb, w.dtype), w.k_scale[g])) * float(w.k_scale[g])
                values = oe.decode(oe.encode(wl.bits_to_f32(vb, w.dtype), w.v_scale[g])) * float(w.v_scale[g])
            else:
                keys, values = on.bits_to_f64(kb, w.kv_dtype), on.bits_to_f64(vb, w.kv_dtype)
            for h in range(g * group, (g + 1) * group):
                oa.attend(q[i, h], keys, values, w.scale)
    return len(seqs)


def oracle_sample_size(w: wl.Workload) -> int:
    return 2 if w.batch >= 2 else 1


# Host-side oracle pool.  It is forked before the first CUDA call (a process
# forked after it can hang) and reads the workloads it was forked with.
_POOL_WORKLOADS: dict = {}


def _oracle_task(name_and_seq):
    name, b = name_and_seq
    w = _POOL_WORKLOADS[name]
    t0 = time.perf_counter()
    oracle_step(w, [b])
    return time.perf_counter() - t0


def start_oracle_pool(workloads):
    """A fork pool of one worker per host core over ``workloads`` (call
    before any CUDA call).  Returns (pool, cores) or (None, 1)."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    if cores < 2:
        return None, 1
    _POOL_WORKLOADS.clear()
    _POOL_WORKLOADS.update({w.name: w for w in workloads})
    return mp.get_context("fork").Pool(cores), cores


def cpu_baseline(w: wl.Workload, budget_s: float = 12.0, pool=None, cores: int = 1) -> dict:
    """The oracle's decode step on a bounded sample of the workload: on every
    host core through ``pool`` (sequences dealt one per task, as many rounds
    as fit in the budget), and on one core."""
    one_budget = budget_s if pool is None else budget_s / 3
    n = oracle_sample_size(w)
    done, t0, i = 0, time.perf_counter(), 0
    while True:
        seqs = [(i * n + j) % w.batch for j in range(n)]
        done += oracle_step(w, seqs)
        i += 1
        el = time.perf_counter() - t0
        if el >= one_budget:
            break
    one = {"value": done / el, "unit": UNIT, "cores": 1,
           "sample": f"{done} of the workload's sequences ({n} per oracle step, all heads), float64, "
                     f"{el:.1f} s on one host thread"}
    if pool is None:
        return dict(one, kind="oracle")
    done_all, t0, rnd = 0, time.perf_counter(), 0
    while True:
        seqs = [(rnd * cores + j) % w.batch for j in range(cores)]
        pool.map(_oracle_task, [(w.name, b) for b in seqs], chunksize=1)
        done_all += len(seqs)
        rnd += 1
        el_all = time.perf_counter() - t0
        if el_all >= budget_s - one_budget:
            break
    return {"value": done_all / el_all, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{done_all} of the workload's sequences (all heads), float64, {el_all:.1f} s on {cores} "
                      f"host cores (one sequence per task, {rnd} rounds)",
            "one_core": one}


def run_reference(args, w: wl.Workload) -> dict:
    """The oracle as the reference arm: each step is one round of the oracle's
    decode step over one sequence per host core (all heads), on every core."""
    pool, cores = start_oracle_pool([w])
    n = cores if pool is not None else oracle_sample_size(w)

    def one_round(i):
        seqs = [(i * n + j) % w.batch for j in range(n)]
        if pool is None:
            oracle_step(w, seqs)
        else:
            pool.map(_oracle_task, [(w.name, b) for b in seqs], chunksize=1)

    for i in range(args.warmup):
        one_round(i)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        one_round(args.warmup + i)
        times.append(time.perf_counter() - t0)
    if pool is not None:
        pool.terminate()
    total = sum(times)
    value = n * args.steps / total
    sample = (f"{n} sequences (all heads) per step of the same workload, float64 oracle, "
              + (f"one per host core on {cores} cores" if pool is not None else "one host thread"))
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores if pool is not None else 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args, w: wl.Workload, rank: int, world: int, local_rank: int) -> dict | None:
    import torch
    import __graft_entry__ as ge
    ge.build()
    import paged_kv_cache_153_gb300 as pkv
    log("library ready")

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    t16 = {"f16": torch.float16, "bf16": torch.bfloat16}
    stream = torch.cuda.Stream(device=dev)
    fp8 = w.fp8
    append_fp8 = pkv.pkv_kv_append_e5m2 if w.kv_dtype == "e5m2" else pkv.pkv_kv_append_fp8
    step_fp8 = pkv.pkv_paged_decode_step_e5m2 if w.kv_dtype == "e5m2" else pkv.pkv_paged_decode_step_fp8
    with torch.cuda.stream(stream):
        def up(bits, dt):
            return torch.from_numpy(np.ascontiguousarray(bits)).view(t16[dt]).to(dev)
        q, k_new, v_new = up(w.q, w.dtype), up(w.k_new, w.dtype), up(w.v_new, w.dtype)
        tables = torch.from_numpy(w.block_tables).to(dev)
        lens = torch.from_numpy(w.context_lens).to(dev)
        slots = torch.empty(w.batch, dtype=torch.int64, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        out = torch.empty_like(q)
        max_ctx = int(w.context_lens.max())
        ws = torch.empty(pkv.pkv_decode_workspace_bytes(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                                        w.max_blocks_per_seq, max_ctx, w.partition_tokens),
                         dtype=torch.uint8, device=dev)
        if fp8:
            nb, H, bs, D = w.k_pool.shape
            k_cache = torch.empty(nb, H, bs, D, dtype=torch.uint8, device=dev)
            v_cache = torch.empty_like(k_cache)
            ks, vs = torch.from_numpy(w.k_scale).to(dev), torch.from_numpy(w.v_scale).to(dev)
            all_slots = torch.arange(nb * bs, dtype=torch.int64, device=dev)
            kr = up(w.k_pool, w.dtype).permute(0, 2, 1, 3).reshape(nb * bs, H, D).contiguous()
            vr = up(w.v_pool, w.dtype).permute(0, 2, 1, 3).reshape(nb * bs, H, D).contiguous()
            append_fp8(kr, vr, all_slots, k_cache, v_cache, ks, vs, err_flag=err, stream=stream)
            del kr, vr
        else:
            k_cache, v_cache = up(w.k_pool, w.kv_dtype), up(w.v_pool, w.kv_dtype)
        stream.synchronize()
    log("inputs resident on the device")

    def step(ev0=None, ev1=None):
        # one fused call: slot mapping + append + attention (decode kernel), then the partial merge
        if ev0 is not None:
            ev0.record(stream)
        if fp8:
            step_fp8(q, k_new, v_new, k_cache, v_cache, ks, vs, tables, lens, out, scale=w.scale,
                     max_context_len=max_ctx, workspace=ws, partition_tokens=w.partition_tokens,
                     slot_mapping_out=slots, err_flag=err, stream=stream)
        else:
            pkv.pkv_paged_decode_step(q, k_new, v_new, k_cache, v_cache, tables, lens, out, scale=w.scale,
                                      max_context_len=max_ctx, workspace=ws, partition_tokens=w.partition_tokens,
                                      slot_mapping_out=slots, err_flag=err, stream=stream)
        if ev1 is not None:
            ev1.record(stream)

    launches_per_step = 2          # decode (with slot mapping and append), combine

    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod

    def barrier():
        if dist is not None:
            dist.barrier()

    for i in range(max(args.warmup, 3)):
        step()
        if i == 0:
            stream.synchronize()
            log(f"first step done, device error word {int(err.item())}")
    stream.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())} during warm-up")
    log("warm-up done")

    # The timed steps run back to back on one stream.  The roofline's kernel
    # time is the same events' average per call: events recorded between
    # calls would end each call's programmatic overlap with the next one and
    # time a launch pattern the loop does not have.
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        barrier()
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for _ in range(args.steps):
            step()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    log(f"timed region done: {elapsed_ms / args.steps:.4f} ms per step")
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())} in the timed region")
    dec_avg_ms = elapsed_ms / args.steps   # this rank's calls, on the launching stream
    if dist is not None:
        elapsed_ms = max_over_ranks(elapsed_ms, dist, dev if dist.get_backend() == "nccl" else "cpu")

    # ---- end to end through the host-buffer entry point ---------------------
    pin = lambda a, dt=None: (torch.from_numpy(np.ascontiguousarray(a)).view(t16[dt]) if dt else
                              torch.from_numpy(np.ascontiguousarray(a))).pin_memory()
    e2e = None
    if not fp8:
        h_q, h_k, h_v = pin(w.q, w.dtype), pin(w.k_new, w.kv_dtype), pin(w.v_new, w.kv_dtype)
        h_t, h_l = pin(w.block_tables), pin(w.context_lens)
        h_out = torch.empty(h_q.shape, dtype=h_q.dtype).pin_memory()
        d_q, d_k, d_v = torch.empty_like(q), torch.empty_like(k_new), torch.empty_like(v_new)
        d_t, d_l, d_o = torch.empty_like(tables), torch.empty_like(lens), torch.empty_like(out)

        def host_step():
            pkv.pkv_decode_step_host(h_q, h_k, h_v, h_t, h_l, h_out, d_q, d_k, d_v, d_t, d_l, slots, d_o,
                                     k_cache, v_cache, scale=w.scale, max_context_len=max_ctx, workspace=ws,
                                     partition_tokens=w.partition_tokens, err_flag=err, stream=stream)
            stream.synchronize()           # the result is read on the host every step
        for _ in range(3):
            host_step()
        n_e2e = max(10, min(args.steps, 2000))
        barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_step()
        e2e_s = time.perf_counter() - t0
        if dist is not None:
            e2e_s = max_over_ranks(e2e_s, dist, dev if dist.get_backend() == "nccl" else "cpu")
        log("end-to-end loop done")
        h2d = sum(x.numel() * x.element_size() for x in (h_q, h_k, h_v, h_t, h_l))
        e2e = {"value": replica_throughput(w.batch * n_e2e, world, e2e_s), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": h_out.numel() * h_out.element_size(), "steps": n_e2e,
               "path": "pkv_decode_step_host (pinned host buffers in, result read back every step)"}

    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    # attention's KV + q + out, plus the appended rows written to the cache
    algo = w.algorithmic_bytes() + 2 * w.batch * w.n_kv_heads * w.head_dim * w.kv_elt_bytes
    achieved = algo / (dec_avg_ms * 1e-3) / 1e9
    value = replica_throughput(w.batch * args.steps, world, elapsed_ms * 1e-3)
    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype, "data": "synthetic",
        "config": dict(describe(w), parallelism=f"replicas x{world}" if world > 1 else "1 GPU"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": ncu_traffic(w.name),
                     "kernel": "pkv_paged_decode_step call (decode kernel with slot mapping and append, then the combine kernel), "
                               "average over the back-to-back calls of the timed region",
                     "algorithmic_bytes_per_launch": algo, "avg_launch_ms": dec_avg_ms,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "frac_of_8TBps": achieved / 8000.0},
        "kv_tokens_per_s": world * int(w.context_lens.sum()) * args.steps / (elapsed_ms * 1e-3),
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "e2e": e2e,
    }
    return res


# ---------------------------------------------------------------------------
# copy-on-write block copy (--workload cow)
# ---------------------------------------------------------------------------
COPY_METRIC = "copy-on-write block copy GB/s (K and V bytes read + written), 1 GPU"
COPY_SHAPE = {"num_blocks": 32768, "n_pairs": 8192, "n_kv_heads": 8, "head_dim": 128, "dtype": "bf16"}


def copy_config() -> dict:
    c = COPY_SHAPE
    block_bytes = c["n_kv_heads"] * 16 * c["head_dim"] * 2
    return {"workload": f"cow: {c['n_pairs']} block copies per step (a fork storm) in a pool of {c['num_blocks']} "
                        f"blocks of {c['n_kv_heads']} KV heads x 16 x {c['head_dim']} {c['dtype']}, K and V caches",
            "block_bytes_per_cache": block_bytes, "l2": f"{4 * c['n_pairs'] * block_bytes / 1e9:.2f} GB moved "
            "per step (larger than L2), no flush", **c}


def oracle_copy_rate(budget_s: float) -> tuple[float, str]:
    """The oracle's block copy on the host: GB/s over a bounded sample."""
    from oracle import slots as osl
    c = COPY_SHAPE
    nb, n = 512, 128
    rng = np.random.Generator(np.random.PCG64(77))
    k = rng.integers(0, 2 ** 16, size=(nb, c["n_kv_heads"], 16, c["head_dim"]), dtype=np.uint16)
    v = k.copy()
    src, dst = wl.copy_pairs(nb, n, seed=78)
    pairs = list(zip(src.tolist(), dst.tolist()))
    moved, t0 = 0, time.perf_counter()
    while True:
        osl.copy_blocks(k, pairs)
        osl.copy_blocks(v, pairs)
        moved += 4 * n * k[0].nbytes
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return moved / el / 1e9, f"{n} block copies per pass in a {nb}-block pool, {el:.1f} s, one host thread"


def copy_bytes_per_step() -> int:
    c = COPY_SHAPE
    return 4 * c["n_pairs"] * c["n_kv_heads"] * 16 * c["head_dim"] * 2


def run_copy(args, rank: int, local_rank: int) -> dict | None:
    import torch
    import __graft_entry__ as ge
    ge.build()
    import paged_kv_cache_153_gb300 as pkv
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    c = COPY_SHAPE
    stream = torch.cuda.Stream(device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1200)
    shape = (c["num_blocks"], c["n_kv_heads"], 16, c["head_dim"])
    with torch.cuda.stream(stream):
        k_cache = torch.randint(-2 ** 15, 2 ** 15, shape, dtype=torch.int16, device=dev, generator=gen).view(
            torch.bfloat16)
        v_cache = torch.randint(-2 ** 15, 2 ** 15, shape, dtype=torch.int16, device=dev, generator=gen).view(
            torch.bfloat16)
        src_np, dst_np = wl.copy_pairs(c["num_blocks"], c["n_pairs"], seed=1201)
        src, dst = torch.from_numpy(src_np).to(dev), torch.from_numpy(dst_np).to(dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream.synchronize()
    moved = 4 * c["n_pairs"] * k_cache[0].numel() * 2

    def step():
        pkv.pkv_copy_blocks(src, dst, k_cache, v_cache, err_flag=err, stream=stream)

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for _ in range(args.steps):
            step()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    elapsed_ms = t_start.elapsed_time(t_end)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())} in the timed region")
    per_ms = elapsed_ms / args.steps
    gbs = moved / (per_ms * 1e-3) / 1e9
    # end to end: the step's pair list from pinned host memory, the error word read back
    h_src, h_dst = torch.from_numpy(src_np).pin_memory(), torch.from_numpy(dst_np).pin_memory()
    h_err = torch.zeros(1, dtype=torch.int32).pin_memory()
    d_src, d_dst = torch.empty_like(src), torch.empty_like(dst)

    def host_step():
        d_src.copy_(h_src, non_blocking=True)
        d_dst.copy_(h_dst, non_blocking=True)
        pkv.pkv_copy_blocks(d_src, d_dst, k_cache, v_cache, err_flag=err, stream=stream)
        h_err.copy_(err, non_blocking=True)
        stream.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(3):
            host_step()
        n_e2e = max(10, min(args.steps, 500))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_step()
        e2e_s = time.perf_counter() - t0
    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    cfg = copy_config()
    return {
        "metric": COPY_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": ncu_traffic("cow"), "kernel": "copy_blocks_kernel (pkv_copy_blocks), average over "
                     "the back-to-back calls of the timed region", "algorithmic_bytes_per_launch": moved,
                     "avg_launch_ms": per_ms, "peak_kind": f"{peak_kind} HBM copy bandwidth"},
        "gpu_launches": args.steps, "clocks": clocks.summary(),
        "e2e": {"value": moved * n_e2e / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(h_src.numel() * 4 + h_dst.numel() * 4), "d2h_bytes_per_step": 4,
                "steps": n_e2e, "path": "pair lists from pinned host memory, pkv_copy_blocks, error word read back"},
    }


# ---------------------------------------------------------------------------
# INT8 per-block min-max cache (--workload int8)
# ---------------------------------------------------------------------------
INT8_METRIC = "INT8-KV decode step tokens/s and achieved HBM GB/s, 1 GPU"


def int8_bytes(w) -> int:
    """KV codes (1 byte per element) + the 16-byte scalars of every (block,
    head) slab read + q + out."""
    nblk = sum(-(-int(n) // 16) for n in w.context_lens)
    return nblk * w.n_kv_heads * (2 * 16 * w.head_dim + 16) + 2 * w.batch * w.n_q_heads * w.head_dim * 2


def run_int8(args, rank: int, local_rank: int) -> dict | None:
    import torch
    import __graft_entry__ as ge
    ge.build()
    import paged_kv_cache_153_gb300 as pkv
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = wl.make("gqa8b")
    bf = torch.bfloat16
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(bf).to(dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        kc = torch.empty(w.k_pool.shape, dtype=torch.uint8, device=dev)
        vc = torch.empty_like(kc)
        prm = torch.empty(w.num_blocks, w.n_kv_heads, 4, dtype=torch.float32, device=dev)
        pkv.pkv_kv_quantize_int8(up(w.k_pool), up(w.v_pool), kc, vc, prm, stream=stream)
        q, kn, vn = up(w.q), up(w.k_new), up(w.v_new)
        tables, lens = torch.from_numpy(w.block_tables).to(dev), torch.from_numpy(w.context_lens).to(dev)
        slots = torch.empty(w.batch, dtype=torch.int64, device=dev)
        out = torch.empty_like(q)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        max_ctx = int(w.context_lens.max())
        ws = torch.empty(pkv.pkv_decode_workspace_bytes(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                                        w.max_blocks_per_seq, max_ctx, 0), dtype=torch.uint8,
                         device=dev)
    stream.synchronize()

    def step():
        # one call: the re-quantising append with its slots from the table, the decode (started early, waiting
        # for the append before it reads the cache), then the combine
        pkv.pkv_paged_decode_step_int8(q, kn, vn, kc, vc, prm, tables, lens, out, scale=w.scale,
                                       max_context_len=max_ctx, workspace=ws, slot_mapping_out=slots, err_flag=err,
                                       stream=stream)

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize(dev)
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        torch.cuda.synchronize(dev)
    per_ms = a.elapsed_time(b) / args.steps
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())}")
    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    algo = int8_bytes(w)
    achieved = algo / (per_ms * 1e-3) / 1e9
    return {
        "metric": INT8_METRIC, "value": w.batch * 1e3 / per_ms, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": dict(describe(w), workload=f"int8: the gqa8b shape with the KV cache as INT8 codes + per-(block, "
                       "head) min-max scalars (bf16 q/out)", step="pkv_paged_decode_step_int8: INT8 append "
                       "(slots from the table, re-quantising the block) + INT8 paged decode attention (decode + "
                       "combine)"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic("int8"), "kernel": "pkv_paged_decode_step_int8 call (append, decode "
                     "and combine launches), average over the timed region",
                     "algorithmic_bytes_per_launch": algo, "avg_launch_ms": per_ms,
                     "peak_kind": f"{peak_kind} HBM copy bandwidth"},
        "gpu_launches": 3 * args.steps, "clocks": clocks.summary(), "e2e": None,
    }


# ---------------------------------------------------------------------------
# model-wide cache, whole-step graph (--workload layers)
# ---------------------------------------------------------------------------
LAYERS_METRIC = "model decode step tokens/s (all layers, one graph launch per step), 1 GPU"


def run_layers(args, rank: int, local_rank: int) -> dict | None:
    import torch
    import __graft_entry__ as ge
    ge.build()
    import paged_kv_cache_153_gb300 as pkv
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    li = wl.make_layers()
    w, L = li.base, li.n_layers
    t16 = {"f16": torch.float16, "bf16": torch.bfloat16}[w.kv_dtype]
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(t16).to(dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        kc, vc, q, kn, vn = up(li.k_pool), up(li.v_pool), up(li.q), up(li.k_new), up(li.v_new)
        tables, lens = torch.from_numpy(w.block_tables).to(dev), torch.from_numpy(w.context_lens).to(dev)
        out = torch.empty_like(q)
        slots = torch.empty(w.batch, dtype=torch.int64, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        max_ctx = int(w.context_lens.max())
        ws = torch.empty(pkv.pkv_decode_workspace_bytes(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim,
                                                        w.max_blocks_per_seq, max_ctx, 0), dtype=torch.uint8,
                         device=dev)
    stream.synchronize()
    graph = pkv.StepGraph(q, kn, vn, kc, vc, tables, lens, out, scale=w.scale, max_context_len=max_ctx,
                          workspace=ws, slot_mapping_out=slots, err_flag=err)

    def eager():
        for l in range(L):
            pkv.pkv_paged_decode_step_layer(q[l], kn[l], vn[l], kc, vc, tables, lens, out[l], layer=l,
                                            scale=w.scale, max_context_len=max_ctx, workspace=ws,
                                            slot_mapping_out=slots, err_flag=err, stream=stream)

    def timed(fn, n):
        for _ in range(args.warmup):
            fn()
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / n

    eager_ms = timed(eager, max(10, min(args.steps, 300)))
    with ClockSampler(local_rank) as clocks:
        graph_ms = timed(lambda: graph.launch(stream), args.steps)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())}")
    # end to end: every layer's queries and new rows from pinned host memory, outputs read back
    h_q, h_k, h_v = (torch.from_numpy(np.ascontiguousarray(a)).view(t16).pin_memory() for a in (li.q, li.k_new, li.v_new))
    h_out = torch.empty(out.shape, dtype=t16).pin_memory()

    def host_step():
        q.copy_(h_q, non_blocking=True)
        kn.copy_(h_k, non_blocking=True)
        vn.copy_(h_v, non_blocking=True)
        graph.launch(stream)
        h_out.copy_(out, non_blocking=True)
        stream.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(3):
            host_step()
        n_e2e = max(10, min(args.steps, 1000))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_step()
        e2e_s = time.perf_counter() - t0
    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    algo = L * (w.algorithmic_bytes() + 2 * w.batch * w.n_kv_heads * w.head_dim * w.kv_elt_bytes)
    achieved = algo / (graph_ms * 1e-3) / 1e9
    return {
        "metric": LAYERS_METRIC, "value": w.batch * 1e3 / graph_ms, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": graph_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype, "data": "synthetic",
        "config": {"workload": f"layers: the tiny shape (batch {w.batch}, {w.n_q_heads}/{w.n_kv_heads} heads, head_dim "
                               f"{w.head_dim}, {w.kv_dtype}) through {L} layers of a [num_blocks, {L}, H_kv, 16, d] "
                               "cache: every layer's fused decode step, one graph launch per model step",
                   "num_layers": L, "batch": w.batch, "eager_ms_per_step": eager_ms,
                   "eager": f"{L} pkv_paged_decode_step_layer calls from Python per step"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": f"pkv_step_graph_launch ({2 * L} launches: decode + combine per layer), "
                     "average over the timed region", "algorithmic_bytes_per_launch": algo,
                     "avg_launch_ms": graph_ms, "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "note": "launch-bound: the bytes per layer are ~0.6 MB"},
        "gpu_launches": 2 * L * args.steps, "clocks": clocks.summary(),
        "e2e": {"value": w.batch * n_e2e / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": int(sum(x.numel() * 2 for x in (h_q, h_k, h_v))),
                "d2h_bytes_per_step": int(h_out.numel() * 2), "steps": n_e2e,
                "path": "per-layer queries and new rows from pinned host memory, one graph launch, outputs read back"},
    }


# ---------------------------------------------------------------------------
# paged prefill / extend attention (--workload prefill)
# ---------------------------------------------------------------------------
PREFILL_METRIC = "paged prefill (causal extend attention) TFLOP/s, 1 GPU"


def prefill_config(pi) -> dict:
    return {"workload": f"prefill: {pi.batch} sequences x ({int(pi.cached_lens[0])} cached + {int(pi.new_lens[0])} "
                        f"new tokens), {pi.n_q_heads} query / {pi.n_kv_heads} KV heads, head_dim {pi.head_dim}, "
                        f"{pi.dtype}, block 16", "batch": pi.batch, "num_q_heads": pi.n_q_heads,
            "num_kv_heads": pi.n_kv_heads, "head_dim": pi.head_dim, "new_tokens": int(pi.new_lens.sum()),
            "cached_tokens": int(pi.cached_lens.sum()), "flops_per_step": pi.flops(),
            "l2": "K/V of the batch fit in L2 and are re-read by every query tile; no flush (compute-bound)"}


def oracle_prefill_rate(pi, budget_s: float) -> tuple[float, str]:
    """The oracle's prefill rows on the host: FLOP/s over a bounded sample."""
    from oracle import numerics as on
    from oracle import prefill as op
    q = on.bits_to_f64(pi.q, pi.dtype)
    kc, vc = on.bits_to_f64(pi.k_pool, pi.dtype), on.bits_to_f64(pi.v_pool, pi.dtype)
    pos = op.prefill_positions(pi.context_lens, pi.cu_seqlens)
    flops, done, t0 = 0, 0, time.perf_counter()
    while True:
        t = (done * 997) % q.shape[0]
        op.paged_prefill_attention(q, kc, vc, pi.block_tables, pi.context_lens, pi.cu_seqlens, pi.scale, rows=[t])
        flops += 4 * pi.head_dim * pi.n_q_heads * (pos[t][1] + 1)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return flops / el / 1e12, f"{done} query tokens (all heads), float64, {el:.1f} s on one host thread"


def run_prefill(args, rank: int, local_rank: int) -> dict | None:
    import torch
    import __graft_entry__ as ge
    ge.build()
    import paged_kv_cache_153_gb300 as pkv
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pi = wl.make_prefill()
    stream = torch.cuda.Stream(device=dev)
    bf = torch.bfloat16
    with torch.cuda.stream(stream):
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(bf).to(dev)
        q, kc, vc = up(pi.q), up(pi.k_pool), up(pi.v_pool)
        tables = torch.from_numpy(pi.block_tables).to(dev)
        lens = torch.from_numpy(pi.context_lens).to(dev)
        cu = torch.from_numpy(pi.cu_seqlens).to(dev)
        out = torch.empty_like(q)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream.synchronize()
    mql = int(pi.new_lens.max())

    def step(q_=q, t_=tables, l_=lens, c_=cu):
        pkv.pkv_paged_prefill_attention(q_, kc, vc, t_, l_, c_, out, scale=pi.scale, max_query_len=mql,
                                        err_flag=err, stream=stream)

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())} during warm-up")
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for _ in range(args.steps):
            step()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    per_ms = t_start.elapsed_time(t_end) / args.steps
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())} in the timed region")
    tflops = pi.flops() / (per_ms * 1e-3) / 1e12
    # end to end: queries, tables, lengths and offsets from pinned host memory, the output read back
    h_q = torch.from_numpy(np.ascontiguousarray(pi.q)).view(bf).pin_memory()
    h_t = torch.from_numpy(pi.block_tables).pin_memory()
    h_l, h_c = torch.from_numpy(pi.context_lens).pin_memory(), torch.from_numpy(pi.cu_seqlens).pin_memory()
    h_out = torch.empty(out.shape, dtype=bf).pin_memory()
    d_q, d_t, d_l, d_c = torch.empty_like(q), torch.empty_like(tables), torch.empty_like(lens), torch.empty_like(cu)

    def host_step():
        for d_, h_ in ((d_q, h_q), (d_t, h_t), (d_l, h_l), (d_c, h_c)):
            d_.copy_(h_, non_blocking=True)
        step(d_q, d_t, d_l, d_c)
        h_out.copy_(out, non_blocking=True)
        stream.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(2):
            host_step()
        n_e2e = max(5, min(args.steps, 100))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            host_step()
        e2e_s = time.perf_counter() - t0
    if rank != 0:
        return None
    peak, kind = 1935.8, "fallback"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        pass
    return {
        "metric": PREFILL_METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": prefill_config(pi),
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "traffic": ncu_traffic("prefill"), "kernel": "paged_prefill_kernel (pkv_paged_prefill_attention), "
                     "average over the back-to-back calls of the timed region",
                     "algorithmic_flops_per_launch": pi.flops(), "avg_launch_ms": per_ms,
                     "peak_kind": f"{kind} dense bf16 (burst)"},
        "gpu_launches": args.steps, "clocks": clocks.summary(),
        "e2e": {"value": pi.flops() * n_e2e / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(sum(x.numel() * x.element_size() for x in (h_q, h_t, h_l, h_c))),
                "d2h_bytes_per_step": int(h_out.numel() * 2), "steps": n_e2e,
                "path": "queries and tables from pinned host memory, pkv_paged_prefill_attention, output read back"},
    }


SINGLE_GPU_WORKLOADS = ("prefill", "cow", "int8", "layers")

# decode configurations a default run times after the headline one
EXTRA_CONFIGS = ("gqa8b", "prefix", "fp8long")


def make_workload(name: str) -> wl.Workload:
    if name == "fp8long_e5m2":
        return wl.make("fp8long", fp8="e5m2")
    return wl.make(name)


def config_summary(res: dict) -> dict:
    """The per-configuration record of a default run: its timing, roofline,
    clocks and end-to-end number (the headline keys of its own line)."""
    keep = ("ms_per_step", "value", "unit", "steps", "dtype", "kv_tokens_per_s", "roofline", "clocks", "e2e",
            "gpu_launches")
    out = {k: res[k] for k in keep if k in res}
    out["workload"] = res["config"]["workload"]
    out["l2"] = res["config"]["l2"]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None,
                    choices=list(wl.CONFIG_NAMES) + ["fp8long_e5m2", "cow", "prefill", "layers", "int8"],
                    help="one workload alone (default: the headline mha7b line with the other large decode "
                         "configurations under 'configs')")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    extras = args.workload is None           # the default run also times EXTRA_CONFIGS
    if args.workload is None:
        args.workload = "mha7b"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    # Single-GPU workloads: refused under torchrun before any CUDA call.  The
    # prefill kernel's clusters share K/V tiles by TMA multicast, which is for
    # single-GPU processes only; the others have no replica path.
    if world > 1 and args.workload in SINGLE_GPU_WORKLOADS:
        if rank == 0:
            line = {"unavailable": f"--workload {args.workload} runs on one GPU only (world size {world} refused "
                                   "before any CUDA call)"}
            if args.impl == "reference":
                line = {"impl": "reference", **line}
            print(json.dumps(line), flush=True)
        return

    if args.workload == "int8":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the int8 bench line has no reference arm; "
                              "its parity is in tests/test_gpu_int8.py"}), flush=True)
            return
        res = run_int8(args, rank, local_rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if args.workload == "layers":
        if args.impl == "reference":
            if rank != 0:
                return
            li = wl.make_layers()
            w = li.base
            t0, n = time.perf_counter(), 0
            while time.perf_counter() - t0 < max(1.0, 0.01 * args.steps):
                oracle_step(w, [n % w.batch])
                n += 1
            el = time.perf_counter() - t0
            rate = n / li.n_layers / el            # one token through every layer
            print(json.dumps({
                "impl": "reference", "metric": LAYERS_METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.batch / rate * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": "layers (oracle: one layer step per sequence, "
                                                            f"x {li.n_layers} layers)"},
                "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                                 "sample": f"{n} single-sequence layer steps, {el:.1f} s, one host thread"},
                "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                flush=True)
            return
        res = run_layers(args, rank, local_rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if args.workload == "prefill":
        pi = wl.make_prefill()
        if args.impl == "reference":
            if rank != 0:
                return
            rate, sample = oracle_prefill_rate(pi, budget_s=max(1.0, 0.05 * args.steps))
            print(json.dumps({
                "impl": "reference", "metric": PREFILL_METRIC, "value": rate, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": pi.flops() / (rate * 1e12) * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": prefill_config(pi),
                "cpu_baseline": {"value": rate, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": sample},
                "e2e": {"value": rate, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                flush=True)
            return
        res = run_prefill(args, rank, local_rank)
        if res is not None:
            if not args.no_cpu_baseline:
                rate, sample = oracle_prefill_rate(pi, budget_s=10.0)
                res["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                                       "sample": sample}
            print(json.dumps(res), flush=True)
        return

    if args.workload == "cow":
        if args.impl == "reference":
            if rank != 0:
                return
            rate, sample = oracle_copy_rate(budget_s=max(1.0, 0.02 * args.steps))
            print(json.dumps({
                "impl": "reference", "metric": COPY_METRIC, "value": rate, "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": copy_bytes_per_step() / (rate * 1e9) * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": copy_config(),
                "cpu_baseline": {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
                "e2e": {"value": rate, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
                flush=True)
            return
        res = run_copy(args, rank, local_rank)
        if res is not None:
            if not args.no_cpu_baseline:
                rate, sample = oracle_copy_rate(budget_s=10.0)
                res["cpu_baseline"] = {"value": rate, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                       "sample": sample}
            print(json.dumps(res), flush=True)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        w = make_workload(args.workload)
        print(json.dumps(run_reference(args, w)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    w = make_workload(args.workload)
    log(f"workload {w.name} generated")
    others = []
    if extras and world == 1:
        others = [make_workload(name) for name in EXTRA_CONFIGS]
        log("other configurations generated")
    pool, cores = None, 1
    if world == 1 and not args.no_cpu_baseline:
        pool, cores = start_oracle_pool([w] + others)      # before the first CUDA call
    res = run_gpu(args, w, rank, world, local_rank)
    if res is not None and others:
        res["configs"] = {}
        for ow in others:
            sub = run_gpu(args, ow, rank, world, local_rank)
            res["configs"][ow.name] = config_summary(sub)
    if res is not None:
        if pool is not None:
            res["cpu_baseline"] = cpu_baseline(w, pool=pool, cores=cores)
            for ow in others:
                res["configs"][ow.name]["cpu_baseline"] = cpu_baseline(ow, budget_s=6.0, pool=pool, cores=cores)
        if extras and world == 1:
            res["gpu_launches"] += sum(c["gpu_launches"] for c in res["configs"].values())
        print(json.dumps(res), flush=True)
    if pool is not None:
        pool.terminate()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
