"""bench.py refuses its single-GPU workloads under a multi-process launch,
before any CUDA call (CPU-only)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROBE = r"""
import contextlib, io, json, sys
sys.argv = ["bench.py", "--workload", sys.argv[1], "--steps", "1", "--warmup", "3"] + sys.argv[2:]
import bench
buf = io.StringIO()
with contextlib.redirect_stdout(buf):
    bench.main()
import torch
print(json.dumps({"out": buf.getvalue(),
                  "library_loaded": "paged_kv_cache_153_gb300" in sys.modules,
                  "cuda_initialized": bool(torch.cuda.is_initialized())}))
"""


@pytest.mark.parametrize("workload", ["prefill", "cow", "int8", "layers"])
@pytest.mark.parametrize("impl", ["ours", "reference"])
def test_single_gpu_workloads_refused_under_torchrun(workload, impl):
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, "-c", PROBE, workload, "--impl", impl], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    rep = json.loads(res.stdout.strip().splitlines()[-1])
    line = json.loads(rep["out"].strip())
    assert "one GPU only" in line["unavailable"]
    assert (line.get("impl") == "reference") == (impl == "reference")
    assert not rep["library_loaded"] and not rep["cuda_initialized"]


def test_other_ranks_print_nothing():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, "-c", PROBE, "prefill"], cwd=ROOT, env=env, capture_output=True,
                         text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    rep = json.loads(res.stdout.strip().splitlines()[-1])
    assert rep["out"] == "" and not rep["library_loaded"]
