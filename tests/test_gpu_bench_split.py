"""The benchmark's path for more than one GPU (the step split across ranks: the
prefill ring over NCCL, the decode merged by cp_lse_ag_out_rs), run at one rank
on one GPU: the same code, with a ring of one step and collectives over one
rank."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_split_step_runs_at_one_rank():
    r = subprocess.run([sys.executable, "bench.py", "--cp-dist", "--steps", "1", "--warmup", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 1 and d["scaling"] == "strong" and d["value"] > 0
    assert "context parallel over 1 ranks" in d["config"]["parallelism"]
    assert d["parts"]["ring_ms"] > 0 and d["parts"]["decode_merge_ms"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
