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


def test_split_workload_matches_the_single_device_step():
    # the split step at one rank (NCCL over one rank) against the single-device kernels on the same
    # seeded workload: the ring-step prefill equals the 16-virtual-rank ring kernel and the decode
    # through cp_lse_ag_out_rs equals ra_cp_decode
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from context_long_sequence_ring_gb300 import ringattn as ra
    ra.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    os.environ.setdefault("MASTER_PORT", "29541")
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=dev)
    try:
        wl = bench.DistWorkload(ra, dev, 0, 1)
        wl.step()
        torch.cuda.synchronize()
        assert ra.device_status() == 0, ra.last_error()
        P, D = bench.PREFILL, bench.DECODE
        o_ref, l_ref = ra.ring_attn_fwd(wl.q, wl.k, wl.v, True, P["N"])      # one rank holds the whole sequence
        e = (wl.o.float() - o_ref.float()).abs()
        assert e.max().item() <= 2e-2 and e.mean().item() <= 5e-4
        assert (wl.lse - l_ref).abs().max().item() <= 1e-3
        od, ld = ra.cp_decode(wl.qd, wl.kc, wl.vc, wl.bt, wl.ctx, D["I"], D["pcp"], D["dcp"], split_blocks=D["split"],
                              out_dtype=torch.float32)
        assert (wl.od - od).abs().max().item() <= 1e-5 and (wl.ld - ld).abs().max().item() <= 1e-5
    finally:
        dist.destroy_process_group()
