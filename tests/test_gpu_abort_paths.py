"""Failure detection of the tcgen05 kernels through their real abort path.

A child process runs with RA_WAIT_LIMIT_CYCLES=64, so the first wait of every
tensor-core kernel that is not satisfied at once expires: the ring kernel in its
three variants and its several-request form, the ring step and the block kernel.  Each kernel must
then record RA_ERR_TIMEOUT in its own module's error word, let its copies and
MMAs in flight land, free tensor memory and return; ra_device_status() must
report the error with the module's name, and the context must stay usable for
the next launch.  No fault, trap or unbounded wait is involved.
"""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys, torch
sys.path.insert(0, sys.argv[1])
from context_long_sequence_ring_gb300 import ringattn as ra
dev = torch.device("cuda:0")
g = torch.Generator().manual_seed(3)
def rnd(*shape):
    return torch.randn(*shape, generator=g).to(torch.bfloat16).to(dev)
out = {}
def status(name):
    st = ra.device_status()
    out[name] = [int(st), ra.last_error() if st else ""]
# ring-order attention: the two-head pipeline, the one-head kernel, the adjacent-tile schedule
q, k, v = rnd(1024, 4, 128), rnd(1024, 2, 128), rnd(1024, 2, 128)
ra.ring_attn_fwd(q, k, v, True, 2)
status("ring")
ra.ring_attn_fwd(q, k, v, True, 2, variant=1)
status("ring_one_head")
ra.ring_attn_fwd(q, k, v, True, 2, variant=3)
status("ring_tiles")
# several requests in one call (rows of the gathered layout: 640 + 384)
ra.ring_attn_fwd_varlen(q, k, v, [640, 384], True, 2)
status("varlen")
# one rank's ring step (the across-devices kernel)
ra.ring_step_fwd(q[:512], k[:512], v[:512], 2, 0, 0, True)
status("ring_step")
# block partial attention
ra.attn_block_fwd(q[:256], k, v, 768, 0, True)
status("block")
# the context still works: a kernel without waits gives the exact result
src = torch.arange(64 * 8, dtype=torch.float32, device=dev).view(64, 8)
idx = torch.randperm(64, generator=g).to(torch.int32).to(dev)
got = ra.gather_rows(src, idx)
out["gather_ok"] = bool(torch.equal(got.cpu(), src.cpu()[idx.long().cpu()]))
out["final_status"] = int(ra.device_status())
print(json.dumps(out))
"""


@pytest.mark.gpu
def test_timeouts_are_reported_per_module_and_context_survives():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    env = dict(os.environ, RA_WAIT_LIMIT_CYCLES="64")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    from context_long_sequence_ring_gb300 import ringattn as ra

    for name, module in (("ring", "ring attention bf16"), ("ring_one_head", "ring attention bf16"),
                         ("ring_tiles", "ring attention bf16"), ("varlen", "ring attention bf16"),
                         ("ring_step", "ring step"), ("block", "block attention bf16")):
        st, msg = res[name]
        assert st == ra.RA_ERR_TIMEOUT, (name, st, msg)
        assert module in msg, (name, msg)
    assert res["gather_ok"]
    assert res["final_status"] == 0
