"""Shared helpers of the GPU parity tests (not collected)."""
import numpy as np
import pytest
import torch

TOL = {
    # bf16 inputs, fp32 accumulation: O max / mean abs error, LSE abs error
    torch.bfloat16: dict(o_max=2e-2, o_mean=2e-3, lse=1e-3),
    torch.float32: dict(o_max=1e-4, o_mean=1e-4, lse=1e-4),
}


def ra_lib():
    """The binding, with the library built; a GPU is required (no skip)."""
    from context_long_sequence_ring_gb300 import build, ringattn
    import os
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    if not os.path.exists(build.LIB):
        build.build()
    ringattn.lib()
    return ringattn


def assert_parity(o_gpu, O_ref, lse_gpu, L_ref, dtype, what=""):
    t = TOL[dtype]
    o = o_gpu.float().cpu().numpy() if hasattr(o_gpu, "cpu") else np.asarray(o_gpu)
    l = lse_gpu.float().cpu().numpy() if hasattr(lse_gpu, "cpu") else np.asarray(lse_gpu)
    e = np.abs(o.astype(np.float64) - O_ref)
    le = np.abs(l.astype(np.float64) - L_ref)
    assert np.isfinite(o).all() and np.isfinite(l).all(), what + ": non-finite output"
    assert e.max() <= t["o_max"], "%s: O max err %.3g" % (what, e.max())
    assert e.mean() <= t["o_mean"], "%s: O mean err %.3g" % (what, e.mean())
    assert le.max() <= t["lse"], "%s: LSE max err %.3g" % (what, le.max())
    return e.max(), e.mean(), le.max()


def check_status(ra):
    st = ra.device_status()
    assert st == 0, "device status %d: %s" % (st, ra.last_error())


gpu = pytest.mark.gpu
