"""The allocation-free decode entry point against the workspace one, through
the C ABI.

Some callers cannot allocate device memory on the decode path: a runtime that
reserves all device memory at start-up and forbids allocation afterwards, an
allocator that cannot hand out raw scratch, or a process whose device
footprint must stay fixed.  ra_cp_decode_noalloc serves them with a fixed
scratch array inside the library; its results must match ra_cp_decode's, call
after call, although every call reuses the same scratch.

This file is named so that pytest collects it last.
"""
import pytest
import torch

from context_long_sequence_ring_gb300 import inputs as I
from tests._gpu import ra_lib, check_status, TOL

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _cache(ra, seed, R, lo, hi, bs, I_, pcp, dcp, Hkv, d):
    W = pcp * dcp
    wl = I.decode_workload(seed, R, lo, hi, bs, pcp, dcp)
    T = wl["total_tokens"]
    kt = I.synth_normal(seed, I.TID_K, (T, Hkv, d), torch.bfloat16).to(DEV)
    vt = I.synth_normal(seed, I.TID_V, (T, Hkv, d), torch.bfloat16).to(DEV)
    ctx = wl["ctx_lens"]
    qsl = torch.zeros(R + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(ctx, 0)
    pos = torch.cat([torch.arange(int(L), dtype=torch.int32) for L in ctx])
    bt = wl["block_table"].to(DEV)
    slot = ra.cp_slot_mapping(qsl.to(DEV), pos.to(DEV), bt, bs, I_, pcp, dcp)
    kc = torch.zeros((W, wl["num_blocks"], Hkv, bs, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    ra.cp_kv_scatter(kt, vt, slot, kc, vc)
    check_status(ra)
    return kc, vc, bt, ctx.to(DEV)


def test_noalloc_decode_matches_workspace_decode_on_consecutive_calls():
    ra = ra_lib()
    R, bs, I_, pcp, dcp, Hq, Hkv, d, split = 6, 64, 16, 2, 2, 8, 2, 128, 2
    kc, vc, bt, ctx = _cache(ra, 21, R, 200, 6000, bs, I_, pcp, dcp, Hkv, d)
    need = ra.cp_decode_workspace_size(R, Hq, d, bt.shape[1], pcp, dcp, split)
    assert need <= 32 << 20
    tol = TOL[torch.bfloat16]
    for call, seed in enumerate((31, 32)):     # two calls in a row share the same scratch
        q = I.synth_normal(seed, I.TID_Q, (R, Hq, d), torch.bfloat16).to(DEV)
        o_ref, l_ref = ra.cp_decode(q, kc, vc, bt, ctx, I_, pcp, dcp, split_blocks=split)
        o, lse = ra.cp_decode_noalloc(q, kc, vc, bt, ctx, I_, pcp, dcp, split_blocks=split)
        check_status(ra)
        e = (o.float() - o_ref.float()).abs()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert e.max().item() <= tol["o_max"], "call %d: O max err %g" % (call, e.max().item())
        assert e.mean().item() <= tol["o_mean"], "call %d: O mean err %g" % (call, e.mean().item())
        assert (lse - l_ref).abs().max().item() <= tol["lse"], "call %d: LSE" % call


def test_noalloc_decode_after_a_larger_call_with_another_split():
    # A large decode leaves its partials in the shared scratch; a smaller one with another split
    # reads only what it wrote itself, so the stale contents must not leak into its result.
    ra = ra_lib()
    bs, I_, pcp, dcp, Hq, Hkv, d = 64, 16, 2, 2, 8, 2, 128
    tol = TOL[torch.bfloat16]
    big = _cache(ra, 23, 12, 3000, 20000, bs, I_, pcp, dcp, Hkv, d)
    small = _cache(ra, 24, 3, 100, 2500, bs, I_, pcp, dcp, Hkv, d)
    for (kc, vc, bt, ctx), R, split, seed in ((big, 12, 1, 41), (small, 3, 3, 42), (big, 12, 2, 43)):
        assert ra.cp_decode_workspace_size(R, Hq, d, bt.shape[1], pcp, dcp, split) <= 32 << 20
        q = I.synth_normal(seed, I.TID_Q, (R, Hq, d), torch.bfloat16).to(DEV)
        o_ref, l_ref = ra.cp_decode(q, kc, vc, bt, ctx, I_, pcp, dcp, split_blocks=split)
        o, lse = ra.cp_decode_noalloc(q, kc, vc, bt, ctx, I_, pcp, dcp, split_blocks=split)
        check_status(ra)
        e = (o.float() - o_ref.float()).abs()
        assert e.max().item() <= tol["o_max"] and e.mean().item() <= tol["o_mean"], "R=%d split=%d" % (R, split)
        assert (lse - l_ref).abs().max().item() <= tol["lse"], "R=%d split=%d" % (R, split)


def test_warm_noalloc_call_commits_no_device_memory():
    ra = ra_lib()
    R, bs, I_, pcp, dcp, Hq, Hkv, d, split = 4, 64, 16, 2, 2, 8, 2, 128, 2
    kc, vc, bt, ctx = _cache(ra, 25, R, 500, 5000, bs, I_, pcp, dcp, Hkv, d)
    q = I.synth_normal(44, I.TID_Q, (R, Hq, d), torch.bfloat16).to(DEV)
    o = torch.empty((R, Hq, d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((R, Hq), dtype=torch.float32, device=DEV)
    ra.cp_decode_noalloc(q, kc, vc, bt, ctx, I_, pcp, dcp, split_blocks=split, o=o, lse=lse)   # warm-up call
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        ra.cp_decode_noalloc(q, kc, vc, bt, ctx, I_, pcp, dcp, split_blocks=split, o=o, lse=lse)
    torch.cuda.synchronize()
    check_status(ra)
    assert torch.cuda.mem_get_info()[0] == free0, "a warm call changed the device's free memory"


def test_noalloc_decode_rejects_a_decode_larger_than_its_scratch():
    ra = ra_lib()
    R, Hq, Hkv, d, bs, I_, pcp, dcp = 2, 32, 8, 128, 64, 16, 2, 4
    q = torch.zeros((R, Hq, d), dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros((pcp * dcp, 4, Hkv, bs, d), dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros((R, 4096), dtype=torch.int32, device=DEV)      # many virtual blocks
    ctx = torch.ones(R, dtype=torch.int32, device=DEV)
    assert ra.cp_decode_workspace_size(R, Hq, d, 4096, pcp, dcp, 1) > 32 << 20
    with pytest.raises(ra.RingAttnError) as ei:
        ra.cp_decode_noalloc(q, kc, kc, bt, ctx, I_, pcp, dcp, split_blocks=1)
    assert ei.value.status == ra.RA_ERR_INVALID_ARG and "scratch" in str(ei.value)
    check_status(ra)
