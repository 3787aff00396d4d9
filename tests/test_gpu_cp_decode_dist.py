"""Decode across devices on one GPU: the per-device split-KV partials
(ra_cp_decode_partials) and step 2 of cp_lse_ag_out_rs (ra_cp_lse_rescale),
against ra_cp_decode and the float64 oracle.  Steps 1 and 3 of the collective
(all-gather of the LSEs, reduce-scatter of the outputs) are emulated by
stacking and summing the devices' tensors."""
import numpy as np
import pytest
import torch

import oracle
from context_long_sequence_ring_gb300 import inputs as I
from tests._gpu import ra_lib, check_status, TOL

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.fixture(scope="module")
def ra():
    return ra_lib()


def _case(ra, seed, R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d):
    W = pcp * dcp
    wl = I.decode_workload(seed, R, lo, hi, bs, pcp, dcp)
    T = wl["total_tokens"]
    kt = I.synth_normal(seed, I.TID_K, (T, Hkv, d), torch.bfloat16)
    vt = I.synth_normal(seed, I.TID_V, (T, Hkv, d), torch.bfloat16)
    q = I.synth_normal(seed, I.TID_Q, (R, Hq, d), torch.bfloat16)
    ctx = wl["ctx_lens"]
    qsl = torch.zeros(R + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(ctx, 0)
    pos = torch.cat([torch.arange(int(L), dtype=torch.int32) for L in ctx])
    bt = wl["block_table"].to(DEV)
    slot = ra.cp_slot_mapping(qsl.to(DEV), pos.to(DEV), bt, bs, I_, pcp, dcp)
    kc = torch.zeros((W, wl["num_blocks"], Hkv, bs, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    ra.cp_kv_scatter(kt.to(DEV), vt.to(DEV), slot, kc, vc)
    check_status(ra)
    # the oracle's own cache, filled by the oracle's slot mapping and scatter from the host tensors
    oslot = oracle.cp_slot_mapping(qsl.numpy(), pos.numpy(), wl["block_table"].numpy(), bs, I_, pcp, dcp)
    kc_np = np.zeros((W, wl["num_blocks"], Hkv, bs, d))
    vc_np = np.zeros_like(kc_np)
    oracle.cp_kv_scatter(kt.double().numpy(), vt.double().numpy(), oslot, kc_np, vc_np, bs)
    return dict(q=q, kt=kt, vt=vt, qsl=qsl, kc=kc, vc=vc, bt=bt, ctx=ctx.to(DEV), W=W, kc_np=kc_np, vc_np=vc_np,
                bt_np=wl["block_table"].numpy(), ctx_np=wl["ctx_lens"].numpy())


CASES = [(3, 300, 5000, 64, 16, 2, 2, 8, 2, 128, 2), (5, 1000, 9000, 128, 16, 2, 4, 32, 8, 128, 4),
         (2, 50, 700, 32, 8, 1, 2, 4, 4, 64, 1)]


@pytest.mark.parametrize("R,lo,hi,bs,I_,pcp,dcp,Hq,Hkv,d,split", CASES)
def test_partials_of_all_devices_match_oracle_and_merge_to_decode(ra, R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d, split):
    c = _case(ra, 61, R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d)
    qd = c["q"].to(DEV)
    op, lp = ra.cp_decode_partials(qd, c["kc"], c["vc"], c["bt"], c["ctx"], I_, pcp, dcp, split_blocks=split)
    o_ref, l_ref = ra.cp_decode(qd, c["kc"], c["vc"], c["bt"], c["ctx"], I_, pcp, dcp, split_blocks=split,
                                out_dtype=torch.float32)
    o, l = ra.lse_merge(op, lp, out_dtype=torch.float32)
    check_status(ra)
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)       # the same kernels, the same merge
    O, L, ns = oracle.cp_decode_partials(c["q"], c["kc_np"], c["vc_np"], c["bt_np"], c["ctx_np"], bs, I_, pcp, dcp,
                                         split)
    assert op.shape[0] == c["W"] * ns
    lg = lp.cpu().numpy()
    fin = np.isfinite(L)
    assert np.array_equal(np.isfinite(lg), fin)                  # the same partials are empty
    tol = TOL[torch.bfloat16]
    assert np.abs(lg[fin] - L[fin]).max() <= tol["lse"]
    e = np.abs(op.cpu().numpy()[fin] - O[fin])
    assert e.max() <= tol["o_max"] and e.mean() <= tol["o_mean"]


@pytest.mark.parametrize("R,lo,hi,bs,I_,pcp,dcp,Hq,Hkv,d,split", CASES[:2])
def test_partials_of_one_device_equal_its_share(ra, R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d, split):
    # a device that holds only its own shard computes exactly its share of the partials
    c = _case(ra, 62, R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d)
    qd = c["q"].to(DEV)
    op, lp = ra.cp_decode_partials(qd, c["kc"], c["vc"], c["bt"], c["ctx"], I_, pcp, dcp, split_blocks=split)
    ns = op.shape[0] // c["W"]
    for w in range(c["W"]):
        ow, lw = ra.cp_decode_partials(qd, c["kc"][w:w + 1].contiguous(), c["vc"][w:w + 1].contiguous(), c["bt"],
                                       c["ctx"], I_, pcp, dcp, dev0=w, split_blocks=split)
        check_status(ra)
        ref_l = lp[w * ns:(w + 1) * ns]
        assert torch.equal(lw, ref_l)
        live = torch.isfinite(lw)
        assert torch.equal(ow[live], op[w * ns:(w + 1) * ns][live])


@pytest.mark.parametrize("group", [1, 2])
def test_dcp_merge_across_emulated_devices(ra, group):
    # devices are grouped `group` per rank; each rank merges its own partials, then the ranks run
    # cp_lse_ag_out_rs: all-gather of LSE (stack), rescale (kernel), reduce-scatter (sum + slice)
    R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d, split = 5, 1000, 9000, 128, 16, 2, 4, 32, 8, 128, 4
    c = _case(ra, 63, R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d)
    qd = c["q"].to(DEV)
    ranks = c["W"] // group
    outs = []
    for w in range(ranks):
        devs = slice(w * group, (w + 1) * group)
        op, lp = ra.cp_decode_partials(qd, c["kc"][devs].contiguous(), c["vc"][devs].contiguous(), c["bt"], c["ctx"],
                                       I_, pcp, dcp, dev0=w * group, split_blocks=split)
        outs.append(ra.lse_merge(op, lp, out_dtype=torch.float32))
    lse_all = torch.stack([x[1] for x in outs])                          # step 1: all-gather
    scaled, lse_tot = [], []
    for w in range(ranks):
        s, lt = ra.cp_lse_rescale(outs[w][0], lse_all, w)                 # step 2, on rank w
        scaled.append(s)
        lse_tot.append(lt)
    total = torch.stack(scaled).sum(0)                                   # step 3: reduce ...
    O = torch.cat([total[w] for w in range(ranks)], dim=1)               # ... and scatter over heads
    L = torch.cat(lse_tot, dim=1)
    check_status(ra)
    o_ref, l_ref = ra.cp_decode(qd, c["kc"], c["vc"], c["bt"], c["ctx"], I_, pcp, dcp, split_blocks=split,
                                out_dtype=torch.float32)
    assert (O - o_ref).abs().max().item() <= 1e-5 and (L - l_ref).abs().max().item() <= 1e-5
    tol = TOL[torch.bfloat16]
    for r in range(R):
        s0, s1 = int(c["qsl"][r]), int(c["qsl"][r + 1])
        Or, Lr = oracle.decode_reference(c["q"][r], c["kt"][s0:s1], c["vt"][s0:s1])
        assert np.abs(O[r].cpu().numpy() - Or).max() <= tol["o_max"]
        assert np.abs(L[r].cpu().numpy() - Lr).max() <= tol["lse"]


def test_lse_rescale_against_the_oracle_collective(ra):
    W, R, Hq, d = 4, 3, 8, 128
    g = torch.Generator().manual_seed(64)
    o = torch.randn((W, R, Hq, d), generator=g, dtype=torch.float64)
    lse = torch.randn((W, R, Hq), generator=g, dtype=torch.float64) * 3
    lse[0, 1, 3] = -np.inf
    lse[:, 2, 6] = -np.inf
    o[0, 1, 3] = np.nan                        # an empty partial's O must not be read
    o[:, 2, 6] = np.nan
    lse_all = lse.float().to(DEV)
    parts = [ra.cp_lse_rescale(o[w].float().to(DEV), lse_all, w) for w in range(W)]
    check_status(ra)
    total = sum(p[0] for p in parts)
    ref = oracle.cp_lse_ag_out_rs(list(np.nan_to_num(o.numpy())), list(lse.numpy()))
    for w in range(W):
        assert np.abs(total[w].cpu().numpy() - ref[w][0]).max() <= 1e-5
        got = parts[w][1].cpu().numpy()
        fin = np.isfinite(ref[w][1])
        assert np.array_equal(np.isfinite(got), fin) and np.abs(got[fin] - ref[w][1][fin]).max() <= 1e-5


def test_a2a_merge_across_emulated_devices(ra):
    # the all-to-all form: each rank lays out its partial by head owner (kernel), the all-to-all is
    # emulated by handing slot v of every rank to rank v, and rank v merges W partials (kernel)
    R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d, split = 5, 1000, 9000, 128, 16, 2, 4, 32, 8, 128, 4
    c = _case(ra, 65, R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d)
    qd = c["q"].to(DEV)
    W = c["W"]
    splits = []
    for w in range(W):
        op, lp = ra.cp_decode_partials(qd, c["kc"][w:w + 1].contiguous(), c["vc"][w:w + 1].contiguous(), c["bt"],
                                       c["ctx"], I_, pcp, dcp, dev0=w, split_blocks=split)
        ow, lw = ra.lse_merge(op, lp, out_dtype=torch.float32)
        splits.append(ra.cp_head_split(ow, lw, W))
    outs = []
    for v in range(W):                                        # rank v receives slot v of every rank
        o_parts = torch.stack([splits[w][0][v] for w in range(W)])
        l_parts = torch.stack([splits[w][1][v] for w in range(W)])
        outs.append(ra.lse_merge(o_parts, l_parts, out_dtype=torch.float32))
    check_status(ra)
    O = torch.cat([x[0] for x in outs], dim=1)
    L = torch.cat([x[1] for x in outs], dim=1)
    o_ref, l_ref = ra.cp_decode(qd, c["kc"], c["vc"], c["bt"], c["ctx"], I_, pcp, dcp, split_blocks=split,
                                out_dtype=torch.float32)
    assert (O - o_ref).abs().max().item() <= 1e-5 and (L - l_ref).abs().max().item() <= 1e-5
    tol = TOL[torch.bfloat16]
    for r in range(R):
        s0, s1 = int(c["qsl"][r]), int(c["qsl"][r + 1])
        Or, Lr = oracle.decode_reference(c["q"][r], c["kt"][s0:s1], c["vt"][s0:s1])
        assert np.abs(O[r].cpu().numpy() - Or).max() <= tol["o_max"]
        assert np.abs(L[r].cpu().numpy() - Lr).max() <= tol["lse"]


def test_head_split_layout_and_empty_rows(ra):
    W, R, Hq, d = 4, 3, 8, 64
    g = torch.Generator().manual_seed(66)
    o = torch.randn((R, Hq, d), generator=g)
    lse = torch.randn((R, Hq), generator=g)
    lse[1, 5] = -float("inf")
    o[1, 5] = float("nan")                                     # not read: its LSE is -inf
    os_, ls_ = ra.cp_head_split(o.to(DEV), lse.to(DEV), W)
    check_status(ra)
    hs = Hq // W
    for v in range(W):
        for j in range(hs):
            h = v * hs + j
            assert torch.equal(ls_[v, :, j].cpu(), lse[:, h])
            want = o[:, h].clone()
            want[~torch.isfinite(lse[:, h])] = 0.0
            assert torch.equal(os_[v, :, j].cpu(), want)


def test_dcp_merge_at_full_decode_size(ra):
    """The 64-request decode workload (contexts U[4096, 131072], Hq=32, Hkv=8, block 128, interleave
    16, pcp=2, dcp=4) with each of the 8 cache devices as its own rank: partials, local merge,
    cp_lse_ag_out_rs with the rescale kernel (all-gather and reduce-scatter emulated), against
    ra_cp_decode on the same cache, and sampled requests against plain attention."""
    R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d, split, seed = 64, 4096, 131072, 128, 16, 2, 4, 32, 8, 128, 16, 4
    W = pcp * dcp
    wl = I.decode_workload(seed, R, lo, hi, bs, pcp, dcp)
    T = wl["total_tokens"]
    tab = I.normal_table(torch.bfloat16)
    kt = ra.synth_fill(I.tensor_key(seed, I.TID_K), tab, (T, Hkv, d))
    vt = ra.synth_fill(I.tensor_key(seed, I.TID_V), tab, (T, Hkv, d))
    ctx = wl["ctx_lens"]
    qsl = torch.zeros(R + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(ctx, 0)
    pos = torch.cat([torch.arange(int(L), dtype=torch.int32) for L in ctx])
    bt = wl["block_table"].to(DEV)
    slot = ra.cp_slot_mapping(qsl.to(DEV), pos.to(DEV), bt, bs, I_, pcp, dcp)
    kc = torch.empty((W, wl["num_blocks"], Hkv, bs, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.empty_like(kc)
    ra.cp_kv_scatter(kt, vt, slot, kc, vc)
    del slot
    q = I.synth_normal(seed, I.TID_Q, (R, Hq, d), torch.bfloat16)
    qd, ctx_d = q.to(DEV), ctx.to(DEV)
    outs = []
    for w in range(W):
        op, lp = ra.cp_decode_partials(qd, kc[w:w + 1], vc[w:w + 1], bt, ctx_d, I_, pcp, dcp, dev0=w,
                                       split_blocks=split)
        outs.append(ra.lse_merge(op, lp, out_dtype=torch.float32))
    lse_all = torch.stack([x[1] for x in outs])
    scaled = [ra.cp_lse_rescale(outs[w][0], lse_all, w) for w in range(W)]
    total = torch.stack([s_[0] for s_ in scaled]).sum(0)
    O = torch.cat([total[w] for w in range(W)], dim=1)
    L = torch.cat([s_[1] for s_ in scaled], dim=1)
    check_status(ra)
    o_ref, l_ref = ra.cp_decode(qd, kc, vc, bt, ctx_d, I_, pcp, dcp, split_blocks=split, out_dtype=torch.float32)
    assert (O - o_ref).abs().max().item() <= 1e-5 and (L - l_ref).abs().max().item() <= 1e-5
    tol = TOL[torch.bfloat16]
    for r in (0, 17, 63):
        s0, s1 = int(qsl[r]), int(qsl[r + 1])
        toks = np.arange(s0, s1)          # the oracle's K/V from the host generator
        kr = I.synth_rows(seed, I.TID_K, toks, Hkv * d, torch.bfloat16).reshape(s1 - s0, Hkv, d)
        vr = I.synth_rows(seed, I.TID_V, toks, Hkv * d, torch.bfloat16).reshape(s1 - s0, Hkv, d)
        Or, Lr = oracle.decode_reference(q[r], kr, vr)
        assert np.abs(O[r].cpu().numpy() - Or).max() <= tol["o_max"]
        assert np.abs(L[r].cpu().numpy() - Lr).max() <= tol["lse"]
