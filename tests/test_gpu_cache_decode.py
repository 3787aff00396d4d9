"""GPU parity of the zigzag partition, row gathers, LSE merge, CP slot mapping,
KV scatter and split-KV decode (C ABI) against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from context_long_sequence_ring_gb300 import inputs as I
from tests._gpu import ra_lib, assert_parity, check_status
from tests._golden import load

pytestmark = [pytest.mark.gpu, pytest.mark.filterwarnings("ignore::RuntimeWarning")]
DEV = torch.device("cuda")


@pytest.fixture(scope="module")
def ra():
    return ra_lib()


# --------------------------------------------------------------------- partition

@pytest.mark.parametrize("case", load("zigzag_hand.json")["cases"], ids=lambda c: c["name"])
def test_zigzag_hand_worked(ra, case):
    perm, restore = ra.zigzag_partition(case["seq_lens"], case["n_ranks"])
    check_status(ra)
    assert perm.cpu().tolist() == case["perm"]
    assert restore.cpu().tolist() == case["restore"]


@pytest.mark.parametrize("lens,N", [([32768, 32768], 8), ([131072], 16), ([0, 5, 1, 1000, 77], 3),
                                    (list(range(1, 600, 7)), 4)])
def test_zigzag_bit_exact_and_round_trip(ra, lens, N):
    perm, restore = ra.zigzag_partition(lens, N)
    check_status(ra)
    p_ref, r_ref, _ = oracle.zigzag_partition(lens, N)
    assert np.array_equal(perm.cpu().numpy(), p_ref)
    assert np.array_equal(restore.cpu().numpy(), r_ref)
    x = torch.randn((sum(lens), 3, 8), device=DEV).to(torch.bfloat16)
    g = ra.gather_rows(x, perm)
    assert torch.equal(g[perm < 0], torch.zeros_like(g[perm < 0]))
    assert torch.equal(ra.gather_rows(g, restore), x)
    check_status(ra)


def test_zigzag_many_requests_spans_parameter_batches(ra):
    lens = [int(x) for x in np.random.default_rng(3).integers(0, 50, size=700)]
    perm, restore = ra.zigzag_partition(lens, 2)
    p_ref, r_ref, _ = oracle.zigzag_partition(lens, 2)
    assert np.array_equal(perm.cpu().numpy(), p_ref) and np.array_equal(restore.cpu().numpy(), r_ref)


def test_gather_odd_row_sizes(ra):
    x = torch.arange(7 * 5, dtype=torch.uint8, device=DEV).reshape(7, 5)
    idx = torch.tensor([6, -1, 0, 3], dtype=torch.int32, device=DEV)
    y = ra.gather_rows(x, idx)
    ref = oracle.gather_rows(x.cpu().numpy(), idx.cpu().numpy())
    assert np.array_equal(y.cpu().numpy(), ref)


def test_gather_out_of_range_index_is_reported(ra):
    x = torch.ones((4, 4), dtype=torch.float32, device=DEV)
    idx = torch.tensor([0, 9], dtype=torch.int32, device=DEV)
    y = ra.gather_rows(x, idx)
    assert ra.device_status() == ra.RA_ERR_DEVICE_BOUNDS
    assert torch.equal(y[1].cpu(), torch.zeros(4))


# --------------------------------------------------------------------- merge

@pytest.mark.parametrize("P,T,H,d", [(1, 5, 3, 8), (3, 17, 4, 128), (64, 64, 32, 128), (8, 2, 2, 64),
                                     (8, 300, 8, 128), (9, 40, 4, 128), (1, 33, 2, 128)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_lse_merge(ra, P, T, H, d, out_dtype):
    g = torch.Generator().manual_seed(P * 1000 + T)
    o = torch.randn((P, T, H, d), generator=g)
    lse = torch.randn((P, T, H), generator=g) * 3
    lse[torch.rand((P, T, H), generator=g) < 0.3] = -float("inf")
    lse[0, 0, 0] = -float("inf")
    if P > 1:
        lse[:, 1, 0] = -float("inf")                     # an all-empty row
        o[:, 1, 0] = float("nan")                        # never read
    om, lm = ra.lse_merge(o.to(DEV), lse.to(DEV), out_dtype)
    check_status(ra)
    O, L = oracle.lse_merge(o.numpy(), lse.numpy())
    e = np.abs(om.float().cpu().numpy() - O)
    assert e.max() <= (2e-2 if out_dtype == torch.bfloat16 else 1e-5)
    lg = lm.cpu().numpy()
    assert np.array_equal(np.isinf(lg), np.isinf(L))
    fin = np.isfinite(L)
    assert np.abs(lg[fin] - L[fin]).max(initial=0) <= 1e-5


@pytest.mark.parametrize("case", load("merge_hand.json")["cases"], ids=lambda c: c["name"])
def test_lse_merge_hand_worked(ra, case):
    from tests._golden import arr
    o = torch.tensor(arr(case["o"]), dtype=torch.float32)         # [P, T=1, d] -> add H
    lse = torch.tensor(arr(case["lse"]), dtype=torch.float32)
    P, T, d = o.shape
    o4 = o.reshape(P, T, 1, d)
    if d % 4:
        o4 = torch.nn.functional.pad(o4, (0, 4 - d % 4))
    om, lm = ra.lse_merge(o4.to(DEV).contiguous(), lse.reshape(P, T, 1).to(DEV).contiguous())
    np.testing.assert_allclose(om[..., :d].reshape(T, d).cpu().numpy(), arr(case["O"]), atol=1e-6)
    np.testing.assert_allclose(lm.reshape(T).cpu().numpy(), arr(case["LSE"]), atol=1e-6)


# --------------------------------------------------------------------- slot mapping

def test_slot_mapping_hand_worked(ra):
    g = load("slot_mapping_hand.json")
    ex = g["slot_example"]
    t = lambda x: torch.tensor(x, dtype=torch.int32, device=DEV)
    slot = ra.cp_slot_mapping(t(ex["query_start_loc"]), t(ex["positions"]), t(ex["block_table"]),
                              g["block_size"], g["interleave"], g["pcp"], g["dcp"])
    check_status(ra)
    assert slot.cpu().tolist() == ex["slot"]
    with pytest.raises(ra.RingAttnError):
        ra.cp_slot_mapping(t(ex["query_start_loc"]), t(ex["positions"]), t(ex["block_table"]), 100, 16, 2, 4)


@pytest.mark.parametrize("bs,I_,pcp,dcp", [(128, 16, 2, 4), (16, 4, 1, 2), (8, 8, 3, 1), (32, 16, 2, 2)])
def test_slot_mapping_bit_exact_random(ra, bs, I_, pcp, dcp):
    wl = I.decode_workload(bs + I_, 9, 1, 3000, bs, pcp, dcp)
    ctx = wl["ctx_lens"]
    qsl = torch.zeros(len(ctx) + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(ctx, 0)
    pos = torch.cat([torch.arange(int(L), dtype=torch.int32) for L in ctx])
    slot = ra.cp_slot_mapping(qsl.to(DEV), pos.to(DEV), wl["block_table"].to(DEV), bs, I_, pcp, dcp)
    check_status(ra)
    ref = oracle.cp_slot_mapping(qsl.numpy(), pos.numpy(), wl["block_table"].numpy(), bs, I_, pcp, dcp)
    assert np.array_equal(slot.cpu().numpy().astype(np.int64), ref)


# --------------------------------------------------------------------- decode

def _decode_case(ra, seed, R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d, split):
    W = pcp * dcp
    wl = I.decode_workload(seed, R, lo, hi, bs, pcp, dcp)
    T = wl["total_tokens"]
    kt = I.synth_normal(seed, I.TID_K, (T, Hkv, d), torch.bfloat16)
    vt = I.synth_normal(seed, I.TID_V, (T, Hkv, d), torch.bfloat16)
    qd = I.synth_normal(seed, I.TID_Q, (R, Hq, d), torch.bfloat16)
    ctx = wl["ctx_lens"]
    qsl = torch.zeros(R + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(ctx, 0)
    pos = torch.cat([torch.arange(int(L), dtype=torch.int32) for L in ctx])
    slot = ra.cp_slot_mapping(qsl.to(DEV), pos.to(DEV), wl["block_table"].to(DEV), bs, I_, pcp, dcp)
    # unwritten cache slots hold NaN: the decode must never read them
    kc = torch.full((W, wl["num_blocks"], Hkv, bs, d), float("nan"), dtype=torch.bfloat16, device=DEV)
    vc = torch.full_like(kc, float("nan"))
    ra.cp_kv_scatter(kt.to(DEV), vt.to(DEV), slot, kc, vc)
    o, lse = ra.cp_decode(qd.to(DEV), kc, vc, wl["block_table"].to(DEV), ctx.to(DEV), I_, pcp, dcp,
                          split_blocks=split)
    check_status(ra)
    return wl, kt, vt, qd, qsl, slot, kc, vc, o, lse


@pytest.mark.parametrize("R,lo,hi,bs,I_,pcp,dcp,Hq,Hkv,d,split", [
    (3, 1, 700, 32, 16, 2, 2, 4, 2, 128, 2),
    (4, 100, 3000, 128, 16, 2, 4, 32, 8, 128, 1),
    (2, 1, 1, 16, 8, 1, 1, 8, 1, 64, 1),           # single-token contexts, GQA group 8
    (3, 200, 2600, 64, 64, 1, 2, 2, 2, 64, 3),     # group 1, interleave = block size
    (5, 512, 512, 64, 16, 2, 2, 16, 4, 128, 100),  # exactly full virtual blocks, one split
])
def test_decode_matches_oracle(ra, R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d, split):
    wl, kt, vt, qd, qsl, slot, kc, vc, o, lse = _decode_case(ra, 4, R, lo, hi, bs, I_, pcp, dcp, Hq, Hkv, d, split)
    for r in range(R):
        s0, s1 = int(qsl[r]), int(qsl[r + 1])
        O, L = oracle.decode_reference(qd[r], kt[s0:s1], vt[s0:s1])
        assert_parity(o[r], O, lse[r], L, torch.bfloat16, "decode request %d" % r)
    # the oracle's own sharded decode, reading the oracle-filled cache, agrees too
    W = pcp * dcp
    kc_np = np.zeros((W, wl["num_blocks"], Hkv, bs, d))
    vc_np = np.zeros_like(kc_np)
    pos = np.concatenate([np.arange(int(L)) for L in wl["ctx_lens"]])
    oslot = oracle.cp_slot_mapping(qsl.numpy(), pos, wl["block_table"].numpy(), bs, I_, pcp, dcp)
    oracle.cp_kv_scatter(kt.double().numpy(), vt.double().numpy(), oslot, kc_np, vc_np, bs)
    O2, L2 = oracle.cp_decode(qd, kc_np, vc_np, wl["block_table"].numpy(), wl["ctx_lens"].numpy(), bs, I_,
                              pcp, dcp, split)
    assert_parity(o, O2, lse, L2, torch.bfloat16, "decode vs sharded oracle")


def test_scatter_places_rows_bit_exact(ra):
    wl, kt, vt, qd, qsl, slot, kc, vc, o, lse = _decode_case(ra, 8, 3, 10, 900, 32, 8, 2, 2, 4, 2, 128, 2)
    s = slot.cpu().numpy()
    kcc = kc.cpu()
    for w in range(s.shape[0]):
        ts = np.nonzero(s[w] >= 0)[0]
        sl = s[w, ts]
        got = kcc[w, sl // 32, :, sl % 32, :]
        assert torch.equal(got, kt[ts])


@pytest.mark.parametrize("split", [16, 8])
def test_decode_full_size_sampled_requests(ra, split):
    """64 requests, context U[4096, 131072], Hq=32, Hkv=8, d=128, block 128, interleave 16, pcp=2, dcp=4:
    full-size slot mapping (bit-exact) + scatter + split-KV decode + merge; sampled requests vs the oracle.
    Split 16 is the bench's launch configuration."""
    seed, R, bs, I_, pcp, dcp, Hq, Hkv, d = 4, 64, 128, 16, 2, 4, 32, 8, 128
    W = pcp * dcp
    wl = I.decode_workload(seed, R, 4096, 131072, bs, pcp, dcp)
    T = wl["total_tokens"]
    tab = I.normal_table(torch.bfloat16)
    kt = ra.synth_fill(I.tensor_key(seed, I.TID_K), tab, (T, Hkv, d))
    vt = ra.synth_fill(I.tensor_key(seed, I.TID_V), tab, (T, Hkv, d))
    qd = I.synth_normal(seed, I.TID_Q, (R, Hq, d), torch.bfloat16)
    ctx = wl["ctx_lens"]
    qsl = torch.zeros(R + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(ctx, 0)
    pos = torch.cat([torch.arange(int(L), dtype=torch.int32) for L in ctx])
    slot = ra.cp_slot_mapping(qsl.to(DEV), pos.to(DEV), wl["block_table"].to(DEV), bs, I_, pcp, dcp)
    check_status(ra)
    ref = oracle.cp_slot_mapping(qsl.numpy(), pos.numpy(), wl["block_table"].numpy(), bs, I_, pcp, dcp)
    assert np.array_equal(slot.cpu().numpy().astype(np.int64), ref)
    del ref
    kc = torch.empty((W, wl["num_blocks"], Hkv, bs, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.empty_like(kc)
    ra.cp_kv_scatter(kt, vt, slot, kc, vc)
    del kt, vt
    o, lse = ra.cp_decode(qd.to(DEV), kc, vc, wl["block_table"].to(DEV), ctx.to(DEV), I_, pcp, dcp, split_blocks=split)
    check_status(ra)
    Ls = ctx.numpy()
    for r in sorted({int(np.argmin(Ls)), int(np.argmax(Ls)), 17}):
        s0, s1 = int(qsl[r]), int(qsl[r + 1])
        rows = np.arange(s0, s1)
        kr = I.synth_rows(seed, I.TID_K, rows, Hkv * d, torch.bfloat16).reshape(-1, Hkv, d)
        vr = I.synth_rows(seed, I.TID_V, rows, Hkv * d, torch.bfloat16).reshape(-1, Hkv, d)
        O, L = oracle.decode_reference(qd[r], kr, vr)
        assert_parity(o[r], O, lse[r], L, torch.bfloat16, "full-size decode request %d" % r)


# --------------------------------------------------------------------- cache reorg (gather)

def test_kv_gather_round_trip_and_oracle(ra):
    """Scatter into the sharded cache, gather back in token order: bit-exact, and equal to the
    oracle's gather from the same cache; a reversed order works too."""
    wl, kt, vt, qd, qsl, slot, kc, vc, o, lse = _decode_case(ra, 9, 3, 10, 900, 32, 8, 2, 2, 4, 2, 128, 2)
    ctx = wl["ctx_lens"]
    pos = torch.cat([torch.arange(int(L), dtype=torch.int32) for L in ctx])
    k2, v2 = ra.cp_kv_gather(kc, vc, wl["block_table"].to(DEV), qsl.to(DEV), pos.to(DEV), 8, 2, 2)
    check_status(ra)
    assert torch.equal(k2.cpu(), kt) and torch.equal(v2.cpu(), vt)
    n = int(ctx[1])
    q2 = torch.tensor([0, 0, n, n], dtype=torch.int32)
    p2 = torch.arange(n - 1, -1, -1, dtype=torch.int32)
    k3, v3 = ra.cp_kv_gather(kc, vc, wl["block_table"].to(DEV), q2.to(DEV), p2.to(DEV), 8, 2, 2)
    kr, vr = oracle.cp_kv_gather(kc.float().cpu().numpy(), vc.float().cpu().numpy(), wl["block_table"].numpy(),
                                 q2.numpy(), p2.numpy(), 32, 8, 2, 2)
    assert np.array_equal(k3.float().cpu().numpy(), kr) and np.array_equal(v3.float().cpu().numpy(), vr)


def test_kv_gather_bad_block_is_reported(ra):
    kc = torch.zeros((2, 3, 1, 16, 64), dtype=torch.bfloat16, device=DEV)
    bt = torch.tensor([[0, 7]], dtype=torch.int32, device=DEV)      # block 7 does not exist
    qsl = torch.tensor([0, 2], dtype=torch.int32, device=DEV)
    pos = torch.tensor([0, 40], dtype=torch.int32, device=DEV)      # token 40 is in virtual block 1
    k, v = ra.cp_kv_gather(kc, kc, bt, qsl, pos, 8, 2, 1)
    assert ra.device_status() == ra.RA_ERR_DEVICE_BOUNDS
    assert torch.equal(k[1].cpu(), torch.zeros_like(k[1].cpu()))


def test_empty_inputs_launch_nothing(ra):
    """Zero tokens / rows are valid and leave the outputs untouched."""
    z32 = torch.zeros(0, dtype=torch.int32, device=DEV)
    out = torch.zeros((8, 0), dtype=torch.int32, device=DEV)
    ra.cp_slot_mapping(torch.zeros(2, dtype=torch.int32, device=DEV), z32,
                       torch.zeros((1, 1), dtype=torch.int32, device=DEV), 128, 16, 2, 4, out=out)
    kc = torch.zeros((8, 1, 1, 128, 128), dtype=torch.bfloat16, device=DEV)
    kz = torch.zeros((0, 1, 128), dtype=torch.bfloat16, device=DEV)
    ra.cp_kv_scatter(kz, kz, torch.zeros((8, 0), dtype=torch.int32, device=DEV), kc, kc)
    y = ra.gather_rows(torch.ones((4, 3), device=DEV), z32)
    assert y.shape == (0, 3)
    perm, restore = ra.zigzag_partition([0, 0], 4)
    assert perm.numel() == 0 and restore.numel() == 0
    check_status(ra)
