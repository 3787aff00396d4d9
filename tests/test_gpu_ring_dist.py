"""The ring step across devices (ra_ring_step_fwd) against the float64 oracle,
alone and driven by the single-process N-rank ring driver, on one GPU."""
import numpy as np
import pytest
import torch

import oracle
from context_long_sequence_ring_gb300 import cp_dist, inputs as I
from tests._gpu import ra_lib, assert_parity, check_status, TOL

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


@pytest.fixture(scope="module")
def ra():
    return ra_lib()


def _local_idx(N, c, r, B=1):
    S = 2 * N * c
    return np.concatenate([b * S + np.concatenate([np.arange(ch * c, ch * c + c) for ch in (r, 2 * N - 1 - r)])
                           for b in range(B)])


def _host_inputs(seed, B, S, Hq, Hkv, d):
    q = I.synth_normal(seed, I.TID_Q, (B * S, Hq, d), torch.bfloat16)
    k = I.synth_normal(seed, I.TID_K, (B * S, Hkv, d), torch.bfloat16)
    v = I.synth_normal(seed, I.TID_V, (B * S, Hkv, d), torch.bfloat16)
    return q, k, v


def _run_rank(ra, q, k, v, N, c, r, B, causal, order):
    """Rank r's steps over the blocks of `order` (its own block first or not): fp32 running result
    in place, the last step into a bf16 output."""
    qi = torch.as_tensor(_local_idx(N, c, r, B))
    ql = q[qi].contiguous().to(DEV)
    o_acc = lse = None
    o_fin = torch.empty(ql.shape, dtype=torch.bfloat16, device=DEV)
    for t, s in enumerate(order):
        si = torch.as_tensor(_local_idx(N, c, s, B))
        kl, vl = k[si].contiguous().to(DEV), v[si].contiguous().to(DEV)
        last = t == len(order) - 1
        if o_acc is None:
            o_acc = torch.empty(ql.shape, dtype=torch.float32, device=DEV)
            lse = torch.empty(ql.shape[:2], dtype=torch.float32, device=DEV)
            ra.ring_step_fwd(ql, kl, vl, N, r, s, causal, None, None, o_fin if last else o_acc, lse, B=B)
        else:
            ra.ring_step_fwd(ql, kl, vl, N, r, s, causal, o_acc, lse, o_fin if last else o_acc, lse, B=B)
    return o_fin, lse, qi.numpy()


def _full_rows(q, k, v, B, S, causal, rows):
    Os, Ls = [], []
    for b in range(B):
        O, L = oracle.full_attention(q[b * S:(b + 1) * S], k[b * S:(b + 1) * S], v[b * S:(b + 1) * S], causal)
        Os.append(O)
        Ls.append(L)
    O, L = np.concatenate(Os), np.concatenate(Ls)
    return O[rows], L[rows]


@pytest.mark.parametrize("N,c,B,Hq,Hkv,d,causal", [
    (2, 256, 1, 4, 2, 128, True),       # whole tiles, head pairs
    (4, 200, 1, 4, 2, 128, True),       # ragged chunks (a 72-row tile)
    (3, 300, 2, 3, 1, 128, True),       # odd group: adjacent tiles, an empty second slot, two sequences
    (4, 128, 1, 8, 8, 64, True),        # d = 64, plain multi-head (adjacent tiles)
    (2, 384, 1, 4, 1, 128, False),      # non-causal
    (8, 16, 1, 2, 2, 128, True),        # tiny chunks inside one tile
    (1, 640, 1, 4, 2, 128, True),       # one rank: the step is the whole attention
])
def test_ring_steps_match_full_attention(ra, N, c, B, Hq, Hkv, d, causal):
    S = 2 * N * c
    q, k, v = _host_inputs(40 + N, B, S, Hq, Hkv, d)
    for r in sorted({0, N // 2, N - 1}):
        o, lse, rows = _run_rank(ra, q, k, v, N, c, r, B, causal, [(r - t) % N for t in range(N)])
        check_status(ra)
        O, L = _full_rows(q, k, v, B, S, causal, rows)
        assert_parity(o, O, lse, L, torch.bfloat16, "rank %d of %d" % (r, N))


@pytest.mark.parametrize("order", ["reverse", "other_first"])
def test_ring_step_order_and_skipped_first_step(ra, order):
    # any order of the blocks reaches the same result; starting on a block the rank's first chunk
    # cannot see leaves those rows at O 0, LSE -inf until a later step fills them in
    N, c, B, Hq, Hkv, d = 4, 256, 1, 4, 2, 128
    S = 2 * N * c
    q, k, v = _host_inputs(48, B, S, Hq, Hkv, d)
    for r in range(N - 1):
        steps = [(r + t) % N for t in range(N)] if order == "reverse" else [(r + 1 + t) % N for t in range(N)]
        o, lse, rows = _run_rank(ra, q, k, v, N, c, r, B, True, steps)
        check_status(ra)
        O, L = _full_rows(q, k, v, B, S, True, rows)
        assert_parity(o, O, lse, L, torch.bfloat16, "rank %d, %s" % (r, order))


@pytest.mark.parametrize("Hq,Hkv,out", [(4, 2, torch.float32), (3, 1, torch.bfloat16)])
def test_ring_step_merges_a_given_running_result(ra, Hq, Hkv, out):
    # one step on a running result that is not the kernel's own (random O, LSE with some -inf rows):
    # the merge epilogue against the oracle's step
    N, c, B, d, r, s = 4, 200, 1, 128, 2, 1
    S = 2 * N * c
    q, k, v = _host_inputs(49, B, S, Hq, Hkv, d)
    g = torch.Generator().manual_seed(50)
    o_in = torch.randn((2 * c, Hq, d), generator=g)
    lse_in = torch.randn((2 * c, Hq), generator=g) * 4
    lse_in[::7, 0] = -float("inf")
    o_in[::7, 0] = 0.0
    qi, si = torch.as_tensor(_local_idx(N, c, r)), torch.as_tensor(_local_idx(N, c, s))
    ql, kl, vl = q[qi].contiguous(), k[si].contiguous(), v[si].contiguous()
    o_out = torch.empty((2 * c, Hq, d), dtype=out, device=DEV)
    lse_out = torch.empty((2 * c, Hq), dtype=torch.float32, device=DEV)
    ra.ring_step_fwd(ql.to(DEV), kl.to(DEV), vl.to(DEV), N, r, s, True, o_in.to(DEV), lse_in.to(DEV), o_out, lse_out)
    check_status(ra)
    O, L = oracle.ring_step(ql, kl, vl, N, r, s, True, o_in.double().numpy(), lse_in.double().numpy())
    fin = np.isfinite(L)
    lo = lse_out.cpu().numpy()
    assert np.array_equal(np.isfinite(lo), fin)
    tol = TOL[torch.bfloat16]
    e = np.abs(o_out.float().cpu().numpy() - O)
    assert e.max() <= tol["o_max"] and e.mean() <= tol["o_mean"], (e.max(), e.mean())
    assert np.abs(lo[fin] - L[fin]).max() <= tol["lse"]


def test_ring_step_rejects_bad_arguments(ra):
    q = torch.zeros((256, 4, 128), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((256, 2, 128), dtype=torch.bfloat16, device=DEV)
    o = torch.zeros((256, 4, 128), dtype=torch.float32, device=DEV)
    lse = torch.zeros((256, 4), dtype=torch.float32, device=DEV)
    with pytest.raises(ra.RingAttnError):
        ra.ring_step_fwd(q, k, k, 2, 2, 0, True)                  # rank outside [0, n_ranks)
    with pytest.raises(ra.RingAttnError):
        ra.ring_step_fwd(q, k, k, 2, 0, 0, True, o, None)          # o_in without lse_in
    # a bf16 output written over the fp32 running output it reads
    st = ra.lib().ra_ring_step_fwd(q.data_ptr(), k.data_ptr(), k.data_ptr(), 1, 4, 2, 128, 128, 2, 0, 1, 1, 0.0,
                                   o.data_ptr(), lse.data_ptr(), o.data_ptr(), ra.RA_BF16, lse.data_ptr(), None)
    assert st == ra.RA_ERR_INVALID_ARG
    check_status(ra)


@pytest.mark.parametrize("N,c,Hq,Hkv", [(4, 384, 8, 2), (3, 200, 6, 2)])
def test_ring_attention_local_driver(ra, N, c, Hq, Hkv):
    # all N ranks in one process: blocks rotate by device copies on a side stream, double-buffered
    d = 128
    S = 2 * N * c
    q, k, v = _host_inputs(51, 1, S, Hq, Hkv, d)
    idx = [torch.as_tensor(_local_idx(N, c, r)) for r in range(N)]
    qs = [q[i].contiguous().to(DEV) for i in idx]
    ks = [k[i].contiguous().to(DEV) for i in idx]
    vs = [v[i].contiguous().to(DEV) for i in idx]
    keep = [x.clone() for x in ks]
    steps = [ra.ring_step_fn(N, r, True) for r in range(N)]
    res = cp_dist.ring_attention_local(qs, ks, vs, step=lambda r, *a: steps[r](*a))
    check_status(ra)
    O, L = oracle.full_attention(q, k, v, True)
    for r in range(N):
        assert_parity(res[r][0], O[idx[r]], res[r][1], L[idx[r]], torch.bfloat16, "rank %d" % r)
        assert torch.equal(ks[r], keep[r])


def test_ring_over_eight_ranks_at_full_size(ra):
    """The S=131072, Hq=32, Hkv=8 prefill as 8 ranks of a ring across devices, emulated in one
    process: every output equals the single-device ring kernel's to the bf16 tolerance, and sampled
    rows equal the oracle's."""
    B, S, Hq, Hkv, d, N, seed = 1, 131072, 32, 8, 128, 8, 5
    tab = I.normal_table(torch.bfloat16)
    q = ra.synth_fill(I.tensor_key(seed, I.TID_Q), tab, (S, Hq, d))
    k = ra.synth_fill(I.tensor_key(seed, I.TID_K), tab, (S, Hkv, d))
    v = ra.synth_fill(I.tensor_key(seed, I.TID_V), tab, (S, Hkv, d))
    o_ref, lse_ref = ra.ring_attn_fwd(q, k, v, True, 16)
    c = S // (2 * N)
    idx = [torch.as_tensor(_local_idx(N, c, r), device=DEV) for r in range(N)]
    steps = [ra.ring_step_fn(N, r, True) for r in range(N)]
    res = cp_dist.ring_attention_local([q[i] for i in idx], [k[i] for i in idx], [v[i] for i in idx],
                                       step=lambda r, *a: steps[r](*a))
    check_status(ra)
    tol = TOL[torch.bfloat16]
    for r in range(N):
        e = (res[r][0].float() - o_ref[idx[r]].float()).abs()
        assert e.max().item() <= tol["o_max"] and e.mean().item() <= tol["o_mean"] / 4, (r, e.max().item())
        assert (res[r][1] - lse_ref[idx[r]]).abs().max().item() <= tol["lse"]
    # sampled rows of ranks 0 and N-1 against the oracle
    rng = np.random.default_rng(57)
    kk = I.synth_rows(seed, I.TID_K, np.arange(S), Hkv * d, torch.bfloat16).reshape(S, Hkv, d).double().numpy()
    vv = I.synth_rows(seed, I.TID_V, np.arange(S), Hkv * d, torch.bfloat16).reshape(S, Hkv, d).double().numpy()
    for r in (0, N - 1):
        loc = np.sort(rng.choice(2 * c, 24, replace=False))
        rows = idx[r].cpu().numpy()[loc]
        qr = I.synth_rows(seed, I.TID_Q, rows, Hq * d, torch.bfloat16).reshape(len(rows), Hq, d)
        O, L = oracle.attention_rows(qr, rows, kk[:rows.max() + 1], vv[:rows.max() + 1], True)
        sel = torch.as_tensor(loc, device=DEV)
        assert_parity(res[r][0][sel], O, res[r][1][sel], L, torch.bfloat16, "rank %d sampled rows" % r)


@pytest.mark.parametrize("N,c,Hq,Hkv,causal,seg", [(4, 256, 4, 2, True, 512), (3, 200, 3, 1, True, 4096),
                                                   (2, 384, 4, 4, False, 700)])
def test_allgather_kv_prefill_emulated(ra, N, c, Hq, Hkv, causal, seg):
    # each rank's K/V all-gathered (emulated by concatenation, which is the gathered order), put back
    # in token order by the row-gather kernel with the partition's restore index, then the rank's two
    # chunks attend over the keys in token order in segments of `seg` keys
    d = 128
    S = 2 * N * c
    q, k, v = _host_inputs(53, 1, S, Hq, Hkv, d)
    perm, restore = ra.zigzag_partition([S], N)
    idx = [torch.as_tensor(_local_idx(N, c, r)) for r in range(N)]
    k_all = torch.cat([k[i] for i in idx]).to(DEV)
    v_all = torch.cat([v[i] for i in idx]).to(DEV)
    k_nat, v_nat = ra.gather_rows(k_all, restore), ra.gather_rows(v_all, restore)
    assert torch.equal(k_nat.cpu(), k)
    O, L = oracle.full_attention(q, k, v, causal)
    for r in range(N):
        ql = q[idx[r]].contiguous().to(DEV)
        o = torch.empty(ql.shape, dtype=torch.bfloat16, device=DEV)
        lse = torch.empty(ql.shape[:2], dtype=torch.float32, device=DEV)
        ra.allgather_attend_fn(S, N, r, causal, seg_tokens=seg)(ql, k_nat, v_nat, o, lse)
        check_status(ra)
        assert_parity(o, O[idx[r]], lse, L[idx[r]], torch.bfloat16, "rank %d" % r)


def test_allgather_kv_prefill_at_full_size(ra):
    """The S=131072, Hq=32, Hkv=8 prefill in the all-gather form over 8 emulated ranks (32768-key
    segments): every output of ranks 0, 3 and 7 equals the single-device ring kernel's to the bf16
    tolerance."""
    S, Hq, Hkv, d, N, seed = 131072, 32, 8, 128, 8, 5
    tab = I.normal_table(torch.bfloat16)
    q = ra.synth_fill(I.tensor_key(seed, I.TID_Q), tab, (S, Hq, d))
    k = ra.synth_fill(I.tensor_key(seed, I.TID_K), tab, (S, Hkv, d))
    v = ra.synth_fill(I.tensor_key(seed, I.TID_V), tab, (S, Hkv, d))
    o_ref, lse_ref = ra.ring_attn_fwd(q, k, v, True, 16)
    perm, restore = ra.zigzag_partition([S], N)
    kz, vz = ra.gather_rows(k, perm), ra.gather_rows(v, perm)          # what the all-gather delivers
    k_nat, v_nat = ra.gather_rows(kz, restore), ra.gather_rows(vz, restore)
    assert torch.equal(k_nat, k) and torch.equal(v_nat, v)
    c = S // (2 * N)
    tol = TOL[torch.bfloat16]
    for r in (0, 3, N - 1):
        rows = perm[r * 2 * c:(r + 1) * 2 * c]
        ql = ra.gather_rows(q, rows)
        o = torch.empty(ql.shape, dtype=torch.bfloat16, device=DEV)
        lse = torch.empty(ql.shape[:2], dtype=torch.float32, device=DEV)
        ra.allgather_attend_fn(S, N, r, True)(ql, k_nat, v_nat, o, lse)
        check_status(ra)
        ro, rl = o_ref[rows.long()], lse_ref[rows.long()]
        e = (o.float() - ro.float()).abs()
        assert e.max().item() <= tol["o_max"] and e.mean().item() <= tol["o_mean"] / 4, (r, e.max().item())
        assert (lse - rl).abs().max().item() <= tol["lse"]
