"""The host side of context parallelism across ranks, on the CPU: the ring
schedule, the ring of K/V blocks over gloo ranks (2 and 4 processes) and the
decode's cp_lse_ag_out_rs collective.  The arithmetic of a step is a stand-in
passed in by the test and written with the float64 oracle, so these tests pin
the orchestration: which block each rank holds at every step, that the
exchanged buffers arrive intact, and that the merged result equals full
attention."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from context_long_sequence_ring_gb300 import cp_dist

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _local_idx(N, c, r, B=1):
    S = 2 * N * c
    return np.concatenate([b * S + np.concatenate([np.arange(ch * c, ch * c + c) for ch in (r, 2 * N - 1 - r)])
                           for b in range(B)])


def _inputs(seed, B, S, Hq, Hkv, d):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B * S, Hq, d), generator=g, dtype=torch.float64)
    k = torch.randn((B * S, Hkv, d), generator=g, dtype=torch.float64)
    v = torch.randn((B * S, Hkv, d), generator=g, dtype=torch.float64)
    return q, k, v


def _oracle_step(N, r, causal, B):
    """Stand-in for the ring-step kernel: the oracle's step, written into the driver's buffers."""
    def step(q, kh, vh, src, o_in, lse_in, o_out, lse_out):
        O, L = oracle.ring_step(q, kh, vh, N, r, src, causal,
                                None if o_in is None else o_in.double().numpy(),
                                None if lse_in is None else lse_in.double().numpy(), B=B)
        o_out.copy_(torch.from_numpy(O))
        lse_out.copy_(torch.from_numpy(L))
    return step


# ---------------------------------------------------------------- schedule

@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
def test_ring_schedule(N):
    for r in range(N):
        sch = cp_dist.ring_schedule(N, r)
        assert [s.t for s in sch] == list(range(N))
        assert [s.src for s in sch] == [(r - t) % N for t in range(N)]   # rank (r - t) mod N at step t
        assert sorted(s.src for s in sch) == list(range(N))              # every block exactly once
        assert all(s.send_to == (r + 1) % N and s.recv_from == (r - 1) % N for s in sch)
        assert [s.exchange for s in sch] == [t + 1 < N for t in range(N)]
        for t in range(N - 1):
            assert sch[t].recv_src == sch[t + 1].src                      # what arrives is held next
            # what rank r-1 sends at step t is the block rank r receives
            assert cp_dist.ring_schedule(N, (r - 1) % N)[t].src == sch[t].recv_src


def test_ring_schedule_rejects_bad_rank():
    with pytest.raises(ValueError):
        cp_dist.ring_schedule(4, 4)
    with pytest.raises(ValueError):
        cp_dist.ring_schedule(0, 0)


def test_buffer_slots_never_receive_into_the_held_or_callers_buffers():
    for t in range(12):
        assert cp_dist._recv_slot(t) != cp_dist._held_slot(t)
        assert cp_dist._recv_slot(t) != 0                      # the caller's K/V are only read
        assert cp_dist._held_slot(t + 1) == cp_dist._recv_slot(t)


# ---------------------------------------------------------------- ring over gloo ranks

def _ring_worker(rank, world, port, causal, B, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        N, c, Hq, Hkv, d = world, 3, 4, 2, 8
        S = 2 * N * c
        q, k, v = _inputs(5, B, S, Hq, Hkv, d)
        idx = torch.as_tensor(_local_idx(N, c, rank, B))
        ql, kl, vl = q[idx].contiguous(), k[idx].contiguous(), v[idx].contiguous()
        k_keep = kl.clone()
        trace = []
        ex = cp_dist.P2PExchange()
        o, lse = cp_dist.ring_attention(ql, kl, vl, step=_oracle_step(N, rank, causal, B), exchange=ex, trace=trace)
        held_ok = all(src == (rank - t) % N and torch.equal(kh, k[torch.as_tensor(_local_idx(N, c, src, B))])
                      for t, src, kh in trace)
        errs = []
        for b in range(B):
            Of, Lf = oracle.full_attention(q[b * S:(b + 1) * S], k[b * S:(b + 1) * S], v[b * S:(b + 1) * S], causal)
            rows = _local_idx(N, c, rank, 1)
            sel = slice(b * 2 * c, (b + 1) * 2 * c)
            errs.append(max(np.abs(o[sel].numpy() - Of[rows]).max(), np.abs(lse[sel].numpy() - Lf[rows]).max()))
        out[rank] = dict(steps=len(trace), held_ok=held_ok, err=float(max(errs)), input_kept=torch.equal(kl, k_keep))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,causal,B", [(2, True, 1), (4, True, 2), (4, False, 1)])
def test_ring_attention_over_gloo_ranks(world, causal, B):
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_ring_worker, args=(world, _free_port(), causal, B, out), nprocs=world, start_method="spawn")
    assert sorted(out.keys()) == list(range(world))
    for r in range(world):
        assert out[r]["steps"] == world
        assert out[r]["held_ok"], "rank %d held the wrong block at some step" % r
        assert out[r]["input_kept"], "rank %d's own K/V were overwritten" % r
        assert out[r]["err"] < 1e-5, "rank %d: error %g against full attention" % (r, out[r]["err"])


def test_one_rank_ring_needs_no_exchange():
    q, k, v = _inputs(6, 1, 8, 2, 1, 4)
    o, lse = cp_dist.ring_attention(q, k, v, step=_oracle_step(1, 0, True, 1))
    Of, Lf = oracle.full_attention(q, k, v, True)
    np.testing.assert_allclose(o.numpy(), Of, atol=1e-12)
    np.testing.assert_allclose(lse.numpy(), Lf, atol=1e-6)
    with pytest.raises(ValueError):
        cp_dist.ring_attention(q, k, v, step=_oracle_step(1, 0, True, 1), n_ranks=2, rank=0)


@pytest.mark.parametrize("N,causal", [(3, True), (4, False), (2, True)])
def test_ring_attention_local_matches_full(N, causal):
    c, Hq, Hkv, d = 2, 2, 1, 4
    S = 2 * N * c
    q, k, v = _inputs(7, 1, S, Hq, Hkv, d)
    idx = [torch.as_tensor(_local_idx(N, c, r)) for r in range(N)]
    ks = [k[i].contiguous() for i in idx]
    keep = [x.clone() for x in ks]

    def step(r, ql, kh, vh, src, o_in, lse_in, o_out, lse_out):
        assert torch.equal(kh, k[idx[src]])
        _oracle_step(N, r, causal, 1)(ql, kh, vh, src, o_in, lse_in, o_out, lse_out)
    res = cp_dist.ring_attention_local([q[i].contiguous() for i in idx], ks, [v[i].contiguous() for i in idx],
                                       step=step)
    Of, Lf = oracle.full_attention(q, k, v, causal)
    for r in range(N):
        np.testing.assert_allclose(res[r][0].numpy(), Of[idx[r]], atol=1e-6)
        np.testing.assert_allclose(res[r][1].numpy(), Lf[idx[r]], atol=1e-5)
        assert torch.equal(ks[r], keep[r])


def _dropout_worker(rank, world, port, out):
    # rank 1 initialises and then never joins the ring: rank 0 must get an error, not a hang
    import datetime
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=20))
    if rank == 1:
        out[rank] = "left"
        return
    N, c = world, 2
    q, k, v = _inputs(8, 1, 2 * N * c, 2, 1, 4)
    idx = torch.as_tensor(_local_idx(N, c, rank))
    ex = cp_dist.P2PExchange(timeout=datetime.timedelta(seconds=3))
    try:
        cp_dist.ring_attention(q[idx].contiguous(), k[idx].contiguous(), v[idx].contiguous(),
                               step=_oracle_step(N, rank, True, 1), exchange=ex)
        out[rank] = "finished"
    except RuntimeError as e:
        out[rank] = "error: " + str(e)[:80]


def test_ring_detects_a_rank_that_never_joins():
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_dropout_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
    assert out[1] == "left"
    assert out[0].startswith("error"), out[0]


# ---------------------------------------------------------------- decode merge over gloo ranks

def _oracle_rescale(o_local, lse_all, w, o_scaled, lse_total):
    """Stand-in for the rescale kernel, from the oracle's merge: O_w e^{LSE_w - LSE} per head,
    placed in the slot of the rank that keeps the head, and the merged LSE of rank w's heads."""
    W, R, Hq = lse_all.shape
    hs = Hq // W
    la = lse_all.double().numpy()
    _, LSE = oracle.lse_merge(np.zeros(la.shape + (1,)), la)
    live = np.isfinite(la[w]) & np.isfinite(LSE)
    wgt = np.where(live, np.exp(la[w] - np.where(np.isfinite(LSE), LSE, 0.0)), 0.0)
    o = np.where(live[..., None], o_local.double().numpy(), 0.0) * wgt[..., None]
    o_scaled.copy_(torch.from_numpy(o.reshape(R, W, hs, -1).transpose(1, 0, 2, 3).copy()))
    lse_total.copy_(torch.from_numpy(LSE[:, w * hs:(w + 1) * hs].copy()))


def _decode_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        g = torch.Generator().manual_seed(11)
        R, Hq, d = 3, 8, 6
        o_all = torch.randn((world, R, Hq, d), generator=g, dtype=torch.float64)
        l_all = torch.randn((world, R, Hq), generator=g, dtype=torch.float64) * 3
        l_all[0, 1, 3] = -np.inf                          # rank 0 stores no key of (request 1, head 3)
        l_all[:, 2, 7] = -np.inf                          # nobody does: O 0, LSE -inf
        o, lse = cp_dist.cp_lse_ag_out_rs(o_all[rank].float(), l_all[rank].float(), rescale=_oracle_rescale)
        ref = oracle.cp_lse_ag_out_rs(list(o_all.numpy()), list(l_all.numpy()))[rank]
        lse_np = lse.numpy()
        fin = np.isfinite(ref[1])
        out[rank] = dict(shape=tuple(o.shape), o_err=float(np.abs(o.numpy() - ref[0]).max()),
                         lse_err=float(np.abs(lse_np[fin] - ref[1][fin]).max()),
                         inf_ok=bool(np.array_equal(np.isinf(lse_np), ~fin)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_cp_lse_ag_out_rs_over_gloo_ranks(world):
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_decode_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for r in range(world):
        assert out[r]["shape"] == (3, 8 // world, 6)
        assert out[r]["o_err"] < 1e-5 and out[r]["lse_err"] < 1e-5, out[r]
        assert out[r]["inf_ok"], out[r]


# ---------------------------------------------------------------- prefill with the K/V all-gathered

def _allgather_worker(rank, world, port, causal, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        N, c, Hq, Hkv, d = world, 3, 4, 2, 8
        S = 2 * N * c
        q, k, v = _inputs(9, 1, S, Hq, Hkv, d)
        idx = torch.as_tensor(_local_idx(N, c, rank))
        _, restore, _ = oracle.zigzag_partition([S], N)
        got = {}

        def gather(src, idx_, dst):                      # stand-in for the row-gather kernel
            dst.copy_(src[idx_.long()])

        def attend(ql, k_nat, v_nat, o, lse):           # stand-in for the attention kernel
            got["k_nat"] = k_nat.clone()
            O, L = oracle.attention_rows(ql, idx.numpy(), k_nat, v_nat, causal)
            o.copy_(torch.from_numpy(O))
            lse.copy_(torch.from_numpy(L))
        o, lse = cp_dist.allgather_kv_attention(q[idx].contiguous(), k[idx].contiguous(), v[idx].contiguous(),
                                                restore=torch.as_tensor(restore), gather=gather, attend=attend)
        Of, Lf = oracle.full_attention(q, k, v, causal)
        out[rank] = dict(k_restored=torch.equal(got["k_nat"], k), o_err=float(np.abs(o.numpy() - Of[idx]).max()),
                         lse_err=float(np.abs(lse.numpy() - Lf[idx]).max()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,causal", [(2, True), (4, True), (3, False)])
def test_allgather_kv_prefill_over_gloo_ranks(world, causal):
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_allgather_worker, args=(world, _free_port(), causal, out), nprocs=world, start_method="spawn")
    for r in range(world):
        assert out[r]["k_restored"], "rank %d: gathered K not back in token order" % r
        assert out[r]["o_err"] < 1e-12 and out[r]["lse_err"] < 1e-6, out[r]    # O in q's float64, LSE fp32


# ---------------------------------------------------------------- decode merge by all-to-all

def _oracle_split(o_local, lse_local, W, o_split, lse_split):
    """Stand-in for the head-split kernel: heads of rank v into slot v."""
    R, Hq, d = o_local.shape
    hs = Hq // W
    o_split.copy_(o_local.reshape(R, W, hs, d).permute(1, 0, 2, 3))
    lse_split.copy_(lse_local.reshape(R, W, hs).permute(1, 0, 2))


def _oracle_merge(o_parts, lse_parts, o, lse):
    O, L = oracle.lse_merge(o_parts.double().numpy(), lse_parts.double().numpy())
    o.copy_(torch.from_numpy(O))
    lse.copy_(torch.from_numpy(L))


def _a2a_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        g = torch.Generator().manual_seed(12)
        R, Hq, d = 3, 8, 6
        o_all = torch.randn((world, R, Hq, d), generator=g, dtype=torch.float64)
        l_all = torch.randn((world, R, Hq), generator=g, dtype=torch.float64) * 3
        l_all[0, 1, 3] = -np.inf
        o, lse = cp_dist.cp_lse_a2a(o_all[rank].float(), l_all[rank].float(), split=_oracle_split,
                                    merge=_oracle_merge)
        ref = oracle.cp_lse_ag_out_rs(list(o_all.numpy()), list(l_all.numpy()))[rank]
        out[rank] = dict(o_err=float(np.abs(o.numpy() - ref[0]).max()), lse_err=float(np.abs(lse.numpy() - ref[1]).max()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_cp_lse_a2a_equals_ag_out_rs_over_gloo_ranks(world):
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_a2a_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for r in range(world):
        assert out[r]["o_err"] < 1e-5 and out[r]["lse_err"] < 1e-5, out[r]
