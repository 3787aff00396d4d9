"""Context parallelism across ranks: the ring of K/V blocks for prefill and the
cp_lse_ag_out_rs merge for decode, driven over torch.distributed.

Sources, by page title and section:
* "Parallelism-CP" diagram: Q/K/V are cut along the sequence across cards,
  K/V rotate on a ring, each card computes its own Q against every K/V block;
  each card stores 1/N of the activations and the K/V rotation overlaps the
  local attention compute.
* guijiagi.com tag page "Ring Attention", article on the distributed challenge
  of long contexts, ring topology: at step t rank i works on the block of rank
  (i - t) mod N and passes what it holds to rank i + 1.
* vLLM-Ascend developer guide "Context Parallel (CP)": the head-tail partition
  (rank r holds chunks r and 2N-1-r) and the DCP decode, whose partial outputs
  are merged by cp_lse_ag_out_rs (all-gather of the LSEs, a local rescale, a
  reduce-scatter of the outputs over heads).

This module only orders work and moves buffers.  Every step of the arithmetic
runs in the library's kernels, which callers pass in as ``step`` (a ring step)
and ``rescale`` (the decode's local rescale); the bindings in ``ringattn``
(``ring_step_fwd``, ``cp_lse_rescale``) are those kernels.  The movement is
torch.distributed point-to-point and collective calls (NCCL between GPUs, gloo
between CPU processes); no kernel here reads another device's memory.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence

import torch
import torch.distributed as dist


# ---------------------------------------------------------------------- schedule

@dataclass(frozen=True)
class RingStep:
    """What rank ``rank`` of an N-rank ring does at step ``t``."""
    t: int
    src: int          # owner of the K/V block held (and computed on) at this step: (rank - t) mod N
    send_to: int      # the held block goes to rank + 1 ...
    recv_from: int    # ... while the block of rank - 1 arrives
    recv_src: int     # owner of the arriving block, held at step t + 1: (rank - t - 1) mod N
    exchange: bool    # False at the last step: nothing is passed on


def ring_schedule(n_ranks: int, rank: int) -> List[RingStep]:
    """The N steps of rank ``rank``: it starts with its own block and after step t holds the block
    of rank (rank - t - 1) mod N."""
    if n_ranks < 1 or not 0 <= rank < n_ranks:
        raise ValueError("need 0 <= rank < n_ranks")
    N = n_ranks
    return [RingStep(t, (rank - t) % N, (rank + 1) % N, (rank - 1) % N, (rank - t - 1) % N, t + 1 < N)
            for t in range(N)]


# ---------------------------------------------------------------------- block exchange

class P2PExchange:
    """Passes a rank's held block to the next rank of the ring and receives the previous rank's
    block, with torch.distributed point-to-point operations (posted together, so no rank waits for
    another to post first).  With NCCL the copies run on NCCL's stream, after the work already on
    the current stream, and ``wait`` makes the current stream wait for them: compute enqueued
    between ``start`` and ``wait`` overlaps the transfer."""

    def __init__(self, group=None, timeout=None):
        """``timeout`` (a datetime.timedelta) bounds each wait where the backend supports it
        (gloo): a rank that never sends or receives then raises an error here instead of
        leaving its neighbours waiting.  With NCCL the wait is a stream dependency and the
        process group's own timeout applies."""
        self.group = group
        self.timeout = timeout
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def _global(self, r):
        return r if self.group is None else dist.get_global_rank(self.group, r)

    def start(self, send: Sequence[torch.Tensor], recv: Sequence[torch.Tensor]):
        nxt = self._global((self.rank + 1) % self.world)
        prv = self._global((self.rank - 1) % self.world)
        ops = [dist.P2POp(dist.isend, t, nxt, self.group) for t in send]
        ops += [dist.P2POp(dist.irecv, t, prv, self.group) for t in recv]
        return dist.batch_isend_irecv(ops)

    def wait(self, handle):
        for work in handle:
            if self.timeout is None:
                work.wait()
            else:
                work.wait(self.timeout)


# ---------------------------------------------------------------------- prefill ring

StepFn = Callable[..., None]


def _held_slot(t: int) -> int:
    """Buffer set holding the block at step t: the caller's own buffers at step 0, then two spare
    sets in turn (so the caller's K/V are never overwritten)."""
    return 0 if t == 0 else 1 + (t - 1) % 2


def _recv_slot(t: int) -> int:
    """Buffer set the block arriving during step t lands in (the one held at step t - 1, t >= 2)."""
    return 1 + t % 2


def ring_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, step: StepFn,
                   exchange=None, n_ranks: Optional[int] = None, rank: Optional[int] = None,
                   out_dtype: Optional[torch.dtype] = None, trace: Optional[list] = None):
    """Ring attention of one rank over N ranks.

    q [rows, Hq, d], k/v [rows, Hkv, d]: this rank's local buffers as the head-tail partition
    gives them (per sequence chunk rank, then chunk 2N-1-rank).  At step t the rank computes its
    queries against the block it holds (that of rank (rank - t) mod N) with
    ``step(q, k_held, v_held, src, o_in, lse_in, o_out, lse_out)``, which folds the block's partial
    into the running (O, LSE) state: o_in/lse_in are None at the first step, o_out is the final
    output at the last step and the fp32 running state before.  Meanwhile ``exchange`` passes the
    held block on and receives the next one into another buffer (double buffering; k and v
    themselves are only read).

    n_ranks and rank default to the exchange's world and rank (one rank without an exchange).
    ``trace``, if given, receives (t, src, copy of the held K) per step.
    Returns (O [rows, Hq, d] in out_dtype (default q's), LSE fp32 [rows, Hq]).
    """
    if exchange is not None:
        n_ranks = exchange.world if n_ranks is None else n_ranks
        rank = exchange.rank if rank is None else rank
    n_ranks = 1 if n_ranks is None else n_ranks
    rank = 0 if rank is None else rank
    if n_ranks > 1 and exchange is None:
        raise ValueError("an exchange is needed for more than one rank")
    rows, Hq, d = q.shape
    o_acc = torch.empty((rows, Hq, d), dtype=torch.float32, device=q.device) if n_ranks > 1 else None
    lse = torch.empty((rows, Hq), dtype=torch.float32, device=q.device)
    o_fin = torch.empty((rows, Hq, d), dtype=out_dtype or q.dtype, device=q.device)
    n_sets = 1 + min(2, n_ranks - 1)
    bufs = [(k, v)] + [(torch.empty_like(k), torch.empty_like(v)) for _ in range(n_sets - 1)]
    for st in ring_schedule(n_ranks, rank):
        kh, vh = bufs[_held_slot(st.t)]
        handle = exchange.start([kh, vh], list(bufs[_recv_slot(st.t)])) if st.exchange else None
        if trace is not None:
            trace.append((st.t, st.src, kh.clone()))
        last = st.t == n_ranks - 1
        step(q, kh, vh, st.src, None if st.t == 0 else o_acc, None if st.t == 0 else lse,
             o_fin if last else o_acc, lse)
        if handle is not None:
            exchange.wait(handle)
    return o_fin, lse


def ring_attention_local(qs: Sequence[torch.Tensor], ks: Sequence[torch.Tensor], vs: Sequence[torch.Tensor], *,
                         step: StepFn, out_dtype: Optional[torch.dtype] = None):
    """All N ranks of the ring in one process, each with its own buffers, stepped together.

    The exchange of step t is a device copy of every rank's held block into the next rank's
    receive buffer, on a side stream that first waits for the computes of step t-1 (which read that
    buffer) and that the computes of step t+1 wait for: the same double buffering and ordering as
    the point-to-point exchange, on one device.  ``step(r, q, k_held, v_held, src, o_in, lse_in,
    o_out, lse_out)`` computes rank r's step.  Returns a list of (O, LSE) per rank.
    """
    N = len(qs)
    cuda = qs[0].is_cuda
    n_sets = 1 + min(2, N - 1)
    bufs = [[(ks[r], vs[r]) for r in range(N)]]
    bufs += [[(torch.empty_like(ks[r]), torch.empty_like(vs[r])) for r in range(N)] for _ in range(n_sets - 1)]
    o_acc = [torch.empty(q.shape, dtype=torch.float32, device=q.device) for q in qs] if N > 1 else [None] * N
    lse = [torch.empty(q.shape[:2], dtype=torch.float32, device=q.device) for q in qs]
    o_fin = [torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device) for q in qs]
    comp = torch.cuda.current_stream() if cuda else None
    side = torch.cuda.Stream(device=qs[0].device) if cuda and N > 1 else None
    for t in range(N):
        held, nxt = bufs[_held_slot(t)], bufs[_recv_slot(t)] if t + 1 < N else None
        done = None
        if nxt is not None:
            if cuda:
                side.wait_stream(comp)        # the receive buffers were read by the computes of step t-1
                with torch.cuda.stream(side):
                    for r in range(N):
                        nxt[(r + 1) % N][0].copy_(held[r][0], non_blocking=True)
                        nxt[(r + 1) % N][1].copy_(held[r][1], non_blocking=True)
                done = torch.cuda.Event()
                done.record(side)
            else:
                for r in range(N):
                    nxt[(r + 1) % N][0].copy_(held[r][0])
                    nxt[(r + 1) % N][1].copy_(held[r][1])
        last = t == N - 1
        for r in range(N):
            step(r, qs[r], held[r][0], held[r][1], (r - t) % N, None if t == 0 else o_acc[r],
                 None if t == 0 else lse[r], o_fin[r] if last else o_acc[r], lse[r])
        if done is not None:
            comp.wait_event(done)
    if side is not None:
        comp.wait_stream(side)   # order the side stream's last reads before the buffers are reused
    return list(zip(o_fin, lse))


def allgather_kv_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, restore: torch.Tensor,
                           gather: Callable[..., None], attend: Callable[..., None], group=None,
                           out_dtype: Optional[torch.dtype] = None):
    """Prefill with the K/V all-gathered instead of passed around a ring: the form the vLLM-Ascend
    "Context Parallel (CP)" page says ships for PCP prefill (every device all-gathers the K/V of the
    layer, attends its own queries over all of it, and drops the gathered K/V after use).

      1. all-gather every rank's local K/V ([rows, Hkv, d], per sequence chunk r then chunk 2N-1-r):
         the result is in the head-tail partition's gathered order;
      2. ``gather(src, restore, dst)`` puts it back in token order with the partition's restore index
         (pcp_allgather_restore_idx);
      3. ``attend(q, k_nat, v_nat, o, lse)`` computes this rank's queries over the keys in token order.

    Returns (O [rows, Hq, d] in out_dtype (default q's), LSE fp32 [rows, Hq]).
    """
    W = dist.get_world_size(group)
    rows = k.shape[0]
    k_all = torch.empty((W * rows,) + tuple(k.shape[1:]), dtype=k.dtype, device=k.device)
    v_all = torch.empty_like(k_all)
    dist.all_gather_into_tensor(k_all, k.contiguous(), group=group)
    dist.all_gather_into_tensor(v_all, v.contiguous(), group=group)
    k_nat = torch.empty((restore.numel(),) + tuple(k.shape[1:]), dtype=k.dtype, device=k.device)
    v_nat = torch.empty_like(k_nat)
    gather(k_all, restore, k_nat)
    gather(v_all, restore, v_nat)
    del k_all, v_all
    o = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    attend(q, k_nat, v_nat, o, lse)
    return o, lse


# ---------------------------------------------------------------------- decode merge

def cp_lse_ag_out_rs(o_local: torch.Tensor, lse_local: torch.Tensor, *, rescale: Callable[..., None],
                     group=None):
    """The decode's merge across the ranks of ``group`` (vLLM-Ascend "Context Parallel (CP)", DCP
    decode): every rank holds its partial O_w [R, Hq, d] (fp32, normalised over the keys it stores)
    and LSE_w [R, Hq].

      1. all-gather the LSEs into [W, R, Hq];
      2. ``rescale(o_local, lse_all, w, o_scaled, lse_total)`` scales O_w by e^{LSE_w - LSE} into
         o_scaled [W, R, Hq/W, d] (the heads of rank v in slot v) and writes the merged LSE of this
         rank's heads into lse_total [R, Hq/W];
      3. reduce-scatter (sum) o_scaled: rank w receives the merged O of heads
         [w*Hq/W, (w+1)*Hq/W).

    Returns (O [R, Hq/W, d] fp32, LSE [R, Hq/W]) of this rank's heads.  Hq must be a multiple of
    the group size.
    """
    W = dist.get_world_size(group)
    w = dist.get_rank(group)
    R, Hq, d = o_local.shape
    if Hq % W != 0:
        raise ValueError("Hq (%d) must be a multiple of the number of ranks (%d)" % (Hq, W))
    # the gathered and scattered tensors are passed as their rank-concatenated (dim 0) views
    lse_all = torch.empty((W, R, Hq), dtype=torch.float32, device=o_local.device)
    dist.all_gather_into_tensor(lse_all.view(W * R, Hq), lse_local.contiguous(), group=group)
    o_scaled = torch.empty((W, R, Hq // W, d), dtype=torch.float32, device=o_local.device)
    lse_total = torch.empty((R, Hq // W), dtype=torch.float32, device=o_local.device)
    rescale(o_local, lse_all, w, o_scaled, lse_total)
    out = torch.empty((R, Hq // W, d), dtype=torch.float32, device=o_local.device)
    dist.reduce_scatter_tensor(out, o_scaled.view(W * R, Hq // W, d), op=dist.ReduceOp.SUM, group=group)
    return out, lse_total


def cp_lse_a2a(o_local: torch.Tensor, lse_local: torch.Tensor, *, split: Callable[..., None],
               merge: Callable[..., None], group=None):
    """The all-to-all form of the decode's merge across the ranks of ``group`` (vLLM-Ascend "Context
    Parallel (CP)", DCP and PCP decode name it beside cp_lse_ag_out_rs): every rank holds its
    partial O_w [R, Hq, d] (fp32, normalised over the keys it stores) and LSE_w [R, Hq].

      1. ``split(o_local, lse_local, W, o_split, lse_split)`` lays them out by the rank that keeps
         each head: o_split [W, R, Hq/W, d], lse_split [W, R, Hq/W];
      2. an all-to-all sends slot v to rank v, which receives the W partials of its heads;
      3. ``merge(o_parts, lse_parts, o, lse)`` merges them (the LSE merge over P = W).

    Returns (O [R, Hq/W, d] fp32, LSE [R, Hq/W]) of this rank's heads, the same as
    cp_lse_ag_out_rs.  Hq must be a multiple of the group size.
    """
    W = dist.get_world_size(group)
    R, Hq, d = o_local.shape
    if Hq % W != 0:
        raise ValueError("Hq (%d) must be a multiple of the number of ranks (%d)" % (Hq, W))
    hs = Hq // W
    dev = o_local.device
    o_split = torch.empty((W, R, hs, d), dtype=torch.float32, device=dev)
    lse_split = torch.empty((W, R, hs), dtype=torch.float32, device=dev)
    split(o_local, lse_local, W, o_split, lse_split)
    o_parts = torch.empty_like(o_split)
    lse_parts = torch.empty_like(lse_split)
    dist.all_to_all_single(o_parts.view(W * R, hs, d), o_split.view(W * R, hs, d), group=group)
    dist.all_to_all_single(lse_parts.view(W * R, hs), lse_split.view(W * R, hs), group=group)
    o = torch.empty((R, hs, d), dtype=torch.float32, device=dev)
    lse = torch.empty((R, hs), dtype=torch.float32, device=dev)
    merge(o_parts, lse_parts, o, lse)
    return o, lse
