"""Float64 attention oracle: the plain definition, the literal N-step ring,
per-rank partials and the LSE merge.  Test infrastructure only.

Conventions (shared with the CUDA library only by documentation):
  q [S, Hq, d], k and v [S, Hkv, d] for ONE sequence, token-major, in natural
  token order; query head h reads key/value head h // (Hq // Hkv) (consecutive
  query heads share a K/V head, GQA).  scale defaults to 1/sqrt(d).  LSE is the
  natural logarithm of the sum of exp(scaled scores).  O is [S, Hq, d] and LSE
  [S, Hq].  With ``causal`` the query at position i sees keys j <= i.

Parity status: every function below is pinned by tests/test_oracle_attention.py
(hand-worked golden values, closed-form special cases, invariants and the
ring/full identity); none is unpinned.
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def _as64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: exact widening to float64
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def _kv_head_of(Hq: int, Hkv: int) -> np.ndarray:
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return np.arange(Hq) // (Hq // Hkv)


def _default_scale(d: int, scale):
    return 1.0 / math.sqrt(d) if (scale is None or scale <= 0) else float(scale)


def _visible(qpos, kpos):
    """Causal rule on original positions: the query at i sees the key at j iff j <= i."""
    return kpos <= qpos


# ---------------------------------------------------------------------------
# Plain definition: softmax(scale * Q K^T) V, one row at a time.
# ("Ring Attention" tag page, attention memory-wall article: Attn = softmax(QK^T/sqrt(d)) V)
# ---------------------------------------------------------------------------

def attention_rows(q_rows, q_pos, k, v, causal: bool, scale=None):
    """Attention of selected query rows against all keys of one sequence.

    q_rows [n, Hq, d] are queries at token positions q_pos [n]; keys/values
    k, v [S, Hkv, d] sit at positions 0..S-1.  Returns (O [n, Hq, d],
    LSE [n, Hq]).  A row with no visible key gets O = 0 and LSE = -inf.
    """
    q_rows, k, v = _as64(q_rows), _as64(k), _as64(v)
    n, Hq, d = q_rows.shape
    S, Hkv, _ = k.shape
    sc = _default_scale(d, scale)
    g_of = _kv_head_of(Hq, Hkv)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    O = np.zeros((n, Hq, d))
    LSE = np.full((n, Hq), NEG_INF)
    kpos = np.arange(S)
    for h in range(Hq):
        g = g_of[h]
        s = sc * (q_rows[:, h, :] @ k[:, g, :].T)          # [n, S]
        if causal:
            s = np.where(_visible(q_pos[:, None], kpos[None, :]), s, NEG_INF)
        M = s.max(axis=1)
        live = np.isfinite(M)
        Ms = np.where(live, M, 0.0)
        e = np.exp(s - Ms[:, None])                         # exp(-inf) = 0
        den = e.sum(axis=1)
        num = e @ v[:, g, :]
        with np.errstate(invalid="ignore", divide="ignore"):
            O[:, h, :] = np.where(live[:, None], num / den[:, None], 0.0)
            LSE[:, h] = np.where(live, M + np.log(den), NEG_INF)
    return O, LSE


def attention_block(q_rows, q_pos0: int, k, v, k_pos0: int, causal: bool, scale=None):
    """Partial attention of a query block against a key block.

    Queries q_rows[i] sit at positions q_pos0 + i, keys/values k[j], v[j] at
    k_pos0 + j.  Returns (O [n, Hq, d], LSE [n, Hq]) of softmax over the visible
    keys of this block only; a row that sees none gets O = 0 and LSE = -inf.
    These are the partials that the merge combines.
    """
    q_rows, k, v = _as64(q_rows), _as64(k), _as64(v)
    n, Hq, d = q_rows.shape
    sc = _default_scale(d, scale)
    g_of = _kv_head_of(Hq, k.shape[1])
    state = (np.full((n, Hq), NEG_INF), np.zeros((n, Hq)), np.zeros((n, Hq, d)))
    qpos = q_pos0 + np.arange(n)
    kpos = k_pos0 + np.arange(len(k))
    state = _block_update(state, q_rows, qpos, k, v, kpos, causal, sc, g_of)
    return _finish(state)


def segmented_attention(q_rows, q_pos0: int, k, v, causal: bool, seg: int, scale=None):
    """Chunked prefill with a bounded key segment per round (vLLM-Ascend
    "Context Parallel (CP)", chunked prefill: a maximum amount of KV per round,
    attention and online-softmax update segment after segment).

    Keys 0..len(k)-1 are cut into segments of `seg` tokens; every segment gives
    a partial (O, LSE) of the query block, and the partials are merged.
    Returns (O, LSE, O_parts, LSE_parts).
    """
    parts_o, parts_l = [], []
    for k0 in range(0, len(k), seg):
        o, l = attention_block(q_rows, q_pos0, k[k0:k0 + seg], v[k0:k0 + seg], k0, causal, scale)
        parts_o.append(o)
        parts_l.append(l)
    Op, Lp = np.stack(parts_o), np.stack(parts_l)
    O, L = lse_merge(Op, Lp)
    return O, L, Op, Lp


def full_attention(q, k, v, causal: bool, scale=None, row_block: int = 1024):
    """Full softmax attention of one sequence (plain definition, float64).

    Rows are evaluated independently, ``row_block`` at a time to bound memory.
    """
    q = _as64(q)
    S = q.shape[0]
    O = np.zeros(q.shape)
    LSE = np.zeros(q.shape[:2])
    for s0 in range(0, S, row_block):
        s1 = min(S, s0 + row_block)
        O[s0:s1], LSE[s0:s1] = attention_rows(q[s0:s1], np.arange(s0, s1), k, v, causal, scale)
    return O, LSE


# ---------------------------------------------------------------------------
# Zigzag chunk ownership (vLLM-Ascend "Context Parallel", head-tail partition):
# the sequence is cut into 2N equal chunks; rank r holds chunk r followed by
# chunk 2N-1-r.
# ---------------------------------------------------------------------------

def rank_chunks(N: int, r: int):
    return (r, 2 * N - 1 - r)


def _rank_positions(N: int, c: int, r: int) -> np.ndarray:
    a, b = rank_chunks(N, r)
    return np.concatenate([np.arange(a * c, (a + 1) * c), np.arange(b * c, (b + 1) * c)])


# ---------------------------------------------------------------------------
# Blockwise online softmax update ("Ring Attention" tag page, memory-wall
# article, key insight: keep a running max and running sum per query row).
# ---------------------------------------------------------------------------

def _block_update(state, qb, qpos, kb, vb, kpos, causal, sc, g_of):
    """One online-softmax update of (m, l, acc) with a K/V block.

    m' = max(m, rowmax s);  alpha = e^{m - m'};  l' = alpha*l + sum_j e^{s_j - m'};
    acc' = alpha*acc + sum_j e^{s_j - m'} v_j.
    """
    m, l, acc = state
    kx = kb[:, g_of, :]                                     # [nk, Hq, d]
    vx = vb[:, g_of, :]
    s = sc * np.einsum("ihd,jhd->ihj", qb, kx)              # [nq, Hq, nk]
    if causal:
        vis = _visible(qpos[:, None], kpos[None, :])        # [nq, nk]
        s = np.where(vis[:, None, :], s, NEG_INF)
    m_new = np.maximum(m, s.max(axis=2))
    m_safe = np.where(np.isfinite(m_new), m_new, 0.0)
    alpha = np.where(np.isfinite(m), np.exp(m - m_safe), 0.0)
    p = np.exp(s - m_safe[:, :, None])
    l_new = alpha * l + p.sum(axis=2)
    acc_new = alpha[:, :, None] * acc + np.einsum("ihj,jhd->ihd", p, vx)
    return m_new, l_new, acc_new


def _finish(state):
    m, l, acc = state
    live = l > 0
    with np.errstate(invalid="ignore", divide="ignore"):
        O = np.where(live[:, :, None], acc / np.where(live, l, 1.0)[:, :, None], 0.0)
        LSE = np.where(live, m + np.log(np.where(live, l, 1.0)), NEG_INF)
    return O, LSE


def ring_attention(q, k, v, causal: bool, n_ranks: int, scale=None):
    """Literal N-step ring over N virtual ranks with the zigzag chunk split.

    Rank r holds Q/K/V of chunks (r, 2N-1-r).  At step t = 0..N-1 every rank
    updates its running state with the K/V block it currently holds, which is
    the block of rank (r - t) mod N, and then passes that block to rank r + 1
    (the buffers are rotated explicitly).  After N steps each rank's state is
    final; the outputs are written back to natural token order.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    S, Hq, d = q.shape
    N = n_ranks
    if N < 1 or S % (2 * N) != 0:
        raise ValueError("S must be a positive multiple of 2*n_ranks")
    c = S // (2 * N)
    sc = _default_scale(d, scale)
    g_of = _kv_head_of(Hq, k.shape[1])
    pos = [_rank_positions(N, c, r) for r in range(N)]
    states = [(np.full((2 * c, Hq), NEG_INF), np.zeros((2 * c, Hq)), np.zeros((2 * c, Hq, d)))
              for _ in range(N)]
    held = [(k[pos[r]], v[pos[r]], pos[r], r) for r in range(N)]    # rank r starts with its own K/V
    for t in range(N):
        for r in range(N):
            kb, vb, kpos, owner = held[r]
            assert owner == (r - t) % N
            states[r] = _block_update(states[r], q[pos[r]], pos[r], kb, vb, kpos, causal, sc, g_of)
        held = [held[(r - 1) % N] for r in range(N)]                 # send to r+1 / receive from r-1
    O = np.zeros((S, Hq, d))
    LSE = np.zeros((S, Hq))
    for r in range(N):
        O[pos[r]], LSE[pos[r]] = _finish(states[r])
    return O, LSE


def ring_partials(q, k, v, causal: bool, n_ranks: int, scale=None):
    """Partial (O, LSE) of every rank's queries against every rank's K/V block.

    Returns (parts, positions): parts[r][s] = (O_rs [2c, Hq, d], LSE_rs [2c, Hq])
    computed directly from the definition over the keys of rank s only (LSE -inf
    and O 0 where nothing is visible), positions[r] = natural positions of rank
    r's local rows.  Merging parts[r][0..N-1] with ``lse_merge`` in any order
    gives rank r's rows of full attention.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    S, Hq, d = q.shape
    N = n_ranks
    c = S // (2 * N)
    pos = [_rank_positions(N, c, r) for r in range(N)]
    parts = []
    for r in range(N):
        row = []
        for s in range(N):
            # attention of rank r's rows over a sequence made of rank s's keys only
            O, LSE = _rows_over_keys(q[pos[r]], pos[r], k[pos[s]], v[pos[s]], pos[s], causal, scale)
            row.append((O, LSE))
        parts.append(row)
    return parts, pos


def ring_step(q_local, k_held, v_held, n_ranks: int, rank: int, src: int, causal: bool,
              o_in=None, lse_in=None, B: int = 1, scale=None):
    """One ring step of one rank, applied to that rank's running result.

    The rank's local buffers are what the head-tail partition gives it: per
    sequence (B of them, equal length 2Nc), chunk `rank` followed by chunk
    2N-1-rank, c rows each.  q_local [B*2c, Hq, d] are rank `rank`'s queries;
    k_held, v_held [B*2c, Hkv, d] are the K/V block that rank holds at this
    step, i.e. the local K/V of rank `src` (src = (rank - t) mod N at step t,
    "Ring Attention" tag page, ring topology).  The partial (O_p, LSE_p) of the
    queries over the visible keys of that block comes from the definition;
    it is then folded into the running (o_in, lse_in) with the LSE merge (the
    blockwise decomposition of the same page: a partial over a key subset is
    carried by its LSE).  Without o_in the partial itself is the result.
    Returns (O [B*2c, Hq, d], LSE [B*2c, Hq]).
    """
    q_local, k_held, v_held = _as64(q_local), _as64(k_held), _as64(v_held)
    N = int(n_ranks)
    rows = q_local.shape[0]
    if rows % (2 * B) != 0 or k_held.shape[0] != rows:
        raise ValueError("local buffers must hold B sequences of 2c rows")
    c = rows // (2 * B)
    qpos = _rank_positions(N, c, rank)
    kpos = _rank_positions(N, c, src)
    O_p = np.zeros(q_local.shape)
    L_p = np.zeros(q_local.shape[:2])
    for b in range(B):
        sl = slice(b * 2 * c, (b + 1) * 2 * c)
        O_p[sl], L_p[sl] = _rows_over_keys(q_local[sl], qpos, k_held[sl], v_held[sl], kpos, causal, scale)
    if o_in is None:
        return O_p, L_p
    return lse_merge(np.stack([_as64(o_in), O_p]), np.stack([_as64(lse_in), L_p]))


def _rows_over_keys(qr, qpos, kk, vv, kpos, causal, scale):
    qr, kk, vv = _as64(qr), _as64(kk), _as64(vv)
    n, Hq, d = qr.shape
    sc = _default_scale(d, scale)
    g_of = _kv_head_of(Hq, kk.shape[1])
    state = (np.full((n, Hq), NEG_INF), np.zeros((n, Hq)), np.zeros((n, Hq, d)))
    # a single block: the update from the empty state is the plain softmax
    state = _block_update(state, qr, np.asarray(qpos), kk, vv, np.asarray(kpos), causal, sc, g_of)
    return _finish(state)


# ---------------------------------------------------------------------------
# LSE merge (vLLM-Ascend "Context Parallel", DCP decode: all-gather the partial
# outputs and LSEs, update the result).
# ---------------------------------------------------------------------------

def lse_merge(o_parts, lse_parts):
    """Merge P partial results: LSE = ln sum_p e^{LSE_p}; O = sum_p e^{LSE_p - LSE} O_p.

    o_parts [P, ..., d], lse_parts [P, ...].  Partials with LSE = -inf carry
    weight 0 (their O is never read); if all are -inf, O = 0 and LSE = -inf.
    """
    o_parts, lse_parts = _as64(o_parts), _as64(lse_parts)
    M = lse_parts.max(axis=0)
    live = np.isfinite(M)
    Ms = np.where(live, M, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - Ms[None]), 0.0)   # [P, ...]
    tot = w.sum(axis=0)
    LSE = np.where(live, Ms + np.log(np.where(live, tot, 1.0)), NEG_INF)
    o_safe = np.where(np.isfinite(lse_parts)[..., None], o_parts, 0.0)
    O = (w[..., None] * o_safe).sum(axis=0) / np.where(live, tot, 1.0)[..., None]
    O = np.where(live[..., None], O, 0.0)
    return O, LSE


# ---------------------------------------------------------------------------
# Causal work per rank under the zigzag split (derived; pinned by closed forms).
# ---------------------------------------------------------------------------

def causal_pairs_per_rank(N: int, c: int):
    """Number of visible (query, key) pairs of each rank's queries, by brute force."""
    S = 2 * N * c
    out = []
    for r in range(N):
        qp = _rank_positions(N, c, r)
        out.append(int(sum(int(p) + 1 for p in qp)))   # query at p sees keys 0..p
    assert sum(out) == S * (S + 1) // 2
    return out


def causal_tiles_per_rank(N: int, c: int, T: int, Tk: int = None):
    """Per rank: (full, partial, skipped) counts of (query tile, key tile) pairs
    when every chunk is cut into query tiles of T and key tiles of Tk tokens
    (Tk defaults to T; the last tile of a chunk may be shorter).

    Classification is by brute force over the positions inside each tile pair:
    'full' if every pair is visible, 'partial' if some are, 'skip' if none.
    """
    Tk = T if Tk is None else Tk

    def tiles(L):
        out = []
        for ch in range(2 * N):
            for i in range(-(-c // L)):
                lo = ch * c + i * L
                out.append((ch, lo, min(ch * c + c, lo + L)))
        return out

    qtiles, ktiles = tiles(T), tiles(Tk)
    res = []
    for r in range(N):
        mine = [t for t in qtiles if t[0] in rank_chunks(N, r)]
        full = part = skip = 0
        for (_, qlo, qhi) in mine:
            for (_, klo, khi) in ktiles:
                qs = np.arange(qlo, qhi)[:, None]
                ks = np.arange(klo, khi)[None, :]
                vis = _visible(qs, ks)
                if vis.all():
                    full += 1
                elif vis.any():
                    part += 1
                else:
                    skip += 1
        res.append((full, part, skip))
    return res
