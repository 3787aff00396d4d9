"""Context-parallel KV cache: slot mapping, scatter into the sharded paged
cache, split-KV decode partials and their merge.  Test infrastructure only.

Source: vLLM-Ascend developer guide "Context Parallel (CP)":
* section "Block table": a virtual block groups the blocks of one CP device
  group, virtual_block_size = block_size * pcp * dcp.  For a token x: block
  index x // virtual_block_size, offset o = x % virtual_block_size, local block
  index o // interleave, device = local_block_index % (pcp * dcp), offset in the
  local block = (local_block_index // (pcp * dcp)) * interleave + o % interleave.
  The implementation requires block_size % interleave == 0.
* section "Decode context parallel (DCP)", decode: every device computes
  attention over its local KV shard and the partial outputs and LSEs are merged
  (cp_lse_ag_out_rs); the PCP decode section adds one more gather before the
  same update, which on one device is the same merge over all W = pcp*dcp
  partials.

Readings (the page is silent; also in the design notes):
* per-device slot arrays cover every token of the batch, -1 where the device
  does not store the token;
* one physical block id per virtual block, used at that index in every
  device's pool;
* devices are numbered flat, 0 <= dev < pcp*dcp;
* cache layout [W, num_blocks, Hkv, block_size, d] (one head's block is
  contiguous);
* the decode query of a request with context length L attends tokens 0..L-1;
* an empty partial (no owned token) has LSE = -inf and weight 0.

Parity status: pinned (hand-worked slot examples, bijection invariant, the
block_size % interleave rule, and decode == plain attention over the original
token K/V).
"""

from __future__ import annotations

import numpy as np

from .attention import attention_rows, lse_merge, NEG_INF, _as64


def _check(block_size, interleave, pcp, dcp):
    if min(block_size, interleave, pcp, dcp) < 1:
        raise ValueError("sizes must be positive")
    if block_size % interleave != 0:
        raise ValueError("block_size % cp_kv_cache_interleave_size must be 0")


def cp_token_location(x: int, block_size: int, interleave: int, pcp: int, dcp: int):
    """(virtual block, device, offset in the device's local block) of token x."""
    _check(block_size, interleave, pcp, dcp)
    vbs = block_size * pcp * dcp
    vb = x // vbs
    o = x % vbs
    lbi = o // interleave
    dev = lbi % (pcp * dcp)
    off = (lbi // (pcp * dcp)) * interleave + o % interleave
    return vb, dev, off


def cp_slot_mapping(query_start_loc, positions, block_table, block_size: int,
                    interleave: int, pcp: int, dcp: int):
    """Per-device slot mapping, int64 [W, T]; -1 where the device does not own the token.

    Token t belongs to request q with query_start_loc[q] <= t < query_start_loc[q+1];
    positions[t] is its position x in that request.
    """
    _check(block_size, interleave, pcp, dcp)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    pos = np.asarray(positions, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    W = pcp * dcp
    T = len(pos)
    req = np.searchsorted(qsl, np.arange(T), side="right") - 1
    vbs = block_size * W
    vb = pos // vbs
    o = pos % vbs
    lbi = o // interleave
    dev = lbi % W
    off = (lbi // W) * interleave + o % interleave
    slot = bt[req, vb] * block_size + off
    out = np.full((W, T), -1, dtype=np.int64)
    out[dev, np.arange(T)] = slot
    return out


def cp_kv_scatter(k, v, slot, k_cache, v_cache, block_size: int):
    """Write token rows k, v [T, Hkv, d] into caches [W, NB, Hkv, bs, d] at slot [W, T]."""
    W, T = slot.shape
    for w in range(W):
        ts = np.nonzero(slot[w] >= 0)[0]
        s = slot[w, ts]
        k_cache[w, s // block_size, :, s % block_size, :] = k[ts]
        v_cache[w, s // block_size, :, s % block_size, :] = v[ts]


def cp_kv_gather(k_cache, v_cache, block_table, query_start_loc, positions, block_size: int,
                 interleave: int, pcp: int, dcp: int):
    """Rows of the sharded cache back in token order (the reorg that makes
    each request's KV contiguous after the context all-gather; vLLM-Ascend
    "Context Parallel (CP)", DCP chunked prefill, MLA: all_gather of the
    context KV, then reorg_kvcache).  Output row t holds the K/V of token
    positions[t] of its request, read from the device and offset the
    block-table formula assigns to it.  Returns (k [T, Hkv, d], v [T, Hkv, d]).
    """
    _check(block_size, interleave, pcp, dcp)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    pos = np.asarray(positions, dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    T = len(pos)
    req = np.searchsorted(qsl, np.arange(T), side="right") - 1
    out_k = np.zeros((T,) + k_cache.shape[2:3] + k_cache.shape[4:], dtype=k_cache.dtype)
    out_v = np.zeros_like(out_k)
    for t in range(T):
        vb, dev, off = cp_token_location(int(pos[t]), block_size, interleave, pcp, dcp)
        blk = bt[req[t], vb]
        out_k[t] = k_cache[dev, blk, :, off, :]
        out_v[t] = v_cache[dev, blk, :, off, :]
    return out_k, out_v


def _device_tokens(w, vb, block_size, interleave, W):
    """Token index x (within the request) held in local slot j of device w, virtual block vb."""
    j = np.arange(block_size)
    lbi = (j // interleave) * W + w
    return vb * block_size * W + lbi * interleave + j % interleave


def cp_decode_partials(q, k_cache, v_cache, block_table, ctx_lens, block_size: int,
                       interleave: int, pcp: int, dcp: int, split_blocks: int, scale=None):
    """Split-KV decode partials read from the sharded cache.

    Partial p = w * n_splits + sp covers device w's local blocks of virtual
    blocks [sp*split_blocks, (sp+1)*split_blocks).  Returns (O [P, R, Hq, d],
    LSE [P, R, Hq], n_splits).
    """
    _check(block_size, interleave, pcp, dcp)
    q = _as64(q)
    R, Hq, d = q.shape
    W = pcp * dcp
    bt = np.asarray(block_table, dtype=np.int64)
    n_splits = -(-bt.shape[1] // split_blocks)
    P = W * n_splits
    O = np.zeros((P, R, Hq, d))
    LSE = np.full((P, R, Hq), NEG_INF)
    Hkv = k_cache.shape[2]
    vbs = block_size * W
    for r in range(R):
        L = int(ctx_lens[r])
        nvb = -(-L // vbs)
        for w in range(W):
            for sp in range(n_splits):
                ks, vs = [], []
                for vb in range(sp * split_blocks, min(nvb, (sp + 1) * split_blocks)):
                    x = _device_tokens(w, vb, block_size, interleave, W)
                    ok = x < L
                    blk = bt[r, vb]
                    ks.append(_as64(k_cache[w, blk][:, ok, :]).transpose(1, 0, 2))
                    vs.append(_as64(v_cache[w, blk][:, ok, :]).transpose(1, 0, 2))
                if not ks or sum(len(a) for a in ks) == 0:
                    continue
                kk = np.concatenate(ks)
                vv = np.concatenate(vs)
                # the query sees every owned key (no mask beyond x < L)
                o, lse = attention_rows(q[r:r + 1], [len(kk)], kk, vv, False, scale)
                O[w * n_splits + sp, r] = o[0]
                LSE[w * n_splits + sp, r] = lse[0]
    assert Hkv == k_cache.shape[2]
    return O, LSE, n_splits


def cp_decode(q, k_cache, v_cache, block_table, ctx_lens, block_size, interleave, pcp, dcp,
              split_blocks, scale=None):
    """Decode output (O [R, Hq, d], LSE [R, Hq]) = merge of all split-KV partials."""
    O_p, L_p, _ = cp_decode_partials(q, k_cache, v_cache, block_table, ctx_lens, block_size,
                                     interleave, pcp, dcp, split_blocks, scale)
    return lse_merge(O_p, L_p)


def cp_lse_ag_out_rs(o_dev, lse_dev):
    """The decode's merge across W devices, in the steps the name spells out
    (vLLM-Ascend "Context Parallel (CP)", DCP decode: cp_lse_ag_out_rs; the
    weights are those of the blockwise decomposition on the "Ring Attention"
    tag page).  Device w holds its own partial O_w [R, Hq, d] (normalised over
    the keys it stores) and LSE_w [R, Hq].
      1. all-gather the LSEs, so every device sees LSE_0 .. LSE_{W-1};
      2. every device rescales its own O_w by e^{LSE_w - LSE} with
         LSE = ln sum_w e^{LSE_w} (a device with LSE_w = -inf contributes 0);
      3. reduce-scatter the rescaled outputs over the head dimension: the sum
         over devices, of which device w keeps heads [w*Hq/W, (w+1)*Hq/W).
    Requires Hq % W == 0.  Returns a list over devices of (O [R, Hq/W, d],
    LSE [R, Hq/W]).
    """
    W = len(o_dev)
    o_dev = [_as64(o) for o in o_dev]
    lse_dev = [_as64(l) for l in lse_dev]
    R, Hq, d = o_dev[0].shape
    if Hq % W != 0:
        raise ValueError("Hq must be a multiple of the number of devices")
    hs = Hq // W
    gathered = np.stack(lse_dev)                                   # step 1: [W, R, Hq] on every device
    M = gathered.max(axis=0)
    live = np.isfinite(M)
    Ms = np.where(live, M, 0.0)
    tot = np.where(np.isfinite(gathered), np.exp(gathered - Ms[None]), 0.0).sum(axis=0)
    LSE = np.where(live, Ms + np.log(np.where(live, tot, 1.0)), NEG_INF)
    scaled = []
    for w in range(W):                                             # step 2, on device w
        wgt = np.where(np.isfinite(lse_dev[w]) & live, np.exp(lse_dev[w] - np.where(live, LSE, 0.0)), 0.0)
        o_safe = np.where(np.isfinite(lse_dev[w])[..., None], o_dev[w], 0.0)
        scaled.append(wgt[..., None] * o_safe)
    out = []
    for w in range(W):                                             # step 3: device w's share of the sum
        heads = slice(w * hs, (w + 1) * hs)
        out.append((sum(x[:, heads] for x in scaled), LSE[:, heads]))
    return out


def decode_reference(q_row, k_tokens, v_tokens, scale=None):
    """Plain attention of one query [Hq, d] over a request's own token K/V
    [L, Hkv, d] (no cache involved): the value the sharded decode must reach."""
    q_row = _as64(q_row)[None]
    o, lse = attention_rows(q_row, [len(k_tokens)], k_tokens, v_tokens, False, scale)
    return o[0], lse[0]


__all__ = ["cp_token_location", "cp_slot_mapping", "cp_kv_scatter", "cp_kv_gather",
           "cp_decode_partials", "cp_decode", "cp_lse_ag_out_rs", "decode_reference"]
