"""Thin Python binding of libringattn.so (argument marshalling only).

Every computation runs in the library's CUDA kernels; this module checks
shapes/dtypes, passes raw device pointers and the current CUDA stream, and
turns a non-zero ``ra_status`` into ``RingAttnError``.  There is no fallback:
if the library is not built, or no GPU is present, calls fail loudly.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from .build import LIB

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA, RA_ERR_TIMEOUT, RA_ERR_DEVICE_BOUNDS = range(6)
RA_F32, RA_BF16 = 0, 1
LAYOUTS = {"natural": 0, "zigzag": 1}

_c = ctypes
_vp, _i32, _i64, _u64, _f32, _sz = _c.c_void_p, _c.c_int32, _c.c_int64, _c.c_uint64, _c.c_float, _c.c_size_t

# name -> argument types (restype is ra_status unless noted)
SIGNATURES = {
    "ra_device_status": [_vp],
    "ra_zigzag_partition": [_c.POINTER(_i64), _i32, _i32, _vp, _vp, _c.POINTER(_i64), _c.POINTER(_i64), _vp],
    "ra_gather_rows": [_vp, _i64, _vp, _vp, _i64, _i64, _vp],
    "ra_rope_gather": [_vp, _i64, _i32, _i32, _c.c_int, _vp, _i64, _vp, _c.c_double, _vp, _vp],
    "ra_ring_attn_fwd": [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _c.c_int, _i32, _i32, _f32,
                         _c.c_int, _vp],
    "ra_ring_attn_fwd_ex": [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _c.c_int, _i32, _i32, _f32,
                            _c.c_int, _i32, _vp],
    "ra_ring_attn_fwd_varlen": [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _c.c_int, _i32, _i32, _f32,
                                _vp],
    "ra_ring_schedule_counts": [_i32, _i32, _i32, _vp, _vp],
    "ra_ring_schedule_counts_ex": [_i32, _i32, _i32, _i32, _vp, _vp],
    "ra_lse_merge": [_vp, _vp, _i32, _i64, _i32, _i32, _vp, _c.c_int, _vp, _vp],
    "ra_ring_step_fwd": [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _vp,
                         _c.c_int, _vp, _vp],
    "ra_attn_block_fwd": [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _i64, _i32, _f32, _vp, _vp, _vp],
    "ra_segmented_prefill_workspace_size": [_i32, _i32, _i32, _i32, _i32, _c.POINTER(_sz)],
    "ra_segmented_prefill_fwd": [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i64, _i32, _f32, _i32, _vp,
                                 _c.c_int, _vp, _vp, _sz, _vp],
    "ra_cp_slot_mapping": [_vp, _vp, _vp, _i32, _i32, _i64, _i32, _i32, _i32, _i32, _vp, _vp],
    "ra_cp_kv_scatter": [_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _i64, _c.c_int, _vp],
    "ra_cp_kv_gather": [_vp, _vp, _vp, _i32, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32, _i32, _i32, _i64,
                        _c.c_int, _vp, _vp, _vp],
    "ra_cp_decode_workspace_size": [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _c.POINTER(_sz)],
    "ra_cp_decode": [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i64, _f32,
                     _i32, _vp, _c.c_int, _vp, _vp, _sz, _vp],
    "ra_cp_decode_noalloc": [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i64,
                             _f32, _i32, _vp, _c.c_int, _vp, _vp],
    "ra_cp_decode_partials": [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                              _i32, _i64, _f32, _i32, _vp, _vp, _c.POINTER(_i32), _vp],
    "ra_cp_lse_rescale": [_vp, _vp, _i32, _i32, _i64, _i32, _i32, _vp, _vp, _vp],
    "ra_cp_head_split": [_vp, _vp, _i32, _i64, _i32, _i32, _vp, _vp, _vp],
    "ra_selftest_wait_timeout": [_i64, _vp],
    "ra_synth_fill": [_u64, _i64, _vp, _i32, _vp, _vp],
}
STRING_FUNCS = ["ra_last_error", "ra_version"]


class RingAttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("ra_status %d: %s" % (status, msg))
        self.status = status


_lib = None


def lib():
    """The loaded library (ctypes), with argument types set."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError("libringattn.so is not built: run __graft_entry__.build() "
                               "(python -m context_long_sequence_ring_gb300.build)")
        L = ctypes.CDLL(LIB)
        for name, args in SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = _c.c_int
        for name in STRING_FUNCS:
            getattr(L, name).restype = _c.c_char_p
            getattr(L, name).argtypes = []
        _lib = L
    return _lib


def last_error() -> str:
    return lib().ra_last_error().decode()


def version() -> str:
    return lib().ra_version().decode()


def _check(status: int):
    if status != RA_OK:
        raise RingAttnError(status, last_error())


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensor must be on a CUDA device")
        if t is not None and not t.is_contiguous():
            raise ValueError("tensor must be contiguous")


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return RA_BF16
    if t.dtype == torch.float32:
        return RA_F32
    raise ValueError("dtype must be bfloat16 or float32")


def device_status() -> int:
    """Synchronise the current stream and return (and clear) the device error status."""
    return lib().ra_device_status(_stream())


# ---------------------------------------------------------------------- partition

def zigzag_partition(seq_lens: Sequence[int], n_ranks: int, device="cuda"):
    """(perm int32 [G], restore int32 [sum L]) of the head-tail partition."""
    n = len(seq_lens)
    arr = (_i64 * max(n, 1))(*[int(x) for x in seq_lens])
    G, T = _i64(0), _i64(0)
    _check(lib().ra_zigzag_partition(arr, n, n_ranks, None, None, _c.byref(G), _c.byref(T), _stream()))
    perm = torch.empty(G.value, dtype=torch.int32, device=device)
    restore = torch.empty(T.value, dtype=torch.int32, device=device)
    if G.value > 0:
        _check(lib().ra_zigzag_partition(arr, n, n_ranks, _ptr(perm), _ptr(restore), None, None, _stream()))
    return perm, restore


def gather_rows(src: torch.Tensor, idx: torch.Tensor, out: Optional[torch.Tensor] = None):
    """out[i] = src[idx[i]] (zero rows where idx < 0); rows are the first dim."""
    _need_cuda(src, idx, out)
    if idx.dtype != torch.int32:
        raise ValueError("idx must be int32")
    rows = idx.numel()
    if out is None:
        out = torch.empty((rows,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] > 0 else 0
    _check(lib().ra_gather_rows(_ptr(src), src.shape[0], _ptr(idx), _ptr(out), rows, row_bytes, _stream()))
    return out


def rope_gather(src: torch.Tensor, positions: torch.Tensor, idx: Optional[torch.Tensor] = None,
                base: float = 10000.0, out: Optional[torch.Tensor] = None):
    """Rotary position embedding fused with a row gather: out[r] = RoPE(src[idx[r]],
    positions[idx[r]]), zero rows where idx < 0.  src [rows, H, d]; positions int32, one per
    source row.  Without idx the rows keep their order (out may be src: in place)."""
    _need_cuda(src, positions, idx, out)
    if src.dim() != 3:
        raise ValueError("src must be [rows, H, d]")
    if positions.dtype != torch.int32 or (idx is not None and idx.dtype != torch.int32):
        raise ValueError("positions and idx must be int32")
    if positions.numel() != src.shape[0]:
        raise ValueError("one position per source row")
    rows = idx.numel() if idx is not None else src.shape[0]
    if out is None:
        out = torch.empty((rows,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    _check(lib().ra_rope_gather(_ptr(src), src.shape[0], src.shape[1], src.shape[2], _dt(src),
                                _ptr(idx) if idx is not None else None, rows, _ptr(positions), float(base),
                                _ptr(out), _stream()))
    return out


# ---------------------------------------------------------------------- attention

def ring_attn_fwd(q, k, v, causal: bool, n_ranks: int, B: int = 1, scale: Optional[float] = None,
                  layout: str = "natural", o=None, lse=None, variant: int = 0):
    """Ring-order attention forward.  q [B*S, Hq, d], k/v [B*S, Hkv, d] token-major.

    Returns (O [B*S, Hq, d] in q's dtype, LSE float32 [B*S, Hq]).  ``variant`` picks the
    bf16 kernel (0 automatic, 1 one head per CTA, 2 two GQA heads per CTA, 3 two adjacent query
    tiles of one head per CTA)."""
    _need_cuda(q, k, v, o, lse)
    rows, Hq, d = q.shape
    Hkv = k.shape[1]
    if rows % B != 0:
        raise ValueError("rows of q must be a multiple of B")
    S = rows // B
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((rows, Hq), dtype=torch.float32, device=q.device)
    _check(lib().ra_ring_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, S, d, _dt(q),
                                     1 if causal else 0, n_ranks, float(scale or 0.0), LAYOUTS[layout], variant,
                                     _stream()))
    return o, lse


def ring_schedule_counts(S: int, n_ranks: int, causal: bool, kv_tile: int = 128, device="cuda"):
    """Per rank: (unmasked, causally masked, skipped) (query tile, key tile) pairs of the kernels' schedule."""
    out = torch.empty((n_ranks, 3), dtype=torch.int64, device=device)
    _check(lib().ra_ring_schedule_counts_ex(S, n_ranks, 1 if causal else 0, kv_tile, _ptr(out), _stream()))
    return out


def ring_attn_fwd_varlen(q, k, v, seq_lens: Sequence[int], causal: bool, n_ranks: int,
                         scale: Optional[float] = None, o=None, lse=None):
    """Ring-order attention over requests of different lengths, on the head-tail gathered layout
    (``zigzag_partition(seq_lens, n_ranks)`` then ``gather_rows``).  q [G, Hq, d], k/v [G, Hkv, d]
    bf16 with G the padded total; returns (O [G, Hq, d], LSE float32 [G, Hq]) in the same order."""
    _need_cuda(q, k, v, o, lse)
    rows, Hq, d = q.shape
    n = len(seq_lens)
    G = sum(-(-int(L) // (2 * n_ranks)) * 2 * n_ranks for L in seq_lens)
    if rows != G or k.shape[0] != G or v.shape[0] != G:
        raise ValueError("q, k, v must have the %d rows of the padded gathered layout" % G)
    arr = (_i64 * max(n, 1))(*[int(x) for x in seq_lens])
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((rows, Hq), dtype=torch.float32, device=q.device)
    _check(lib().ra_ring_attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), arr, n, Hq, k.shape[1], d,
                                         _dt(q), 1 if causal else 0, n_ranks, float(scale or 0.0), _stream()))
    return o, lse


def ring_step_fwd(q, k, v, n_ranks: int, rank: int, src: int, causal: bool, o_in=None, lse_in=None,
                  o_out=None, lse_out=None, B: int = 1, scale: Optional[float] = None):
    """One ring step of rank ``rank``: its local queries q [B*2c, Hq, d] (chunks rank and 2N-1-rank
    of each sequence) against the held block k/v [B*2c, Hkv, d] of rank ``src``, folded into the
    running result (o_in fp32 [B*2c, Hq, d], lse_in [B*2c, Hq]; None at the first step).  o_out
    (fp32 or bf16; may be o_in when fp32) and lse_out (may be lse_in) receive the result; fp32
    buffers are made when they are not given.  Returns (o_out, lse_out)."""
    _need_cuda(q, k, v, o_in, lse_in, o_out, lse_out)
    rows, Hq, d = q.shape
    if rows % (2 * B) != 0 or k.shape[0] != rows or v.shape[0] != rows:
        raise ValueError("q, k, v must hold B sequences of 2c local rows each")
    if o_out is None:
        o_out = torch.empty((rows, Hq, d), dtype=torch.float32, device=q.device)
    if lse_out is None:
        lse_out = torch.empty((rows, Hq), dtype=torch.float32, device=q.device)
    _check(lib().ra_ring_step_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, k.shape[1], rows // (2 * B), d, n_ranks, rank,
                                  src, 1 if causal else 0, float(scale or 0.0), _ptr(o_in), _ptr(lse_in),
                                  _ptr(o_out), _dt(o_out), _ptr(lse_out), _stream()))
    return o_out, lse_out


def ring_step_fn(n_ranks: int, rank: int, causal: bool, B: int = 1, scale: Optional[float] = None):
    """The step callable of ``cp_dist.ring_attention`` for rank ``rank``, on ra_ring_step_fwd."""
    def step(q, k, v, src, o_in, lse_in, o_out, lse_out):
        ring_step_fwd(q, k, v, n_ranks, rank, src, causal, o_in, lse_in, o_out, lse_out, B=B, scale=scale)
    return step


def attn_block_fwd(q, k, v, q_pos0: int, k_pos0: int, causal: bool, scale: Optional[float] = None,
                   o_part=None, lse_part=None):
    """Partial attention of q [Tq, Hq, d] (positions q_pos0..) over k/v [Tk, Hkv, d] (positions k_pos0..)
    -> (O_part fp32 [Tq, Hq, d], LSE_part [Tq, Hq]); -inf / 0 for rows with no visible key."""
    _need_cuda(q, k, v, o_part, lse_part)
    Tq, Hq, d = q.shape
    Tk, Hkv, _ = k.shape
    if o_part is None:
        o_part = torch.empty((Tq, Hq, d), dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty((Tq, Hq), dtype=torch.float32, device=q.device)
    _check(lib().ra_attn_block_fwd(_ptr(q), _ptr(k), _ptr(v), Tq, Tk, Hq, Hkv, d, int(q_pos0), int(k_pos0),
                                   1 if causal else 0, float(scale or 0.0), _ptr(o_part), _ptr(lse_part),
                                   _stream()))
    return o_part, lse_part


def segmented_prefill_fwd(q, k, v, q_pos0: int, seg_tokens: int, causal: bool = True,
                          scale: Optional[float] = None, out_dtype=torch.bfloat16, workspace=None, o=None, lse=None):
    """Chunked prefill of q [Tq, Hq, d] (positions q_pos0..) over k/v [Tk, Hkv, d] (positions 0..) in
    key segments of seg_tokens -> (O [Tq, Hq, d], LSE [Tq, Hq]).  O takes out_dtype, or the dtype of a
    given ``o``."""
    _need_cuda(q, k, v, workspace, o, lse)
    Tq, Hq, d = q.shape
    Tk, Hkv, _ = k.shape
    n = _sz(0)
    _check(lib().ra_segmented_prefill_workspace_size(Tq, Tk, Hq, d, seg_tokens, _c.byref(n)))
    if workspace is None:
        workspace = torch.empty(n.value, dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty((Tq, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, device=q.device)
    out_dtype = o.dtype
    _check(lib().ra_segmented_prefill_fwd(_ptr(q), _ptr(k), _ptr(v), Tq, Tk, Hq, Hkv, d, int(q_pos0),
                                          1 if causal else 0, float(scale or 0.0), seg_tokens, _ptr(o),
                                          RA_BF16 if out_dtype == torch.bfloat16 else RA_F32, _ptr(lse),
                                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream()))
    return o, lse


def allgather_attend_fn(seq_len: int, n_ranks: int, rank: int, causal: bool = True, B: int = 1,
                        seg_tokens: int = 32768, scale: Optional[float] = None):
    """The attend callable of ``cp_dist.allgather_kv_attention`` for rank ``rank``: each of its local
    chunks (per sequence chunk rank and chunk 2N-1-rank, c = seq_len/2N rows each) attends over the
    sequence's keys in token order, in key segments of seg_tokens (ra_segmented_prefill_fwd), into
    the rank's output rows."""
    c = seq_len // (2 * n_ranks)

    def attend(q, k_nat, v_nat, o, lse):
        for b in range(B):
            for half, ch in enumerate((rank, 2 * n_ranks - 1 - rank)):
                rows = slice((b * 2 + half) * c, (b * 2 + half + 1) * c)
                tk = (ch + 1) * c if causal else seq_len      # keys after the chunk are never visible
                keys = slice(b * seq_len, b * seq_len + tk)
                segmented_prefill_fwd(q[rows], k_nat[keys], v_nat[keys], ch * c, seg_tokens, causal, scale,
                                      o=o[rows], lse=lse[rows])
    return attend


def lse_merge(o_parts, lse_parts, out_dtype=torch.float32, o=None, lse=None):
    """Merge partials o_parts [P, T, H, d] fp32 with lse_parts [P, T, H] -> (O [T, H, d], LSE [T, H]).
    O takes out_dtype, or the dtype of a given ``o``."""
    _need_cuda(o_parts, lse_parts, o, lse)
    P, T, H, d = o_parts.shape
    if o is None:
        o = torch.empty((T, H, d), dtype=out_dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=o_parts.device)
    _check(lib().ra_lse_merge(_ptr(o_parts), _ptr(lse_parts), P, T, H, d, _ptr(o),
                              RA_BF16 if o.dtype == torch.bfloat16 else RA_F32, _ptr(lse), _stream()))
    return o, lse


# ---------------------------------------------------------------------- KV cache

def cp_slot_mapping(query_start_loc, positions, block_table, block_size: int, interleave: int, pcp: int,
                    dcp: int, out=None):
    _need_cuda(query_start_loc, positions, block_table, out)
    R = query_start_loc.numel() - 1
    T = positions.numel()
    W = pcp * dcp
    if out is None:
        out = torch.empty((W, T), dtype=torch.int32, device=positions.device)
    _check(lib().ra_cp_slot_mapping(_ptr(query_start_loc), _ptr(positions), _ptr(block_table),
                                    block_table.shape[1], R, T, block_size, interleave, pcp, dcp, _ptr(out),
                                    _stream()))
    return out


def cp_kv_scatter(k, v, slot, k_cache, v_cache):
    _need_cuda(k, v, slot, k_cache, v_cache)
    W, NB, Hkv, bs, d = k_cache.shape
    _check(lib().ra_cp_kv_scatter(_ptr(k), _ptr(v), _ptr(slot), _ptr(k_cache), _ptr(v_cache), k.shape[0], W, Hkv,
                                  d, bs, NB, _dt(k), _stream()))


def cp_kv_gather(k_cache, v_cache, block_table, query_start_loc, positions, interleave: int, pcp: int, dcp: int,
                 k_out=None, v_out=None):
    """Token rows out of the sharded cache: row t = token positions[t] of its request -> (k [T, Hkv, d], v)."""
    _need_cuda(k_cache, v_cache, block_table, query_start_loc, positions, k_out, v_out)
    W, NB, Hkv, bs, d = k_cache.shape
    T = positions.numel()
    if k_out is None:
        k_out = torch.empty((T, Hkv, d), dtype=k_cache.dtype, device=k_cache.device)
    if v_out is None:
        v_out = torch.empty_like(k_out)
    _check(lib().ra_cp_kv_gather(_ptr(k_cache), _ptr(v_cache), _ptr(block_table), block_table.shape[1],
                                 _ptr(query_start_loc), _ptr(positions), query_start_loc.numel() - 1, T, Hkv, d, bs,
                                 interleave, pcp, dcp, NB, _dt(k_cache), _ptr(k_out), _ptr(v_out), _stream()))
    return k_out, v_out


def cp_decode_workspace_size(R, Hq, d, max_vblocks, pcp, dcp, split_blocks) -> int:
    n = _sz(0)
    _check(lib().ra_cp_decode_workspace_size(R, Hq, d, max_vblocks, pcp, dcp, split_blocks, _c.byref(n)))
    return n.value


def cp_decode(q, k_cache, v_cache, block_table, ctx_lens, interleave: int, pcp: int, dcp: int,
              split_blocks: int = 8, scale: Optional[float] = None, out_dtype=torch.bfloat16,
              workspace=None, o=None, lse=None):
    """Decode of one query token per request over the sharded cache -> (O [R, Hq, d], LSE [R, Hq])."""
    _need_cuda(q, k_cache, v_cache, block_table, ctx_lens, workspace, o, lse)
    R, Hq, d = q.shape
    W, NB, Hkv, bs, _ = k_cache.shape
    if W != pcp * dcp:
        raise ValueError("cache has %d devices, pcp*dcp = %d" % (W, pcp * dcp))
    max_vb = block_table.shape[1]
    need = cp_decode_workspace_size(R, Hq, d, max_vb, pcp, dcp, split_blocks)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if o is None:
        o = torch.empty((R, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((R, Hq), dtype=torch.float32, device=q.device)
    _check(lib().ra_cp_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), R, Hq, Hkv,
                              d, bs, interleave, pcp, dcp, max_vb, NB, float(scale or 0.0), split_blocks, _ptr(o),
                              RA_BF16 if o.dtype == torch.bfloat16 else RA_F32, _ptr(lse), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream()))
    return o, lse


def cp_decode_noalloc(q, k_cache, v_cache, block_table, ctx_lens, interleave: int, pcp: int, dcp: int,
                      split_blocks: int = 8, scale: Optional[float] = None, out_dtype=torch.bfloat16, o=None,
                      lse=None):
    """cp_decode without a workspace, for callers that cannot allocate device memory on the decode
    path: the partials live in a fixed 32 MiB scratch array inside the library (shared by all
    calls; calls that overlap on the GPU race).  Outputs o/lse may be passed in preallocated."""
    _need_cuda(q, k_cache, v_cache, block_table, ctx_lens, o, lse)
    R, Hq, d = q.shape
    W, NB, Hkv, bs, _ = k_cache.shape
    if o is None:
        o = torch.empty((R, Hq, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((R, Hq), dtype=torch.float32, device=q.device)
    _check(lib().ra_cp_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), R,
                                      Hq, Hkv, d, bs, interleave, pcp, dcp, block_table.shape[1], NB,
                                      float(scale or 0.0), split_blocks, _ptr(o),
                                      RA_BF16 if o.dtype == torch.bfloat16 else RA_F32, _ptr(lse), _stream()))
    return o, lse


def cp_decode_partials(q, k_cache, v_cache, block_table, ctx_lens, interleave: int, pcp: int, dcp: int,
                       dev0: int = 0, split_blocks: int = 8, scale: Optional[float] = None, o_parts=None,
                       lse_parts=None):
    """Split-KV partials of the devices whose shards k_cache/v_cache [n_dev, NB, Hkv, bs, d] hold
    (devices dev0 .. dev0+n_dev-1 of pcp*dcp) -> (O_parts fp32 [P, R, Hq, d], LSE_parts [P, R, Hq]),
    partial p = (w - dev0) * n_splits + s.  A partial with LSE -inf has no token and unwritten O."""
    _need_cuda(q, k_cache, v_cache, block_table, ctx_lens, o_parts, lse_parts)
    R, Hq, d = q.shape
    n_dev, NB, Hkv, bs, _ = k_cache.shape
    max_vb = block_table.shape[1]
    P = _i32(0)
    args = (_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), R, Hq, Hkv, d, bs, interleave,
            pcp, dcp, dev0, n_dev, max_vb, NB, float(scale or 0.0), split_blocks)
    _check(lib().ra_cp_decode_partials(*args, None, None, _c.byref(P), _stream()))
    if o_parts is None:
        o_parts = torch.empty((P.value, R, Hq, d), dtype=torch.float32, device=q.device)
    if lse_parts is None:
        lse_parts = torch.empty((P.value, R, Hq), dtype=torch.float32, device=q.device)
    _check(lib().ra_cp_decode_partials(*args, _ptr(o_parts), _ptr(lse_parts), None, _stream()))
    return o_parts, lse_parts


def cp_lse_rescale(o_local, lse_all, w: int, o_scaled=None, lse_total=None):
    """Step 2 of cp_lse_ag_out_rs on device w: o_local fp32 [R, Hq, d], lse_all [W, R, Hq] ->
    (o_scaled [W, R, Hq/W, d], lse_total [R, Hq/W])."""
    _need_cuda(o_local, lse_all, o_scaled, lse_total)
    R, Hq, d = o_local.shape
    W = lse_all.shape[0]
    if o_scaled is None:
        o_scaled = torch.empty((W, R, Hq // W, d), dtype=torch.float32, device=o_local.device)
    if lse_total is None:
        lse_total = torch.empty((R, Hq // W), dtype=torch.float32, device=o_local.device)
    _check(lib().ra_cp_lse_rescale(_ptr(o_local), _ptr(lse_all), W, w, R, Hq, d, _ptr(o_scaled), _ptr(lse_total),
                                   _stream()))
    return o_scaled, lse_total


def cp_head_split(o_local, lse_local, W: int, o_split=None, lse_split=None):
    """All-to-all form of the decode merge: o_local fp32 [R, Hq, d], lse_local [R, Hq] ->
    (o_split [W, R, Hq/W, d], lse_split [W, R, Hq/W]) laid out by the device that keeps each head."""
    _need_cuda(o_local, lse_local, o_split, lse_split)
    R, Hq, d = o_local.shape
    if o_split is None:
        o_split = torch.empty((W, R, Hq // W, d), dtype=torch.float32, device=o_local.device)
    if lse_split is None:
        lse_split = torch.empty((W, R, Hq // W), dtype=torch.float32, device=o_local.device)
    _check(lib().ra_cp_head_split(_ptr(o_local), _ptr(lse_local), W, R, Hq, d, _ptr(o_split), _ptr(lse_split),
                                  _stream()))
    return o_split, lse_split


def cp_head_split_fn():
    """The split callable of ``cp_dist.cp_lse_a2a``, on ra_cp_head_split."""
    def split(o_local, lse_local, W, o_split, lse_split):
        cp_head_split(o_local, lse_local, W, o_split, lse_split)
    return split


def lse_merge_fn(out_dtype=torch.float32):
    """The merge callable of ``cp_dist.cp_lse_a2a``, on ra_lse_merge."""
    def merge(o_parts, lse_parts, o, lse):
        lse_merge(o_parts, lse_parts, out_dtype=out_dtype, o=o, lse=lse)
    return merge


def cp_lse_rescale_fn():
    """The rescale callable of ``cp_dist.cp_lse_ag_out_rs``, on ra_cp_lse_rescale."""
    def rescale(o_local, lse_all, w, o_scaled, lse_total):
        cp_lse_rescale(o_local, lse_all, w, o_scaled, lse_total)
    return rescale


# ---------------------------------------------------------------------- misc

def selftest_wait_timeout(limit_cycles: int):
    _check(lib().ra_selftest_wait_timeout(int(limit_cycles), _stream()))


_TABLES = {}


def synth_fill(key: int, table_cpu: torch.Tensor, shape, device="cuda"):
    """Device tensor of the counter-based draw (see inputs.py) with the given key and value table."""
    dev = torch.device(device)
    tk = (table_cpu.dtype, dev)
    if tk not in _TABLES:
        _TABLES[tk] = table_cpu.to(dev)
    table = _TABLES[tk]
    out = torch.empty(tuple(shape), dtype=table_cpu.dtype, device=dev)
    _check(lib().ra_synth_fill(_u64(key), out.numel(), _ptr(table), table.element_size(), _ptr(out), _stream()))
    return out
