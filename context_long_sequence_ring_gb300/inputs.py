"""Seeded synthetic inputs shared by the tests, ``bench.py`` and ``smoke()``.

This module holds no attention, softmax, partition or cache-addressing
arithmetic: it only draws numbers.  Both the CUDA path and the float64 oracle
receive tensors built here (or, for device-resident tensors too large to build
on the host, the same values produced on the GPU by the library's
``ra_synth_fill`` kernel from the same counter-based definition below).

Generator definition (counter-based, so any element can be drawn on its own):

* ``mix64`` is the SplitMix64 output finaliser (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014): two
  xor-shift-multiply rounds with the published constants and a final xor-shift.
* A tensor is named by ``(seed, tensor_id)``; its key is
  ``mix64((seed * GOLDEN) ^ (tensor_id << 32))`` (all arithmetic mod 2**64).
* Element ``i`` (flat index in the tensor's logical, row-major layout) draws
  ``u = mix64(key + (i + 1) * GOLDEN)``.
* The value is ``TABLE[u >> 48]``, where ``TABLE[j]`` is the standard normal
  quantile of ``(j + 0.5) / 65536`` (float64), rounded once to the tensor's
  dtype (round-to-nearest-even).  Values are therefore N(0, 1) quantised to
  65536 equiprobable levels, with tails cut near +/-4.3.

Integer inputs (context lengths, block-table permutations) use
``torch.Generator().manual_seed(seed)``.
"""

from __future__ import annotations

from statistics import NormalDist

import numpy as np
import torch

GOLDEN = 0x9E3779B97F4A7C15
MIX_C1 = 0xBF58476D1CE4E5B9
MIX_C2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1

# tensor ids within one seed
TID_Q, TID_K, TID_V = 0, 1, 2


def _mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX_C1) & MASK64
    z = ((z ^ (z >> 27)) * MIX_C2) & MASK64
    return z ^ (z >> 31)


def tensor_key(seed: int, tensor_id: int) -> int:
    """64-bit key of tensor ``tensor_id`` drawn under ``seed``."""
    return _mix64_int(((seed * GOLDEN) & MASK64) ^ ((tensor_id << 32) & MASK64))


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    z ^= z >> np.uint64(30)
    z *= np.uint64(MIX_C1)
    z ^= z >> np.uint64(27)
    z *= np.uint64(MIX_C2)
    z ^= z >> np.uint64(31)
    return z


def draw_u16(key: int, flat_index: np.ndarray) -> np.ndarray:
    """Top 16 bits of ``mix64(key + (i + 1) * GOLDEN)`` for each index ``i``."""
    i = np.asarray(flat_index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(key) + (i + np.uint64(1)) * np.uint64(GOLDEN)
    return (_mix64_np(z) >> np.uint64(48)).astype(np.int64)


_TABLE_CACHE: dict = {}


def normal_table(dtype: torch.dtype) -> torch.Tensor:
    """The 65536-entry quantile table, rounded once to ``dtype`` (CPU tensor)."""
    if dtype not in _TABLE_CACHE:
        nd = NormalDist()
        t64 = torch.tensor([nd.inv_cdf((j + 0.5) / 65536.0) for j in range(65536)],
                           dtype=torch.float64)
        _TABLE_CACHE[dtype] = t64.to(dtype)
    return _TABLE_CACHE[dtype]


def synth_normal(seed: int, tensor_id: int, shape, dtype: torch.dtype,
                 chunk: int = 1 << 16) -> torch.Tensor:
    """Whole tensor of the counter-based N(0,1) draw (CPU)."""
    n = int(np.prod(shape)) if len(shape) else 1
    key = tensor_key(seed, tensor_id)
    table = normal_table(dtype)
    out = torch.empty(n, dtype=dtype)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        u = draw_u16(key, np.arange(s, e, dtype=np.uint64))
        out[s:e] = table[torch.from_numpy(u)]
    return out.reshape(shape)


def synth_normal_at(seed: int, tensor_id: int, flat_index: np.ndarray,
                    dtype: torch.dtype) -> torch.Tensor:
    """Selected elements (by flat index) of the counter-based N(0,1) draw."""
    key = tensor_key(seed, tensor_id)
    u = draw_u16(key, np.asarray(flat_index, dtype=np.uint64).ravel())
    return normal_table(dtype)[torch.from_numpy(u)].reshape(np.shape(flat_index))


def synth_rows(seed: int, tensor_id: int, rows: np.ndarray, row_elems: int,
               dtype: torch.dtype) -> torch.Tensor:
    """Rows ``rows`` of a row-major tensor with ``row_elems`` elements per row."""
    rows = np.asarray(rows, dtype=np.int64)
    idx = rows[:, None] * row_elems + np.arange(row_elems, dtype=np.int64)[None, :]
    return synth_normal_at(seed, tensor_id, idx.astype(np.uint64), dtype)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

def prefill_inputs(seed: int, B: int, S: int, Hq: int, Hkv: int, d: int,
                   dtype: torch.dtype):
    """Q [B*S, Hq, d], K/V [B*S, Hkv, d], token-major natural order (CPU)."""
    q = synth_normal(seed, TID_Q, (B * S, Hq, d), dtype)
    k = synth_normal(seed, TID_K, (B * S, Hkv, d), dtype)
    v = synth_normal(seed, TID_V, (B * S, Hkv, d), dtype)
    return q, k, v


def decode_workload(seed: int, R: int, ctx_lo: int, ctx_hi: int, block_size: int,
                    pcp: int, dcp: int):
    """Context lengths, request token offsets and a shuffled block table.

    Context lengths are uniform integers in [ctx_lo, ctx_hi].  Each request
    owns ceil(L / (block_size*pcp*dcp)) virtual blocks; the physical block ids
    are a seeded random permutation of the pool, handed out request by request.
    Returns a dict of CPU int tensors plus sizes.
    """
    g = torch.Generator().manual_seed(seed)
    ctx = torch.randint(ctx_lo, ctx_hi + 1, (R,), generator=g, dtype=torch.int64)
    vbs = block_size * pcp * dcp
    nvb = [(int(L) + vbs - 1) // vbs for L in ctx]
    num_blocks = sum(nvb)
    max_vb = max(nvb)
    ids = torch.randperm(num_blocks, generator=g).to(torch.int32)
    bt = torch.full((R, max_vb), -1, dtype=torch.int32)
    pos = 0
    for r in range(R):
        bt[r, :nvb[r]] = ids[pos:pos + nvb[r]]
        pos += nvb[r]
    tok_start = torch.zeros(R + 1, dtype=torch.int64)
    tok_start[1:] = torch.cumsum(ctx, 0)
    return {"ctx_lens": ctx.to(torch.int32), "block_table": bt, "num_blocks": num_blocks,
            "max_vblocks": max_vb, "tok_start": tok_start,
            "total_tokens": int(tok_start[-1])}


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = [
    "GOLDEN", "TID_Q", "TID_K", "TID_V", "tensor_key", "draw_u16", "normal_table",
    "synth_normal", "synth_normal_at", "synth_rows", "prefill_inputs",
    "decode_workload", "ceil_div",
]
