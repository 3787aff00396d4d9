"""Head-tail (zigzag) token partition and its restore index.  Test
infrastructure only.

Source: vLLM-Ascend developer guide "Context Parallel (CP)", section
"Prefill context parallel (PCP)" / head-tail token partition: each sequence is
padded to a multiple of 2*pcp, cut into 2*pcp equal parts, part i is paired
with part 2*pcp-1-i and the pair goes to one device; because an all-gather of
the per-device buffers interleaves requests, an index restoring the original
order is computed (pcp_allgather_restore_idx).

Readings where the page is silent or garbled (also listed in the design notes):
* "pad to length 2*pcp" is read as "pad to a multiple of 2*pcp";
* rank r stores chunk r first, then chunk 2N-1-r;
* gathered order = rank-major, then request, then (chunk r, chunk 2N-1-r),
  which is what concatenating every rank's buffer (each holding all requests
  in order) produces;
* original tokens are packed request after request without padding; a padded
  position has perm = -1;
* restore[i] is the gathered position of original token i (perm^-1).

Parity status: pinned (hand-worked example, bijection and round-trip tests).
"""

from __future__ import annotations

import numpy as np


def zigzag_partition(seq_lens, n_ranks: int):
    """Return (perm [G], restore [sum L], padded_lens [R]) as int64 arrays."""
    N = int(n_ranks)
    if N < 1:
        raise ValueError("n_ranks must be >= 1")
    L = [int(x) for x in seq_lens]
    if any(x < 0 for x in L):
        raise ValueError("negative sequence length")
    Lp = [-(-x // (2 * N)) * (2 * N) for x in L]          # pad to a multiple of 2N
    c = [x // (2 * N) for x in Lp]                          # chunk length per request
    start = np.concatenate([[0], np.cumsum(L)]).astype(np.int64)
    pieces = []
    for r in range(N):                                      # rank-major
        for q in range(len(L)):                             # then request
            for chunk in (r, 2 * N - 1 - r):                # head part, then tail part
                p = chunk * c[q] + np.arange(c[q], dtype=np.int64)
                pieces.append(np.where(p < L[q], start[q] + p, -1))
    perm = np.concatenate(pieces) if pieces else np.zeros(0, dtype=np.int64)
    restore = np.full(int(start[-1]), -1, dtype=np.int64)
    g = np.nonzero(perm >= 0)[0]
    restore[perm[g]] = g
    return perm.astype(np.int64), restore, np.asarray(Lp, dtype=np.int64)


def gather_rows(src, idx):
    """dst[i] = src[idx[i]], or a zero row where idx[i] < 0."""
    src = np.asarray(src)
    idx = np.asarray(idx, dtype=np.int64)
    dst = np.zeros((len(idx),) + src.shape[1:], dtype=src.dtype)
    ok = idx >= 0
    dst[ok] = src[idx[ok]]
    return dst
