// Ring schedule of the zigzag (head-tail) partition, shared by the ring
// kernels: which K/V tiles a 128-row query tile meets, in ring order, and the
// causal mask of a (query tile, key tile) pair by original position.
//
// Sources: guijiagi.com "Ring Attention" tag page (ring step t: rank i works on
// the K/V block of rank (i - t) mod N); vLLM-Ascend "Context Parallel (CP)"
// head-tail partition (rank r owns chunks r and 2N-1-r of equal length c).
// Chunks are numbered globally, 0 .. 2N-1, in sequence order.
#pragma once

#include "ra_attn_tc.cuh"

namespace {

struct Sched {
  int N, c, nt, causal;  // ranks, chunk length, 128-row query tiles per chunk, causal flag
  int bnk, ntk;          // key tile length and key tiles per chunk
};

// Iterates the K/V tiles one query tile (chunk qc, tile qi) meets, in ring
// order: ranks s = r, r-1, ..., each rank's head chunk s, then its tail chunk
// 2N-1-s.  Under the causal mask chunks after qc are skipped and, in qc itself,
// only key tiles that start at or before the tile's last query are visited.
struct KvIter {
  int N, ntk, causal, qc, r, diag_lim;
  int t, h, ki;
  __device__ void init(const Sched& s, int qc_, int qi) {
    N = s.N; ntk = s.ntk; causal = s.causal; qc = qc_;
    r = qc < N ? qc : 2 * N - 1 - qc;
    const int q_valid = min(BM, s.c - qi * BM);
    diag_lim = min(ntk, (qi * BM + q_valid - 1) / s.bnk + 1);
    t = 0; h = 0; ki = -1;
  }
  __device__ bool next(int& kc, int& kt) {
    while (t < N) {
      const int s = r - t < 0 ? r - t + N : r - t;  // rank whose block is held at step t ((r-t) mod N
                                                      // without an integer division, which costs the
                                                      // softmax warps about 1 % of the kernel)
      const int ch = h == 0 ? s : 2 * N - 1 - s;  // its head, then its tail chunk
      const int lim = !causal ? ntk : (ch < qc ? ntk : (ch == qc ? diag_lim : 0));
      ++ki;
      if (ki < lim) { kc = ch; kt = ki; return true; }
      ki = -1;
      if (++h == 2) { h = 0; ++t; }
    }
    return false;
  }
};

__device__ __forceinline__ int n_kv_tiles(const Sched& s, int qc, int qi) {
  if (!s.causal) return 2 * s.N * s.ntk;
  const int q_valid = min(BM, s.c - qi * BM);
  return qc * s.ntk + min(s.ntk, (qi * BM + q_valid - 1) / s.bnk + 1);
}

// Causal mask of key tile (kc, kt) for query row `row` of tile (qc, qi):
// the number of leading visible columns and whether any column is masked.
__device__ __forceinline__ void tile_mask(const Sched& s, int qc, int qi, int kc, int kt, int row, int& col_lim,
                                          bool& masked) {
  const int kv_valid = min(s.bnk, s.c - kt * s.bnk);
  const bool same = s.causal && kc == qc;
  col_lim = same ? min(kv_valid, qi * BM + row - kt * s.bnk + 1) : kv_valid;
  masked = (same && kt * s.bnk + kv_valid - 1 > qi * BM) || kv_valid < s.bnk;
}

}  // namespace
