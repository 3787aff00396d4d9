// Two-head tcgen05 attention pipeline shared by the ring-order kernel and the
// block-partial kernel.  A schedule policy Pol supplies (device side):
//   Pol(const Args&, int item)          decode the CTA's work item
//   int tiles()                          query tiles of the CTA, one after the other (0, 1 or 2)
//   int kvh()                            the K/V head both slots read
//   void set_tile(int ti)                select query tile ti
//   int q_head(int h); int32_t q_row(int h); int q_valid(int h)
//                                        slot h (0, 1) of the tile: its query head, the TMA
//                                        row of its first query and its valid rows (two heads
//                                        of a GQA group, or two adjacent query tiles of one head)
//   int n_kv()                           K/V tiles the query tile meets
//   KvPos; kv_begin(KvPos&); bool kv_next(KvPos&)   those tiles in order (KvPos::row = TMA row)
//   void mask(const KvPos&, int h, int row, int& col_lim, bool& masked)
//   void store_o(int h, int row, int col0, const uint32_t (&o)[32], float inv_l)
//   void store_lse(int h, int row, float lse)
//   void write_empty(int tid, int nthreads)   outputs of a CTA with no query tile to run (tiles() == 0)
//   void skipped_rows(int h, int row)    outputs of slot h, row `row` of the CTA's query tiles that
//                                        tiles() leaves out (called once per softmax thread first)
//   void prepare_row(int h, int row, float lse2, float inv_l)
//                                        called before the store_o calls of a stored row, with the
//                                        row's log2-sum-exp (-inf if it saw no key)
// and Args carries scale_log2 and wait_limit.  PolicyDefaults gives the last two as no-ops.
#pragma once

#include "ra_attn_tc.cuh"

namespace {
using namespace ra::sm100;

// ===========================================================================
// Two-slot tcgen05 attention kernel, templated on a schedule policy: a CTA
// runs two 128-row query tiles ("slots") that read the same K/V tiles, so
// every K/V tile TMA brings in feeds two score tiles.  The slots are two query
// heads of one GQA group at the same rows, or two adjacent query tiles of one
// head (which meet the same keys up to one diagonal tile).  The policy
// supplies the slots, the K/V tiles they meet (and in which order), the causal
// mask and where the output goes: ring order over virtual ranks for the ring
// kernel, a plain key range at absolute positions for block partials.
// Roles (384 threads): warp 0 TMA, warp 1 TMEM allocation + MMA issue, warps
// 4..7 softmax of slot 0, warps 8..11 softmax of slot 1 (warps 2, 3 idle).
// Tensor memory: S_h = cols [128h, 128h+128), O_h = cols [256+128h, ...).
// P_h (bf16, two per column) overwrites the first 64 columns of S_h and is
// the A operand of O_h += P_h V straight from tensor memory, so P never
// touches shared memory.  One thread issues every MMA, in the order
//   PV0_j, S0_{j+1}, PV1_j, S1_{j+1}
// which staggers the two slots: each softmax warpgroup works while the tensor
// core serves the other slot (measured faster than one issuer per slot).
// tcgen05 operations of one thread execute in issue order, so S_h(j+1) may
// overwrite the columns PV_h(j) reads.  A softmax warpgroup only waits for
// the previous P.V when it must rescale O (lazy rescale, threshold 2^8).
// ===========================================================================
// No-op defaults of the two optional policy hooks.
struct PolicyDefaults {
  __device__ void skipped_rows(int, int) const {}
  __device__ void prepare_row(int, int, float, float) {}
};

template <int D>
struct __align__(1024) Smem2 {
  uint8_t q[2][BM * D * 2];
  uint8_t k[STAGES][BN * D * 2];
  uint8_t v[STAGES][BN * D * 2];
  uint64_t q_full, q_empty, k_full[STAGES], k_empty[STAGES], v_full[STAGES], v_empty[STAGES];
  uint64_t s_full[2], p_full[2], pv_done[2], o_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kThreads2 = 384;

template <int D, class Pol>
__global__ void __launch_bounds__(kThreads2, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ typename Pol::Args args) {
  constexpr int SLABS = D / 64;
  constexpr uint32_t kTileBytes = BM * D * 2;
  constexpr uint32_t kIdescS = idesc_bf16_f32(BM, BN, 0, 0);
  constexpr uint32_t kIdescO = idesc_bf16_f32(BM, D, 0, 1);

  extern __shared__ uint8_t smem_raw[];
  Smem2<D>& sm = *reinterpret_cast<Smem2<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Pol pol(args, blockIdx.x);
  const int n_tiles = pol.tiles();
  if (n_tiles == 0) {  // nothing visible: the policy writes the empty result
    pol.write_empty(threadIdx.x, blockDim.x);
    return;
  }
  volatile int* abort_flag = &sm.abort_flag;
  const long long lim = args.wait_limit;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    mbar_init(smem_u32(&sm.q_empty), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.k_empty[s]), 1);
      mbar_init(smem_u32(&sm.v_full[s]), 1);
      mbar_init(smem_u32(&sm.v_empty[s]), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(smem_u32(&sm.s_full[h]), 1);
      mbar_init(smem_u32(&sm.p_full[h]), 128);
      mbar_init(smem_u32(&sm.pv_done[h]), 1);
      mbar_init(smem_u32(&sm.o_empty[h]), 128);
    }
    mbar_init(smem_u32(&sm.drain), 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint32_t kv_cnt = 0;
      // copies issued so far (stage phase of the last one), awaited before an aborted CTA exits
      bool q_iss = false, k_iss[STAGES] = {false, false}, v_iss[STAGES] = {false, false};
      uint32_t q_ph = 0, k_ph[STAGES] = {0, 0}, v_ph[STAGES] = {0, 0};
      bool ok = true;
      for (int ti = 0; ti < n_tiles && ok; ++ti) {
        pol.set_tile(ti);
        if (!(ok = mbar_wait(smem_u32(&sm.q_empty), (ti & 1) ^ 1, abort_flag, lim, 101))) break;
        const uint32_t qb = smem_u32(&sm.q_full);
        mbar_arrive_expect_tx(qb, 2 * kTileBytes);
        for (int h = 0; h < 2; ++h) {
          const int32_t qrow = pol.q_row(h);
          for (int s = 0; s < SLABS; ++s)
            tma_load_3d(smem_u32(sm.q[h] + s * BM * 128), &tmQ, qb, 64 * s, pol.q_head(h), qrow);
        }
        q_iss = true;
        q_ph = ti & 1;
        typename Pol::KvPos kp;
        pol.kv_begin(kp);
        while (pol.kv_next(kp)) {
          const int st = kv_cnt % STAGES;
          const uint32_t ph = (kv_cnt / STAGES) & 1;
          const int32_t krow = kp.row;
          if (!(ok = mbar_wait(smem_u32(&sm.k_empty[st]), ph ^ 1, abort_flag, lim, 102))) break;
          mbar_arrive_expect_tx(smem_u32(&sm.k_full[st]), kTileBytes);
          for (int s = 0; s < SLABS; ++s)
            tma_load_3d(smem_u32(sm.k[st] + s * BN * 128), &tmK, smem_u32(&sm.k_full[st]), 64 * s, pol.kvh(), krow);
          k_iss[st] = true;
          k_ph[st] = ph;
          if (!(ok = mbar_wait(smem_u32(&sm.v_empty[st]), ph ^ 1, abort_flag, lim, 103))) break;
          mbar_arrive_expect_tx(smem_u32(&sm.v_full[st]), kTileBytes);
          for (int s = 0; s < SLABS; ++s)
            tma_load_3d(smem_u32(sm.v[st] + s * BN * 128), &tmV, smem_u32(&sm.v_full[st]), 64 * s, pol.kvh(), krow);
          v_iss[st] = true;
          v_ph[st] = ph;
          ++kv_cnt;
        }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA exits
        if (q_iss) mbar_wait_quiesce(smem_u32(&sm.q_full), q_ph, 1 << 22);
        for (int s = 0; s < STAGES; ++s) {
          if (k_iss[s]) mbar_wait_quiesce(smem_u32(&sm.k_full[s]), k_ph[s], 1 << 22);
          if (v_iss[s]) mbar_wait_quiesce(smem_u32(&sm.v_full[s]), v_ph[s], 1 << 22);
        }
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      uint32_t kv_cnt = 0, pf_cnt[2] = {0, 0};
      bool ok = true;
      // descriptors of k-step 0; a k-step adds its byte offset / 16 to the start-address field
      const uint64_t dq[2] = {desc_sw128(smem_u32(sm.q[0]), 16, 1024), desc_sw128(smem_u32(sm.q[1]), 16, 1024)};
      const uint64_t dk[STAGES] = {desc_sw128(smem_u32(sm.k[0]), 16, 1024), desc_sw128(smem_u32(sm.k[1]), 16, 1024)};
      const uint64_t dv[STAGES] = {desc_sw128(smem_u32(sm.v[0]), BN * 128, 1024),
                                   desc_sw128(smem_u32(sm.v[1]), BN * 128, 1024)};
      // Whether slot 1's P is known to be ready: tested while the last score MMAs of slot 0 are still
      // queued, so that the barrier check overlaps tensor work instead of following it.
      bool p1_ready = false;
      auto issue_s = [&](int h, int st) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off16 = ((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + h * BN, dq[h] + off16, dk[st] + off16, kIdescS, kk > 0 ? 1u : 0u);
          if (h == 0 && kk == D / 16 - 3) p1_ready = mbar_test_wait(smem_u32(&sm.p_full[1]), pf_cnt[1] & 1);
        }
        mma_commit(smem_u32(&sm.s_full[h]));
      };
      auto issue_pv = [&](int h, int st, bool first) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ts(tmem + kColO + h * D, tmem + h * BN + kk * 8, dv[st] + ((kk * 16 * 128) >> 4), kIdescO,
                      (kk > 0 || !first) ? 1u : 0u);
        mma_commit(smem_u32(&sm.pv_done[h]));
      };
      for (int ti = 0; ti < n_tiles && ok; ++ti) {
        pol.set_tile(ti);
        const int nkv = pol.n_kv();
        if (!(ok = mbar_wait(smem_u32(&sm.q_full), ti & 1, abort_flag, lim, 110))) break;
        // prologue: both score tiles of K/V tile 0
        {
          const int st = kv_cnt % STAGES;
          if (!(ok = mbar_wait(smem_u32(&sm.k_full[st]), (kv_cnt / STAGES) & 1, abort_flag, lim, 111))) break;
          tc_fence_after();
          issue_s(0, st);
          issue_s(1, st);
          mma_commit(smem_u32(&sm.k_empty[st]));
          if (nkv == 1) mma_commit(smem_u32(&sm.q_empty));
        }
        for (int j = 0; j < nkv && ok; ++j) {
          const uint32_t c = kv_cnt + j;
          const int st = c % STAGES;
          const uint32_t ph = (c / STAGES) & 1;
          const bool more = j + 1 < nkv;
          const int st1 = (c + 1) % STAGES;
          const uint32_t ph1 = ((c + 1) / STAGES) & 1;
          // The waits that do not depend on the softmax come first, while slot 0's P is still being
          // made: after P_0 lands nothing but the MMAs stands between it and the tensor core.
          if (!(ok = mbar_wait(smem_u32(&sm.v_full[st]), ph, abort_flag, lim, 113))) break;
          if (more && !(ok = mbar_wait(smem_u32(&sm.k_full[st1]), ph1, abort_flag, lim, 115))) break;
          if (j == 0 && !(ok = mbar_wait(smem_u32(&sm.o_empty[0]), (ti & 1) ^ 1, abort_flag, lim, 114))) break;
          if (j == 0 && !(ok = mbar_wait(smem_u32(&sm.o_empty[1]), (ti & 1) ^ 1, abort_flag, lim, 117))) break;
          // O_0 += P_0 V_j, then S_0 of tile j+1
          if (!(ok = mbar_wait(smem_u32(&sm.p_full[0]), pf_cnt[0] & 1, abort_flag, lim, 112))) break;
          ++pf_cnt[0];
          tc_fence_after();
          issue_pv(0, st, j == 0);
          p1_ready = false;
          if (more) issue_s(0, st1);
          // O_1 += P_1 V_j
          if (!p1_ready && !(ok = mbar_wait(smem_u32(&sm.p_full[1]), pf_cnt[1] & 1, abort_flag, lim, 116))) break;
          ++pf_cnt[1];
          tc_fence_after();
          issue_pv(1, st, j == 0);
          mma_commit(smem_u32(&sm.v_empty[st]));
          if (more) {
            issue_s(1, st1);
            mma_commit(smem_u32(&sm.k_empty[st1]));
            if (j + 1 == nkv - 1) mma_commit(smem_u32(&sm.q_empty));
          }
        }
        kv_cnt += nkv;
      }
      mma_commit(smem_u32(&sm.drain));
      if (!mbar_wait_quiesce(smem_u32(&sm.drain), 0, ok ? lim : (1 << 22)) && ok) {
        *abort_flag = 1;
        ra_record_error(RA_ERR_TIMEOUT, 118);
      }
    }
  } else if (warp >= 4) {
    // ============================================================ softmax + epilogue (head h)
    const int h = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t colS = h * BN, colO = kColO + h * D;
    uint32_t s_cnt = 0, pv_base = 0;
    bool ok = true;
    pol.skipped_rows(h, row);
    for (int ti = 0; ti < n_tiles && ok; ++ti) {
      pol.set_tile(ti);
      const int q_valid = pol.q_valid(h);
      const int nkv = pol.n_kv();
      typename Pol::KvPos kp;
      pol.kv_begin(kp);
      float m = -CUDART_INF_F, l = 0.f;
      for (int j = 0; j < nkv; ++j) {
        pol.kv_next(kp);
        if (!(ok = mbar_wait(smem_u32(&sm.s_full[h]), s_cnt & 1, abort_flag, lim, 120 + h))) break;
        ++s_cnt;
        tc_fence_after();
        int col_lim;
        bool masked;
        pol.mask(kp, h, row, col_lim, masked);
        uint32_t pk[BN / 2];
        const float alpha = softmax_row(t_lane + colS, j, masked, col_lim, args.scale_log2, m, l, pk);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O_h must hold P_{j-1} V_{j-1} before it is rescaled
          if (!(ok = mbar_wait(smem_u32(&sm.pv_done[h]), (pv_base + j - 1) & 1, abort_flag, lim, 124 + h))) break;
          tc_fence_after();
#pragma unroll
          for (int c4 = 0; c4 < D / 32; ++c4) {
            uint32_t orr[32];
            tmem_ld32(t_lane + colO + 32 * c4, orr);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tmem_st32(t_lane + colO + 32 * c4, orr);
          }
        }
        // P_h into the first 64 columns of S_h
        tmem_st32(t_lane + colS, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
        tmem_st32(t_lane + colS + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.p_full[h]));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = mbar_wait(smem_u32(&sm.pv_done[h]), (pv_base + nkv - 1) & 1, abort_flag, lim, 126 + h))) break;
      pv_base += nkv;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool row_ok = row < q_valid;
      if (row_ok) pol.prepare_row(h, row, l > 0.f ? m + log2f(l) : -CUDART_INF_F, inv_l);
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t orr[32];
        tmem_ld32(t_lane + colO + 32 * c4, orr);
        tmem_wait_ld();
        if (row_ok) pol.store_o(h, row, 32 * c4, orr, inv_l);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.o_empty[h]));
      if (row_ok) pol.store_lse(h, row, l > 0.f ? (m + log2f(l)) * kLn2 : -CUDART_INF_F);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}


}  // namespace
