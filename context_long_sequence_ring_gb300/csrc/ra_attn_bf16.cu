// Ring-order attention forward, bf16 in / fp32 accumulate, on the 5th-gen
// tensor cores (tcgen05.mma into tensor memory), fed by TMA.
//
// Method sources: "Parallelism-CP" diagram (Q/K/V split along the sequence;
// K/V rotate around a ring of N ranks until every Q block has met every K/V
// block); guijiagi.com "Ring Attention" tag page (ring step t: rank i uses the
// K/V block of rank (i - t) mod N while the next block is in flight; the
// blockwise decomposition softmax(QK^T)V = sum_j e^{s_j} V_j / sum_j e^{s_j}
// with a running max and sum); vLLM-Ascend "Context Parallel (CP)" head-tail
// partition (rank r owns chunks r and 2N-1-r); the causal mask is applied on
// original positions.
//
// Single-GPU mapping of the ring:
//  * the N ranks are virtual; a CTA owns one work item = one query head and a
//    mirrored pair of 128-row query tiles of one rank (tile j of chunk r and
//    tile nt-1-j of chunk 2N-1-r), so every item carries the same causal work
//    (the zigzag balance, per tile instead of per rank);
//  * for each query tile the K/V tiles are visited in ring order: ranks
//    s = r, r-1, ..., r-N+1 (mod N), each rank's chunks s and 2N-1-s in turn;
//    chunks that the causal mask hides are skipped, the diagonal tile is
//    masked element-wise;
//  * the ring's "receive the next block while computing this one" becomes a
//    two-stage TMA ring of K and V tiles in shared memory guarded by mbarriers.
//
// Roles (192 threads): warp 0 issues TMA loads, warp 1 allocates tensor memory
// and issues the MMAs (one thread), warps 2..5 run the online softmax (one
// query row per thread, TMEM lane = row) and the epilogue.
//
// Tensor memory (512 columns): S0 = cols [0,128), S1 = [128,256) (double
// buffered scores), O = [256, 256+D).  Shared memory (1024-aligned, 128-byte
// swizzle, as TMA writes it): Q [128 x D], K[2] and V[2] [128 x D], P [128 x 128].
//
// Per K/V tile j the MMA thread issues S_j = Q K_j^T (D/16 MMAs of
// 128x128x16), then O += P_{j-1} V_{j-1} (8 MMAs of 128xDx16) once the softmax
// has published P_{j-1}; the softmax of tile j overlaps P_{j-1} V_{j-1} and
// S_{j+1}.  O is rescaled in tensor memory only when a row's running max grows
// by more than 2^8 (the stale max is exact as long as l and O use the same
// reference and P stays in range).
#include "ra_attn_pair.cuh"
#include "ra_ring_sched.cuh"

RA_DEFINE_ERROR_FETCH(fetch_error_attn_bf16)

namespace {

using namespace ra::sm100;

struct Params {
  int B, Hq, Hkv, S, N, c, nt, causal, layout, group;
  int ntp, mirrored;  // adjacent-tile schedule: tile pairs per chunk, mirrored pairs per CTA
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  long long wait_limit;
};

__device__ __forceinline__ int64_t token_row(const Params& p, int b, int ch, int off) {
  if (p.layout == RA_LAYOUT_NATURAL) return static_cast<int64_t>(b) * p.S + static_cast<int64_t>(ch) * p.c + off;
  const int rank = ch < p.N ? ch : 2 * p.N - 1 - ch;
  const int half = ch < p.N ? 0 : 1;
  return ((static_cast<int64_t>(rank) * p.B + b) * 2 + half) * p.c + off;
}

// Work item -> (b, hq, rank r, j).  The query heads that share one K/V head
// are innermost so that concurrent CTAs stream the same K/V tiles (L2 reuse).
struct Item {
  int b, hq, g, r, j;
};
__device__ __forceinline__ Item decode_item(const Params& p, int idx) {
  Item it;
  const int hg = idx % p.group; idx /= p.group;
  it.j = idx % p.nt; idx /= p.nt;
  it.r = idx % p.N; idx /= p.N;
  it.g = idx % p.Hkv; idx /= p.Hkv;
  it.b = idx;
  it.hq = it.g * p.group + hg;
  return it;
}
// The two query tiles of an item: (chunk r, tile j) and (chunk 2N-1-r, tile nt-1-j).
__device__ __forceinline__ void tile_of(const Params& p, const Item& it, int ti, int& qc, int& qi) {
  if (ti == 0) { qc = it.r; qi = it.j; }
  else { qc = 2 * p.N - 1 - it.r; qi = p.nt - 1 - it.j; }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    ring_attn_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const Params p) {
  constexpr int SLABS = D / 64;                     // 64-column (128-byte) slabs of a Q/K/V tile
  constexpr uint32_t kTileBytes = BM * D * 2;       // one Q, K or V tile
  constexpr uint32_t kIdescS = idesc_bf16_f32(BM, BN, 0, 0);  // S = Q K^T, both K-major
  constexpr uint32_t kIdescO = idesc_bf16_f32(BM, D, 0, 1);   // O += P V, V is MN-major

  extern __shared__ uint8_t smem_raw[];
  Smem<D>& sm = *reinterpret_cast<Smem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Item it = decode_item(p, blockIdx.x);
  const Sched sch{p.N, p.c, p.nt, p.causal, BN, p.nt};
  volatile int* abort_flag = &sm.abort_flag;
  const long long lim = p.wait_limit;

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    mbar_init(smem_u32(&sm.q_empty), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.k_empty[s]), 1);
      mbar_init(smem_u32(&sm.v_full[s]), 1);
      mbar_init(smem_u32(&sm.v_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sm.s_full[s]), 1);
      mbar_init(smem_u32(&sm.s_empty[s]), 128);
    }
    mbar_init(smem_u32(&sm.p_full), 128);
    mbar_init(smem_u32(&sm.pv_done), 1);
    mbar_init(smem_u32(&sm.o_empty), 128);
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
      for (int ti = 0; ti < 2 && ok; ++ti) {
        int qc, qi;
        tile_of(p, it, ti, qc, qi);
        if (!(ok = mbar_wait(smem_u32(&sm.q_empty), (ti & 1) ^ 1, abort_flag, lim, 1))) break;
        const uint32_t qb = smem_u32(&sm.q_full);
        mbar_arrive_expect_tx(qb, kTileBytes);
        const int32_t qrow = static_cast<int32_t>(token_row(p, it.b, qc, qi * BM));
        for (int s = 0; s < SLABS; ++s) tma_load_3d(smem_u32(sm.q + s * BM * 128), &tmQ, qb, 64 * s, it.hq, qrow);
        q_iss = true;
        q_ph = ti & 1;
        KvIter kv;
        kv.init(sch, qc, qi);
        int kc, kt;
        while (kv.next(kc, kt)) {
          const int st = kv_cnt % STAGES;
          const uint32_t ph = (kv_cnt / STAGES) & 1;
          const int32_t krow = static_cast<int32_t>(token_row(p, it.b, kc, kt * BN));
          if (!(ok = mbar_wait(smem_u32(&sm.k_empty[st]), ph ^ 1, abort_flag, lim, 2))) break;
          mbar_arrive_expect_tx(smem_u32(&sm.k_full[st]), kTileBytes);
          for (int s = 0; s < SLABS; ++s)
            tma_load_3d(smem_u32(sm.k[st] + s * BN * 128), &tmK, smem_u32(&sm.k_full[st]), 64 * s, it.g, krow);
          k_iss[st] = true;
          k_ph[st] = ph;
          if (!(ok = mbar_wait(smem_u32(&sm.v_empty[st]), ph ^ 1, abort_flag, lim, 3))) break;
          mbar_arrive_expect_tx(smem_u32(&sm.v_full[st]), kTileBytes);
          for (int s = 0; s < SLABS; ++s)
            tma_load_3d(smem_u32(sm.v[st] + s * BN * 128), &tmV, smem_u32(&sm.v_full[st]), 64 * s, it.g, krow);
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
      uint32_t kv_cnt = 0, s_cnt = 0, pv_cnt = 0;
      bool ok = true;
      const uint32_t q_base = smem_u32(sm.q), p_base = smem_u32(sm.p);
      for (int ti = 0; ti < 2 && ok; ++ti) {
        int qc, qi;
        tile_of(p, it, ti, qc, qi);
        const int nkv = n_kv_tiles(sch, qc, qi);
        if (!(ok = mbar_wait(smem_u32(&sm.q_full), ti & 1, abort_flag, lim, 10))) break;
        int prev_st = 0;
        uint32_t prev_ph = 0;
        // O += P_{jj} V_{jj}
        auto do_pv = [&](int st, uint32_t ph, bool first) -> bool {
          if (!mbar_wait(smem_u32(&sm.p_full), pv_cnt & 1, abort_flag, lim, 11)) return false;
          if (!mbar_wait(smem_u32(&sm.v_full[st]), ph, abort_flag, lim, 12)) return false;
          if (first && !mbar_wait(smem_u32(&sm.o_empty), (ti & 1) ^ 1, abort_flag, lim, 13)) return false;
          tc_fence_after();
          const uint32_t v_base = smem_u32(sm.v[st]);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t ad = desc_sw128(p_base + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = desc_sw128(v_base + kk * 16 * 128, BN * 128, 1024);
            mma_bf16_ss(tmem + kColO, ad, bd, kIdescO, (kk > 0 || !first) ? 1u : 0u);
          }
          mma_commit(smem_u32(&sm.pv_done));
          mma_commit(smem_u32(&sm.v_empty[st]));
          ++pv_cnt;
          return true;
        };
        for (int j = 0; j < nkv && ok; ++j) {
          const int st = kv_cnt % STAGES;
          const uint32_t ph = (kv_cnt / STAGES) & 1;
          const int sb = s_cnt & 1;
          const uint32_t sph = (s_cnt >> 1) & 1;
          if (!(ok = mbar_wait(smem_u32(&sm.k_full[st]), ph, abort_flag, lim, 14))) break;
          if (!(ok = mbar_wait(smem_u32(&sm.s_empty[sb]), sph ^ 1, abort_flag, lim, 15))) break;
          tc_fence_after();
          const uint32_t k_base = smem_u32(sm.k[st]);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
            const uint64_t ad = desc_sw128(q_base + off, 16, 1024);
            const uint64_t bd = desc_sw128(k_base + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16, 1024);
            mma_bf16_ss(tmem + kColS0 + sb * BN, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
          }
          mma_commit(smem_u32(&sm.s_full[sb]));
          mma_commit(smem_u32(&sm.k_empty[st]));
          if (j == nkv - 1) mma_commit(smem_u32(&sm.q_empty));
          ++s_cnt;
          if (j > 0 && !(ok = do_pv(prev_st, prev_ph, j - 1 == 0))) break;
          prev_st = st;
          prev_ph = ph;
          ++kv_cnt;
        }
        if (ok) ok = do_pv(prev_st, prev_ph, nkv - 1 == 0);
      }
      // make sure no MMA is still writing tensor memory before it is freed
      mma_commit(smem_u32(&sm.drain));
      if (!mbar_wait_quiesce(smem_u32(&sm.drain), 0, ok ? lim : (1 << 22)) && ok) {
        *abort_flag = 1;
        ra_record_error(RA_ERR_TIMEOUT, 16);
      }
    }
  } else {
    // ============================================================ softmax + epilogue
    const int quarter = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;          // query row inside the tile
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t p_base = smem_u32(sm.p);
    uint32_t s_cnt = 0, pv_cnt = 0;
    bool ok = true;
    for (int ti = 0; ti < 2 && ok; ++ti) {
      int qc, qi;
      tile_of(p, it, ti, qc, qi);
      const int q_valid = min(BM, p.c - qi * BM);
      const int nkv = n_kv_tiles(sch, qc, qi);
      KvIter kv;
      kv.init(sch, qc, qi);
      float m = -CUDART_INF_F, l = 0.f;
      for (int j = 0; j < nkv; ++j) {
        int kc = 0, kt = 0;
        kv.next(kc, kt);
        const int sb = s_cnt & 1;
        const uint32_t sph = (s_cnt >> 1) & 1;
        if (!(ok = mbar_wait(smem_u32(&sm.s_full[sb]), sph, abort_flag, lim, 20))) break;
        tc_fence_after();
        int col_lim;
        bool masked;
        tile_mask(sch, qc, qi, kc, kt, row, col_lim, masked);
        uint32_t pk[BN / 2];
        const float alpha = softmax_row(t_lane + kColS0 + sb * BN, j, masked, col_lim, p.scale_log2, m, l, pk);
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.s_empty[sb]));
        ++s_cnt;
        if (j > 0) {
          // P_{j-1} V_{j-1} must be complete: P buffer reuse and O rescale
          if (!(ok = mbar_wait(smem_u32(&sm.pv_done), pv_cnt & 1, abort_flag, lim, 21))) break;
          ++pv_cnt;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) {
              uint32_t orr[32];
              tmem_ld32(t_lane + kColO + 32 * c4, orr);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
              tmem_st32(t_lane + kColO + 32 * c4, orr);
            }
            tmem_wait_st();
          }
        }
        // P (bf16, 128-byte swizzle, K-major) into shared memory
#pragma unroll
        for (int ch = 0; ch < BN / 8; ++ch) {
          const int slab = ch >> 3, c16 = ch & 7;
          const uint32_t addr = p_base + slab * (BM * 128) + row * 128 + ((c16 ^ (row & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * ch]),
                       "r"(pk[4 * ch + 1]), "r"(pk[4 * ch + 2]), "r"(pk[4 * ch + 3])
                       : "memory");
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.p_full));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = mbar_wait(smem_u32(&sm.pv_done), pv_cnt & 1, abort_flag, lim, 22))) break;
      ++pv_cnt;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool row_ok = row < q_valid;
      const int64_t trow = token_row(p, it.b, qc, qi * BM + row);
      __nv_bfloat16* orow = p.o + (trow * p.Hq + it.hq) * D;
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t orr[32];
        tmem_ld32(t_lane + kColO + 32 * c4, orr);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 pk;
            pk.x = f2_bf16x2(__uint_as_float(orr[i]) * inv_l, __uint_as_float(orr[i + 1]) * inv_l);
            pk.y = f2_bf16x2(__uint_as_float(orr[i + 2]) * inv_l, __uint_as_float(orr[i + 3]) * inv_l);
            pk.z = f2_bf16x2(__uint_as_float(orr[i + 4]) * inv_l, __uint_as_float(orr[i + 5]) * inv_l);
            pk.w = f2_bf16x2(__uint_as_float(orr[i + 6]) * inv_l, __uint_as_float(orr[i + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + 32 * c4 + i) = pk;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.o_empty));
      if (row_ok) p.lse[trow * p.Hq + it.hq] = l > 0.f ? (m + log2f(l)) * kLn2 : -CUDART_INF_F;
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

struct Item2 {
  int b, hq0, g, r, j;
};
__device__ __forceinline__ Item2 decode_item2(const Params& p, int idx) {
  Item2 it;
  const int pairs = p.group / 2;
  const int hp = idx % pairs; idx /= pairs;
  it.j = idx % p.nt; idx /= p.nt;
  it.r = idx % p.N; idx /= p.N;
  it.g = idx % p.Hkv; idx /= p.Hkv;
  it.b = idx;
  it.hq0 = it.g * p.group + 2 * hp;
  return it;
}


// Ring schedule: a mirrored pair of query tiles of one virtual rank, K/V tiles
// in ring order, causal mask by original position, bf16 output.
template <int D>
struct RingPolicy : PolicyDefaults {
  using Args = Params;
  struct KvPos {
    KvIter it;
    int kc, kt;
    int32_t row;
  };
  const Params& p;
  Item2 item;
  Sched sch;
  int qc, qi;
  __device__ RingPolicy(const Params& a, int idx)
      : p(a), item(decode_item2(a, idx)), sch{a.N, a.c, a.nt, a.causal, BN, a.nt}, qc(0), qi(0) {}
  __device__ int tiles() const { return 2; }
  __device__ int kvh() const { return item.g; }
  __device__ void set_tile(int ti) {
    const Item it1{item.b, item.hq0, item.g, item.r, item.j};
    tile_of(p, it1, ti, qc, qi);
  }
  __device__ int q_head(int h) const { return item.hq0 + h; }
  __device__ int32_t q_row(int) const { return static_cast<int32_t>(token_row(p, item.b, qc, qi * BM)); }
  __device__ int q_valid(int) const { return min(BM, p.c - qi * BM); }
  __device__ int n_kv() const { return n_kv_tiles(sch, qc, qi); }
  __device__ void kv_begin(KvPos& k) const { k.it.init(sch, qc, qi); }
  __device__ bool kv_next(KvPos& k) const {
    if (!k.it.next(k.kc, k.kt)) return false;
    k.row = static_cast<int32_t>(token_row(p, item.b, k.kc, k.kt * BN));
    return true;
  }
  __device__ void mask(const KvPos& k, int, int row, int& col_lim, bool& masked) const {
    tile_mask(sch, qc, qi, k.kc, k.kt, row, col_lim, masked);
  }
  __device__ void store_o(int h, int row, int col0, const uint32_t (&o)[32], float inv_l) const {
    const int64_t trow = token_row(p, item.b, qc, qi * BM + row);
    __nv_bfloat16* dst = p.o + (trow * p.Hq + item.hq0 + h) * D + col0;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      uint4 pk;
      pk.x = f2_bf16x2(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l);
      pk.y = f2_bf16x2(__uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
      pk.z = f2_bf16x2(__uint_as_float(o[i + 4]) * inv_l, __uint_as_float(o[i + 5]) * inv_l);
      pk.w = f2_bf16x2(__uint_as_float(o[i + 6]) * inv_l, __uint_as_float(o[i + 7]) * inv_l);
      *reinterpret_cast<uint4*>(dst + i) = pk;
    }
  }
  __device__ void store_lse(int h, int row, float lse) const {
    p.lse[token_row(p, item.b, qc, qi * BM + row) * p.Hq + item.hq0 + h] = lse;
  }
  __device__ void write_empty(int, int) const {}  // every ring query tile meets at least one key tile
};

// Adjacent-tile schedule, for any GQA group (odd ones and plain multi-head
// attention included): one query head, with two adjacent 128-row query tiles
// of one chunk, 2i and 2i+1, as the two slots.  The K/V tiles are those the
// later tile meets, a superset of the earlier tile's under the causal mask
// (one extra diagonal tile, fully masked for the earlier one), in ring order.
// Mirrored: the CTA then runs the mirrored pair of chunk 2N-1-r, which evens
// out the causal work as the head-pair schedule does with single tiles;
// otherwise (small problems, to fill the SMs) one pair per CTA, the heaviest
// pairs first.  A missing second tile (odd tile count) is an empty slot.
template <int D>
struct RingTilePolicy : PolicyDefaults {
  using Args = Params;
  using KvPos = typename RingPolicy<D>::KvPos;
  const Params& p;
  Sched sch;
  int b, hq, g, r, jp, qc, pr;
  __device__ RingTilePolicy(const Params& a, int idx) : p(a), sch{a.N, a.c, a.nt, a.causal, BN, a.nt} {
    const int hg = idx % a.group; idx /= a.group;
    if (a.mirrored) {
      jp = idx % a.ntp; idx /= a.ntp;
      r = idx % a.N; idx /= a.N;
      g = idx % a.Hkv; idx /= a.Hkv;
      b = idx;
    } else {
      g = idx % a.Hkv; idx /= a.Hkv;
      b = idx % a.B; idx /= a.B;
      jp = a.ntp - 1 - idx % a.ntp; idx /= a.ntp;
      r = 2 * a.N - 1 - idx;  // chunk index, last (heaviest) first
    }
    hq = g * a.group + hg;
    qc = r;
    pr = jp;
  }
  __device__ int tiles() const { return p.mirrored ? 2 : 1; }
  __device__ int kvh() const { return g; }
  __device__ void set_tile(int ti) {
    if (ti == 0) { qc = r; pr = jp; }
    else { qc = 2 * p.N - 1 - r; pr = p.ntp - 1 - jp; }
  }
  __device__ int q_head(int) const { return hq; }
  __device__ int32_t q_row(int h) const {
    return static_cast<int32_t>(token_row(p, b, qc, (2 * pr + h) * BM));
  }
  __device__ int q_valid(int h) const { return max(0, min(BM, p.c - (2 * pr + h) * BM)); }
  __device__ int kv_tile() const { return min(2 * pr + 1, p.nt - 1); }
  __device__ int n_kv() const { return n_kv_tiles(sch, qc, kv_tile()); }
  __device__ void kv_begin(KvPos& k) const { k.it.init(sch, qc, kv_tile()); }
  __device__ bool kv_next(KvPos& k) const {
    if (!k.it.next(k.kc, k.kt)) return false;
    k.row = static_cast<int32_t>(token_row(p, b, k.kc, k.kt * BN));
    return true;
  }
  __device__ void mask(const KvPos& k, int h, int row, int& col_lim, bool& masked) const {
    tile_mask(sch, qc, 2 * pr + h, k.kc, k.kt, row, col_lim, masked);
  }
  __device__ void store_o(int h, int row, int col0, const uint32_t (&o)[32], float inv_l) const {
    const int64_t trow = token_row(p, b, qc, (2 * pr + h) * BM + row);
    __nv_bfloat16* dst = p.o + (trow * p.Hq + hq) * D + col0;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      uint4 pk;
      pk.x = f2_bf16x2(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l);
      pk.y = f2_bf16x2(__uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
      pk.z = f2_bf16x2(__uint_as_float(o[i + 4]) * inv_l, __uint_as_float(o[i + 5]) * inv_l);
      pk.w = f2_bf16x2(__uint_as_float(o[i + 6]) * inv_l, __uint_as_float(o[i + 7]) * inv_l);
      *reinterpret_cast<uint4*>(dst + i) = pk;
    }
  }
  __device__ void store_lse(int h, int row, float lse) const {
    p.lse[token_row(p, b, qc, (2 * pr + h) * BM + row) * p.Hq + hq] = lse;
  }
  __device__ void write_empty(int, int) const {}  // every ring query tile meets at least one key tile
};

// ------------------------------------------------------------------ varlen
// Several requests of different lengths in one call, in the layout the
// head-tail partition gathers them to: rank-major, then request, then the
// request's chunk r and chunk 2N-1-r.  Request b is padded to L'_b, a
// multiple of 2N, and cut into chunks of c_b = L'_b / 2N tokens, so its row
// (rank r, half, offset) is r * T_rank + 2 * pre_b + half * c_b + offset with
// T_rank = 2 * sum_b c_b and pre_b = sum_{b' < b} c_b'.  Keys at positions at
// or past the request's real length (the padding) are masked.
constexpr int kMaxVarlenSeqs = 256;

struct VarlenParams {
  int num_seqs, Hq, Hkv, group, N, causal, mirrored;
  int T_rank;
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  long long wait_limit;
  int items_pre[kMaxVarlenSeqs + 1];  // CTAs before request b
  int c[kMaxVarlenSeqs];              // chunk length of request b
  int len[kMaxVarlenSeqs];            // real length of request b
  int pre[kMaxVarlenSeqs];            // sum of the chunk lengths of requests before b
};

// Adjacent-tile schedule (as RingTilePolicy) within one request of a varlen call.
template <int D>
struct RingVarlenPolicy : PolicyDefaults {
  using Args = VarlenParams;
  using KvPos = typename RingPolicy<D>::KvPos;
  const VarlenParams& p;
  Sched sch;
  int b, hq, g, r, jp, qc, pr, ntp;
  __device__ RingVarlenPolicy(const VarlenParams& a, int idx) : p(a) {
    int lo = 0, hi = a.num_seqs;   // the request: last b with items_pre[b] <= idx
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.items_pre[mid] <= idx) lo = mid; else hi = mid;
    }
    b = lo;
    idx -= a.items_pre[b];
    const int c = a.c[b], nt = (c + BM - 1) / BM;
    ntp = (nt + 1) / 2;
    sch = Sched{a.N, c, nt, a.causal, BN, nt};
    const int hg = idx % a.group; idx /= a.group;
    if (a.mirrored) {
      jp = idx % ntp; idx /= ntp;
      r = idx % a.N; idx /= a.N;
      g = idx;
    } else {
      g = idx % a.Hkv; idx /= a.Hkv;
      jp = ntp - 1 - idx % ntp; idx /= ntp;
      r = 2 * a.N - 1 - idx;
    }
    hq = g * a.group + hg;
    qc = r;
    pr = jp;
  }
  __device__ int32_t row_of(int ch, int off) const {
    const int rank = ch < p.N ? ch : 2 * p.N - 1 - ch;
    const int half = ch < p.N ? 0 : 1;
    return rank * p.T_rank + 2 * p.pre[b] + half * p.c[b] + off;
  }
  __device__ int tiles() const { return p.mirrored ? 2 : 1; }
  __device__ int kvh() const { return g; }
  __device__ void set_tile(int ti) {
    if (ti == 0) { qc = r; pr = jp; }
    else { qc = 2 * p.N - 1 - r; pr = ntp - 1 - jp; }
  }
  __device__ int q_head(int) const { return hq; }
  __device__ int32_t q_row(int h) const { return row_of(qc, (2 * pr + h) * BM); }
  __device__ int q_valid(int h) const { return max(0, min(BM, p.c[b] - (2 * pr + h) * BM)); }
  __device__ int kv_tile() const { return min(2 * pr + 1, sch.nt - 1); }
  __device__ int n_kv() const { return n_kv_tiles(sch, qc, kv_tile()); }
  __device__ void kv_begin(KvPos& k) const { k.it.init(sch, qc, kv_tile()); }
  __device__ bool kv_next(KvPos& k) const {
    if (!k.it.next(k.kc, k.kt)) return false;
    k.row = row_of(k.kc, k.kt * BN);
    return true;
  }
  __device__ void mask(const KvPos& k, int h, int row, int& col_lim, bool& masked) const {
    tile_mask(sch, qc, 2 * pr + h, k.kc, k.kt, row, col_lim, masked);
    const int real = p.len[b] - (k.kc * p.c[b] + k.kt * BN);   // keys of the tile before the padding
    if (real < col_lim) {
      col_lim = real > 0 ? real : 0;
      masked = true;
    }
  }
  __device__ void store_o(int h, int row, int col0, const uint32_t (&o)[32], float inv_l) const {
    const int64_t trow = row_of(qc, (2 * pr + h) * BM + row);
    __nv_bfloat16* dst = p.o + (trow * p.Hq + hq) * D + col0;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      uint4 pk;
      pk.x = f2_bf16x2(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l);
      pk.y = f2_bf16x2(__uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
      pk.z = f2_bf16x2(__uint_as_float(o[i + 4]) * inv_l, __uint_as_float(o[i + 5]) * inv_l);
      pk.w = f2_bf16x2(__uint_as_float(o[i + 6]) * inv_l, __uint_as_float(o[i + 7]) * inv_l);
      *reinterpret_cast<uint4*>(dst + i) = pk;
    }
  }
  __device__ void store_lse(int h, int row, float lse) const {
    p.lse[static_cast<int64_t>(row_of(qc, (2 * pr + h) * BM + row)) * p.Hq + hq] = lse;
  }
  __device__ void write_empty(int, int) const {}  // every query tile meets at least its own first key tile
};

// Per-rank tile classification with the kernels' own iterator (for tests):
// visited tiles that need no mask, visited tiles with a causal mask, skipped.
__global__ void schedule_counts_kernel(Sched s, unsigned long long* counts) {
  const int n_tiles = 2 * s.N * s.nt;  // query tiles of the whole sequence
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < n_tiles; idx += gridDim.x * blockDim.x) {
    const int qc = idx / s.nt, qi = idx % s.nt;
    const int r = qc < s.N ? qc : 2 * s.N - 1 - qc;
    KvIter kv;
    kv.init(s, qc, qi);
    int kc, kt;
    unsigned long long full = 0, diag = 0, seen = 0;
    while (kv.next(kc, kt)) {
      ++seen;
      const int kvv = min(s.bnk, s.c - kt * s.bnk);
      const bool d = s.causal && kc == qc && kt * s.bnk + kvv - 1 > qi * BM;
      if (d) ++diag; else ++full;
    }
    if (static_cast<int>(seen) != n_kv_tiles(s, qc, qi)) ra_record_error(RA_ERR_DEVICE_BOUNDS, 30);
    atomicAdd(&counts[r * 3 + 0], full);
    atomicAdd(&counts[r * 3 + 1], diag);
    atomicAdd(&counts[r * 3 + 2], static_cast<unsigned long long>(2 * s.N * s.ntk) - seen);
  }
}

template <int D>
ra_status launch_bf16(const void* q, const void* k, const void* v, const Params& prm, int variant,
                      cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  const int64_t rows = static_cast<int64_t>(prm.B) * prm.S;
  ra_status st;
  if ((st = make_map(&mq, q, D, prm.Hq, rows)) != RA_OK) return st;
  if ((st = make_map(&mk, k, D, prm.Hkv, rows)) != RA_OK) return st;
  if ((st = make_map(&mv, v, D, prm.Hkv, rows)) != RA_OK) return st;
  const int64_t tiles = static_cast<int64_t>(prm.B) * prm.Hq * prm.N * prm.nt;  // mirrored tile pairs x heads
  if (variant == 2) {
    const size_t smem = sizeof(Smem2<D>) + 1024;
    RA_CUDA_TRY(cudaFuncSetAttribute(attn_pair_kernel<D, RingPolicy<D>>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
    attn_pair_kernel<D, RingPolicy<D>><<<static_cast<unsigned>(tiles / 2), kThreads2, smem, stream>>>(mq, mk, mv,
                                                                                                     prm);
    RA_LAUNCH_CHECK("attn_pair_kernel<RingPolicy>");
    return RA_OK;
  }
  if (variant == 3) {
    const int64_t items = static_cast<int64_t>(prm.B) * prm.Hq * prm.ntp * (prm.mirrored ? prm.N : 2 * prm.N);
    const size_t smem = sizeof(Smem2<D>) + 1024;
    RA_CUDA_TRY(cudaFuncSetAttribute(attn_pair_kernel<D, RingTilePolicy<D>>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
    attn_pair_kernel<D, RingTilePolicy<D>><<<static_cast<unsigned>(items), kThreads2, smem, stream>>>(mq, mk, mv,
                                                                                                       prm);
    RA_LAUNCH_CHECK("attn_pair_kernel<RingTilePolicy>");
    return RA_OK;
  }
  const size_t smem = sizeof(Smem<D>) + 1024;
  RA_CUDA_TRY(cudaFuncSetAttribute(ring_attn_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem)));
  ring_attn_bf16_kernel<D><<<static_cast<unsigned>(tiles), kThreads, smem, stream>>>(mq, mk, mv, prm);
  RA_LAUNCH_CHECK("ring_attn_bf16_kernel");
  return RA_OK;
}

template <int D>
ra_status launch_varlen(const void* q, const void* k, const void* v, int64_t rows, const VarlenParams& prm,
                        int64_t items, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  ra_status st;
  if ((st = make_map(&mq, q, D, prm.Hq, rows)) != RA_OK) return st;
  if ((st = make_map(&mk, k, D, prm.Hkv, rows)) != RA_OK) return st;
  if ((st = make_map(&mv, v, D, prm.Hkv, rows)) != RA_OK) return st;
  const size_t smem = sizeof(Smem2<D>) + 1024;
  RA_CUDA_TRY(cudaFuncSetAttribute(attn_pair_kernel<D, RingVarlenPolicy<D>>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
  attn_pair_kernel<D, RingVarlenPolicy<D>><<<static_cast<unsigned>(items), kThreads2, smem, stream>>>(mq, mk, mv,
                                                                                                       prm);
  RA_LAUNCH_CHECK("attn_pair_kernel<RingVarlenPolicy>");
  return RA_OK;
}

}  // namespace

namespace ra {
ra_status ring_attn_fwd_f32(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                            int Hkv, int S, int d, int causal, int N, float scale, int layout,
                            cudaStream_t stream);


}  // namespace ra

extern "C" ra_status ra_ring_attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                                         int32_t B, int32_t Hq, int32_t Hkv, int32_t S, int32_t d, ra_dtype dt,
                                         int32_t causal, int32_t n_ranks, float scale, ra_layout layout,
                                         int32_t variant, ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(variant >= 0 && variant <= 3, "variant must be 0, 1, 2 or 3");
  RA_REQUIRE(B >= 1 && Hq >= 1 && Hkv >= 1 && S >= 1, "B, Hq, Hkv, S must be >= 1");
  RA_REQUIRE(Hq % Hkv == 0, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  RA_REQUIRE(n_ranks >= 1, "n_ranks must be >= 1 (got %d)", n_ranks);
  RA_REQUIRE(S % (2 * n_ranks) == 0, "S (%d) must be a multiple of 2*n_ranks (%d); pad with ra_zigzag_partition",
             S, 2 * n_ranks);
  RA_REQUIRE(static_cast<int64_t>(B) * S < (int64_t(1) << 31), "B*S must be < 2^31");
  RA_REQUIRE(dt == RA_F32 || dt == RA_BF16, "unknown dtype");
  RA_REQUIRE(layout == RA_LAYOUT_NATURAL || layout == RA_LAYOUT_ZIGZAG, "unknown layout");
  if (d != 64 && d != 128) return ra::fail(RA_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", d);
  RA_REQUIRE(q && k && v && o && lse, "NULL pointer");
  RA_REQUIRE(ra::aligned16(q) && ra::aligned16(k) && ra::aligned16(v) && ra::aligned16(o) &&
                 reinterpret_cast<uintptr_t>(lse) % 4 == 0,
             "q, k, v, o must be 16-byte aligned");
  const float sc = scale > 0.f ? scale : 1.f / sqrtf(static_cast<float>(d));
  if (dt == RA_F32) return ra::ring_attn_fwd_f32(q, k, v, o, lse, B, Hq, Hkv, S, d, causal ? 1 : 0, n_ranks, sc,
                                                 layout, stream);
  Params prm;
  prm.B = B; prm.Hq = Hq; prm.Hkv = Hkv; prm.S = S; prm.N = n_ranks; prm.c = S / (2 * n_ranks);
  prm.nt = static_cast<int>(ra::ceil_div(prm.c, BM));
  prm.causal = causal ? 1 : 0; prm.layout = layout; prm.group = Hq / Hkv;
  prm.scale_log2 = sc * 1.4426950408889634f;
  prm.o = static_cast<__nv_bfloat16*>(o); prm.lse = lse;
  prm.wait_limit = ra::wait_limit();
  const int64_t items = static_cast<int64_t>(B) * Hkv * n_ranks * prm.nt * prm.group;
  RA_REQUIRE(items < (int64_t(1) << 31), "too many work items");
  prm.ntp = (prm.nt + 1) / 2;
  prm.mirrored = 1;
  if (variant == 0) variant = (prm.group % 2 == 0) ? 2 : 3;
  RA_REQUIRE(variant != 2 || prm.group % 2 == 0, "the two-head variant needs an even Hq/Hkv");
  if (variant == 3) {
    // mirrored pairs halve the CTA count; keep them only while that still fills two waves
    int dev = 0, sms = 0;
    RA_CUDA_TRY(cudaGetDevice(&dev));
    RA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    prm.mirrored = static_cast<int64_t>(B) * Hq * n_ranks * prm.ntp >= 2 * static_cast<int64_t>(sms) ? 1 : 0;
  }
  if (d == 128) return launch_bf16<128>(q, k, v, prm, variant, stream);
  return launch_bf16<64>(q, k, v, prm, variant, stream);
}

extern "C" ra_status ra_ring_attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                             const int64_t* seq_lens, int32_t num_seqs, int32_t Hq, int32_t Hkv,
                                             int32_t d, ra_dtype dt, int32_t causal, int32_t n_ranks, float scale,
                                             ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(seq_lens != nullptr, "seq_lens is NULL");
  RA_REQUIRE(num_seqs >= 1 && num_seqs <= kMaxVarlenSeqs, "num_seqs must be in [1, %d] (got %d)", kMaxVarlenSeqs,
             num_seqs);
  RA_REQUIRE(Hq >= 1 && Hkv >= 1, "Hq, Hkv must be >= 1");
  RA_REQUIRE(Hq % Hkv == 0, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  RA_REQUIRE(n_ranks >= 1, "n_ranks must be >= 1 (got %d)", n_ranks);
  RA_REQUIRE(dt == RA_F32 || dt == RA_BF16, "unknown dtype");
  if (dt != RA_BF16) return ra::fail(RA_ERR_UNSUPPORTED, "the varlen call runs on bf16 inputs only");
  if (d != 64 && d != 128) return ra::fail(RA_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", d);
  VarlenParams prm;
  prm.num_seqs = num_seqs; prm.Hq = Hq; prm.Hkv = Hkv; prm.group = Hq / Hkv; prm.N = n_ranks;
  prm.causal = causal ? 1 : 0;
  int64_t G = 0, csum = 0, pairs = 0;
  for (int b = 0; b < num_seqs; ++b) {
    RA_REQUIRE(seq_lens[b] >= 0, "negative sequence length at %d", b);
    const int64_t Lp = ra::ceil_div(seq_lens[b], 2 * n_ranks) * 2 * n_ranks;
    RA_REQUIRE(Lp < (int64_t(1) << 31), "sequence %d too long", b);
    prm.c[b] = static_cast<int>(Lp / (2 * n_ranks));
    prm.len[b] = static_cast<int>(seq_lens[b]);
    prm.pre[b] = static_cast<int>(csum);
    csum += prm.c[b];
    G += Lp;
    pairs += (ra::ceil_div(prm.c[b], BM) + 1) / 2;
    RA_REQUIRE(G < (int64_t(1) << 31), "total padded length must be < 2^31");
  }
  if (G == 0) return RA_OK;
  RA_REQUIRE(q && k && v && o && lse, "NULL pointer");
  RA_REQUIRE(ra::aligned16(q) && ra::aligned16(k) && ra::aligned16(v) && ra::aligned16(o) &&
                 reinterpret_cast<uintptr_t>(lse) % 4 == 0,
             "q, k, v, o must be 16-byte aligned");
  prm.T_rank = static_cast<int>(2 * csum);
  int dev = 0, sms = 0;
  RA_CUDA_TRY(cudaGetDevice(&dev));
  RA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  // mirrored pairs halve the CTA count; keep them only while that still fills two waves
  prm.mirrored = static_cast<int64_t>(Hq) * n_ranks * pairs >= 2 * static_cast<int64_t>(sms) ? 1 : 0;
  int64_t items = 0;
  for (int b = 0; b < num_seqs; ++b) {
    prm.items_pre[b] = static_cast<int>(items);
    const int64_t ntp = (ra::ceil_div(prm.c[b], BM) + 1) / 2;
    items += static_cast<int64_t>(Hq) * ntp * (prm.mirrored ? n_ranks : 2 * n_ranks);
    RA_REQUIRE(items < (int64_t(1) << 31), "too many work items");
  }
  prm.items_pre[num_seqs] = static_cast<int>(items);
  const float sc = scale > 0.f ? scale : 1.f / sqrtf(static_cast<float>(d));
  prm.scale_log2 = sc * 1.4426950408889634f;
  prm.o = static_cast<__nv_bfloat16*>(o); prm.lse = lse;
  prm.wait_limit = ra::wait_limit();
  if (d == 128) return launch_varlen<128>(q, k, v, G, prm, items, stream);
  return launch_varlen<64>(q, k, v, G, prm, items, stream);
}

extern "C" ra_status ra_ring_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int32_t B,
                                      int32_t Hq, int32_t Hkv, int32_t S, int32_t d, ra_dtype dt, int32_t causal,
                                      int32_t n_ranks, float scale, ra_layout layout, ra_stream stream) {
  return ra_ring_attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, S, d, dt, causal, n_ranks, scale, layout, 0, stream);
}

extern "C" ra_status ra_ring_schedule_counts_ex(int32_t S, int32_t n_ranks, int32_t causal, int32_t kv_tile,
                                                int64_t* counts, ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(n_ranks >= 1 && S >= 1 && S % (2 * n_ranks) == 0, "S must be a positive multiple of 2*n_ranks");
  RA_REQUIRE(kv_tile == 64 || kv_tile == 128, "kv_tile must be 64 or 128");
  RA_REQUIRE(counts != nullptr && reinterpret_cast<uintptr_t>(counts) % 8 == 0, "counts must be 8-byte aligned");
  const int c = S / (2 * n_ranks);
  Sched s{n_ranks, c, static_cast<int>(ra::ceil_div(c, BM)), causal ? 1 : 0, kv_tile,
          static_cast<int>(ra::ceil_div(c, kv_tile))};
  RA_CUDA_TRY(cudaMemsetAsync(counts, 0, sizeof(int64_t) * 3 * n_ranks, stream));
  const int n_tiles = 2 * s.N * s.nt;
  schedule_counts_kernel<<<static_cast<unsigned>(ra::ceil_div(n_tiles, 128)), 128, 0, stream>>>(
      s, reinterpret_cast<unsigned long long*>(counts));
  RA_LAUNCH_CHECK("schedule_counts_kernel");
  return RA_OK;
}

extern "C" ra_status ra_ring_schedule_counts(int32_t S, int32_t n_ranks, int32_t causal, int64_t* counts,
                                             ra_stream stream) {
  return ra_ring_schedule_counts_ex(S, n_ranks, causal, 128, counts, stream);
}

