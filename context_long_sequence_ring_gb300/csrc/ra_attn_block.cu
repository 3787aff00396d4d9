// Block partial attention on the tcgen05 tensor cores and the segmented
// (bounded-KV-per-round) chunked prefill built on it.
//
// Sources: guijiagi.com "Ring Attention" tag page (each ring step is the
// attention of the local Q block against the K/V block held at that step,
// folded in with the blockwise decomposition); vLLM-Ascend developer guide
// "Context Parallel (CP)", chunked prefill (a maximum amount of KV per round,
// attention and online-softmax update segment after segment).
#include "ra_attn_pair.cuh"

RA_DEFINE_ERROR_FETCH(fetch_error_attn_block)

namespace {
using namespace ra::sm100;

// ===========================================================================
// Block partial attention: queries at positions q_pos0 + i against keys at
// positions k_pos0 + j (one K/V block of a ring step, or one segment of a
// chunked prefill), causal by absolute position.  Output: the partial's O
// (fp32, already normalised by its own row sum) and LSE, to be combined with
// other partials by the LSE merge.  A row with no visible key gets O = 0 and
// LSE = -inf.  Even GQA groups run the two-slot kernel with BlockPolicy (two
// heads per CTA); odd groups with at least two query tiles run it with
// BlockTilePolicy (two adjacent query tiles per CTA); a single query tile of an
// odd group runs the one-head kernel below: one CTA per (128-row query tile,
// query head), with the pipeline of the one-head ring kernel (TMA producer,
// one MMA thread, a softmax warpgroup, P via shared memory, double-buffered S).
// ===========================================================================
struct BlockParams {
  int Tq, Tk, Hq, Hkv, group, causal;
  long long q_pos0, k_pos0;
  float scale_log2;
  float* o;    // [Tq, Hq, D] fp32
  float* lse;  // [Tq, Hq]
  long long wait_limit;
};

// Key tiles [0, nk) a query tile meets (tiles of BN keys, the last may be short).
__device__ __forceinline__ int block_n_kv(const BlockParams& p, int qt) {
  const int ntk = (p.Tk + BN - 1) / BN;
  if (!p.causal) return ntk;
  const int q_valid = min(BM, p.Tq - qt * BM);
  const long long last_q = p.q_pos0 + static_cast<long long>(qt) * BM + q_valid - 1;
  if (last_q < p.k_pos0) return 0;
  const long long seen = (last_q - p.k_pos0) / BN + 1;
  return static_cast<int>(seen < ntk ? seen : ntk);
}

// Causal mask of key tile kt for query row `row` of tile qt, by absolute position.
__device__ __forceinline__ void block_mask(const BlockParams& p, int qt, int kt, int row, int& col_lim,
                                           bool& masked) {
  const int kv_valid = min(BN, p.Tk - kt * BN);
  col_lim = kv_valid;
  masked = kv_valid < BN;
  if (p.causal) {
    const long long qpos = p.q_pos0 + static_cast<long long>(qt) * BM + row;
    const long long kpos0 = p.k_pos0 + static_cast<long long>(kt) * BN;
    const long long vis = qpos - kpos0 + 1;   // keys of this tile visible to the row
    col_lim = vis < 0 ? 0 : (vis > kv_valid ? kv_valid : static_cast<int>(vis));
    masked = masked || kpos0 + kv_valid - 1 > p.q_pos0 + static_cast<long long>(qt) * BM;
  }
}

// Block schedule for the two-head kernel (GQA groups of even size): one query
// tile and a head pair per CTA, key tiles 0..n-1 of the block in order, fp32
// partial output.
template <int D>
struct BlockPolicy : PolicyDefaults {
  using Args = BlockParams;
  struct KvPos {
    int kt;
    int32_t row;
  };
  const BlockParams& p;
  int qt, h0, g, nkv;
  __device__ BlockPolicy(const BlockParams& a, int idx) : p(a) {
    const int pairs = a.Hq / 2;
    h0 = 2 * (idx % pairs);
    qt = idx / pairs;
    g = h0 / a.group;
    nkv = block_n_kv(a, qt);
  }
  __device__ int tiles() const { return nkv > 0 ? 1 : 0; }
  __device__ int kvh() const { return g; }
  __device__ void set_tile(int) {}
  __device__ int q_head(int h) const { return h0 + h; }
  __device__ int32_t q_row(int) const { return qt * BM; }
  __device__ int q_valid(int) const { return min(BM, p.Tq - qt * BM); }
  __device__ int n_kv() const { return nkv; }
  __device__ void kv_begin(KvPos& k) const { k.kt = -1; }
  __device__ bool kv_next(KvPos& k) const {
    if (++k.kt >= nkv) return false;
    k.row = k.kt * BN;
    return true;
  }
  __device__ void mask(const KvPos& k, int, int row, int& col_lim, bool& masked) const {
    block_mask(p, qt, k.kt, row, col_lim, masked);
  }
  __device__ void store_o(int h, int row, int col0, const uint32_t (&o)[32], float inv_l) const {
    float* dst = p.o + (static_cast<int64_t>(qt * BM + row) * p.Hq + h0 + h) * D + col0;
#pragma unroll
    for (int i = 0; i < 32; i += 4)
      *reinterpret_cast<float4*>(dst + i) =
          make_float4(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l,
                      __uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
  }
  __device__ void store_lse(int h, int row, float lse) const {
    p.lse[static_cast<int64_t>(qt * BM + row) * p.Hq + h0 + h] = lse;
  }
  __device__ void write_empty(int tid, int nthreads) const {
    const int qv = q_valid(0);
    for (int i = tid; i < 2 * qv * D; i += nthreads) {
      const int h = i / (qv * D), r = (i / D) % qv, e = i % D;
      const int64_t at = static_cast<int64_t>(qt * BM + r) * p.Hq + h0 + h;
      p.o[at * D + e] = 0.f;
      if (e == 0) p.lse[at] = -CUDART_INF_F;
    }
  }
};

// Block schedule on adjacent query tiles, for any GQA group: one query head,
// query tiles 2i and 2i+1 as the two slots, the key tiles the later one meets
// (under the causal mask a superset of the earlier tile's).  A slot past the
// last query tile is empty.
template <int D>
struct BlockTilePolicy : PolicyDefaults {
  using Args = BlockParams;
  using KvPos = typename BlockPolicy<D>::KvPos;
  const BlockParams& p;
  int qp, hq, g, ntq, nkv;
  __device__ BlockTilePolicy(const BlockParams& a, int idx) : p(a) {
    hq = idx % a.Hq;
    qp = idx / a.Hq;
    g = hq / a.group;
    ntq = (a.Tq + BM - 1) / BM;
    nkv = block_n_kv(a, min(2 * qp + 1, ntq - 1));
  }
  __device__ int tiles() const { return nkv > 0 ? 1 : 0; }
  __device__ int kvh() const { return g; }
  __device__ void set_tile(int) {}
  __device__ int q_head(int) const { return hq; }
  __device__ int32_t q_row(int h) const { return (2 * qp + h) * BM; }
  __device__ int q_valid(int h) const { return max(0, min(BM, p.Tq - (2 * qp + h) * BM)); }
  __device__ int n_kv() const { return nkv; }
  __device__ void kv_begin(KvPos& k) const { k.kt = -1; }
  __device__ bool kv_next(KvPos& k) const {
    if (++k.kt >= nkv) return false;
    k.row = k.kt * BN;
    return true;
  }
  __device__ void mask(const KvPos& k, int h, int row, int& col_lim, bool& masked) const {
    block_mask(p, 2 * qp + h, k.kt, row, col_lim, masked);
  }
  __device__ void store_o(int h, int row, int col0, const uint32_t (&o)[32], float inv_l) const {
    float* dst = p.o + (static_cast<int64_t>((2 * qp + h) * BM + row) * p.Hq + hq) * D + col0;
#pragma unroll
    for (int i = 0; i < 32; i += 4)
      *reinterpret_cast<float4*>(dst + i) =
          make_float4(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l,
                      __uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
  }
  __device__ void store_lse(int h, int row, float lse) const {
    p.lse[static_cast<int64_t>((2 * qp + h) * BM + row) * p.Hq + hq] = lse;
  }
  __device__ void write_empty(int tid, int nthreads) const {
    for (int h = 0; h < 2; ++h) {
      const int qv = q_valid(h);
      for (int i = tid; i < qv * D; i += nthreads) {
        const int r = i / D, e = i % D;
        const int64_t at = static_cast<int64_t>((2 * qp + h) * BM + r) * p.Hq + hq;
        p.o[at * D + e] = 0.f;
        if (e == 0) p.lse[at] = -CUDART_INF_F;
      }
    }
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    block_attn_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const BlockParams p) {
  constexpr int SLABS = D / 64;
  constexpr uint32_t kTileBytes = BM * D * 2;
  constexpr uint32_t kIdescS = idesc_bf16_f32(BM, BN, 0, 0);
  constexpr uint32_t kIdescO = idesc_bf16_f32(BM, D, 0, 1);

  extern __shared__ uint8_t smem_raw[];
  Smem<D>& sm = *reinterpret_cast<Smem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.x % p.Hq, qt = blockIdx.x / p.Hq;
  const int g = hq / p.group;
  const int nkv = block_n_kv(p, qt);
  const int q_valid = min(BM, p.Tq - qt * BM);
  volatile int* abort_flag = &sm.abort_flag;
  const long long lim = p.wait_limit;

  if (nkv == 0) {  // every key of the block is after every query of the tile
    for (int i = threadIdx.x; i < q_valid * D; i += blockDim.x) {
      const int r = i / D, e = i % D;
      p.o[(static_cast<int64_t>(qt * BM + r) * p.Hq + hq) * D + e] = 0.f;
      if (e == 0) p.lse[static_cast<int64_t>(qt * BM + r) * p.Hq + hq] = -CUDART_INF_F;
    }
    return;
  }

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
      bool ok = true;
      // copies issued so far (stage phase of the last one), awaited before an aborted CTA exits
      bool q_iss = false, k_iss[STAGES] = {false, false}, v_iss[STAGES] = {false, false};
      uint32_t q_ph = 0, k_ph[STAGES] = {0, 0}, v_ph[STAGES] = {0, 0};
      const uint32_t qb = smem_u32(&sm.q_full);
      mbar_arrive_expect_tx(qb, kTileBytes);
      for (int s = 0; s < SLABS; ++s) tma_load_3d(smem_u32(sm.q + s * BM * 128), &tmQ, qb, 64 * s, hq, qt * BM);
      q_iss = true;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % STAGES;
        const uint32_t ph = (j / STAGES) & 1;
        if (!(ok = mbar_wait(smem_u32(&sm.k_empty[st]), ph ^ 1, abort_flag, lim, 302))) break;
        mbar_arrive_expect_tx(smem_u32(&sm.k_full[st]), kTileBytes);
        for (int s = 0; s < SLABS; ++s)
          tma_load_3d(smem_u32(sm.k[st] + s * BN * 128), &tmK, smem_u32(&sm.k_full[st]), 64 * s, g, j * BN);
          k_iss[st] = true;
          k_ph[st] = ph;
        if (!(ok = mbar_wait(smem_u32(&sm.v_empty[st]), ph ^ 1, abort_flag, lim, 303))) break;
        mbar_arrive_expect_tx(smem_u32(&sm.v_full[st]), kTileBytes);
        for (int s = 0; s < SLABS; ++s)
          tma_load_3d(smem_u32(sm.v[st] + s * BN * 128), &tmV, smem_u32(&sm.v_full[st]), 64 * s, g, j * BN);
          v_iss[st] = true;
          v_ph[st] = ph;
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
      bool ok = mbar_wait(smem_u32(&sm.q_full), 0, abort_flag, lim, 310);
      const uint32_t q_base = smem_u32(sm.q), p_base = smem_u32(sm.p);
      uint32_t pv_cnt = 0;
      auto do_pv = [&](int jj) -> bool {
        const int st = jj % STAGES;
        if (!mbar_wait(smem_u32(&sm.p_full), pv_cnt & 1, abort_flag, lim, 311)) return false;
        if (!mbar_wait(smem_u32(&sm.v_full[st]), (jj / STAGES) & 1, abort_flag, lim, 312)) return false;
        tc_fence_after();
        const uint32_t v_base = smem_u32(sm.v[st]);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ss(tmem + kColO, desc_sw128(p_base + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024),
                      desc_sw128(v_base + kk * 16 * 128, BN * 128, 1024), kIdescO, (kk > 0 || jj > 0) ? 1u : 0u);
        mma_commit(smem_u32(&sm.pv_done));
        mma_commit(smem_u32(&sm.v_empty[st]));
        ++pv_cnt;
        return true;
      };
      for (int j = 0; j < nkv && ok; ++j) {
        const int st = j % STAGES, sb = j & 1;
        if (!(ok = mbar_wait(smem_u32(&sm.k_full[st]), (j / STAGES) & 1, abort_flag, lim, 314))) break;
        if (!(ok = mbar_wait(smem_u32(&sm.s_empty[sb]), ((j >> 1) & 1) ^ 1, abort_flag, lim, 315))) break;
        tc_fence_after();
        const uint32_t k_base = smem_u32(sm.k[st]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + kColS0 + sb * BN, desc_sw128(q_base + off, 16, 1024),
                      desc_sw128(k_base + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16, 1024), kIdescS,
                      kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm.s_full[sb]));
        mma_commit(smem_u32(&sm.k_empty[st]));
        if (j > 0 && !(ok = do_pv(j - 1))) break;
      }
      if (ok) ok = do_pv(nkv - 1);
      mma_commit(smem_u32(&sm.drain));
      if (!mbar_wait_quiesce(smem_u32(&sm.drain), 0, ok ? lim : (1 << 22)) && ok) {
        *abort_flag = 1;
        ra_record_error(RA_ERR_TIMEOUT, 316);
      }
    }
  } else if (warp >= 2) {
    // ============================================================ softmax + epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t p_base = smem_u32(sm.p);
    float m = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      int col_lim;
      bool masked;
      block_mask(p, qt, j, row, col_lim, masked);
      if (!(ok = mbar_wait(smem_u32(&sm.s_full[sb]), (j >> 1) & 1, abort_flag, lim, 320))) break;
      tc_fence_after();
      uint32_t pk[BN / 2];
      const float alpha = softmax_row(t_lane + kColS0 + sb * BN, j, masked, col_lim, p.scale_log2, m, l, pk);
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.s_empty[sb]));
      if (j > 0) {
        // P_{j-1} V_{j-1} must be complete: P buffer reuse and O rescale
        if (!(ok = mbar_wait(smem_u32(&sm.pv_done), (j - 1) & 1, abort_flag, lim, 321))) break;
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
#pragma unroll
      for (int ch = 0; ch < BN / 8; ++ch) {
        const int slab = ch >> 3, c16 = ch & 7;
        const uint32_t addr = p_base + slab * (BM * 128) + row * 128 + ((c16 ^ (row & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * ch]), "r"(pk[4 * ch + 1]),
                     "r"(pk[4 * ch + 2]), "r"(pk[4 * ch + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.p_full));
    }
    if (ok && mbar_wait(smem_u32(&sm.pv_done), (nkv - 1) & 1, abort_flag, lim, 322)) {
      tc_fence_after();
      const bool live = l > 0.f;
      const float inv_l = live ? 1.f / l : 0.f;
      const bool row_ok = row < q_valid;
      float* orow = p.o + (static_cast<int64_t>(qt * BM + row) * p.Hq + hq) * D;
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t orr[32];
        tmem_ld32(t_lane + kColO + 32 * c4, orr);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(orow + 32 * c4 + i) =
                make_float4(__uint_as_float(orr[i]) * inv_l, __uint_as_float(orr[i + 1]) * inv_l,
                            __uint_as_float(orr[i + 2]) * inv_l, __uint_as_float(orr[i + 3]) * inv_l);
        }
      }
      if (row_ok)
        p.lse[static_cast<int64_t>(qt * BM + row) * p.Hq + hq] = live ? (m + log2f(l)) * kLn2 : -CUDART_INF_F;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
ra_status launch_block(const void* q, const void* k, const void* v, const BlockParams& bp, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  ra_status st;
  if ((st = make_map(&mq, q, D, bp.Hq, bp.Tq)) != RA_OK) return st;
  if ((st = make_map(&mk, k, D, bp.Hkv, bp.Tk)) != RA_OK) return st;
  if ((st = make_map(&mv, v, D, bp.Hkv, bp.Tk)) != RA_OK) return st;
  if (bp.group % 2 == 0) {  // two query heads of one GQA group per CTA
    const size_t smem = sizeof(Smem2<D>) + 1024;
    RA_CUDA_TRY(cudaFuncSetAttribute(attn_pair_kernel<D, BlockPolicy<D>>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)));
    const int64_t grid = ra::ceil_div(bp.Tq, BM) * (bp.Hq / 2);
    attn_pair_kernel<D, BlockPolicy<D>><<<static_cast<unsigned>(grid), kThreads2, smem, stream>>>(mq, mk, mv, bp);
    RA_LAUNCH_CHECK("attn_pair_kernel<BlockPolicy>");
    return RA_OK;
  }
  if (ra::ceil_div(bp.Tq, BM) >= 2) {  // two adjacent query tiles of one head per CTA
    const size_t smem = sizeof(Smem2<D>) + 1024;
    RA_CUDA_TRY(cudaFuncSetAttribute(attn_pair_kernel<D, BlockTilePolicy<D>>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
    const int64_t grid = ra::ceil_div(ra::ceil_div(bp.Tq, BM), 2) * bp.Hq;
    attn_pair_kernel<D, BlockTilePolicy<D>><<<static_cast<unsigned>(grid), kThreads2, smem, stream>>>(mq, mk, mv,
                                                                                                       bp);
    RA_LAUNCH_CHECK("attn_pair_kernel<BlockTilePolicy>");
    return RA_OK;
  }
  const size_t smem = sizeof(Smem<D>) + 1024;
  RA_CUDA_TRY(cudaFuncSetAttribute(block_attn_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem)));
  const int64_t grid = ra::ceil_div(bp.Tq, BM) * bp.Hq;
  block_attn_bf16_kernel<D><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(mq, mk, mv, bp);
  RA_LAUNCH_CHECK("block_attn_bf16_kernel");
  return RA_OK;
}

ra_status check_block_args(const void* q, const void* k, const void* v, int32_t Tq, int32_t Tk, int32_t Hq,
                           int32_t Hkv, int32_t d, int64_t q_pos0, int64_t k_pos0) {
  RA_REQUIRE(Tq >= 1 && Tk >= 1 && Hq >= 1 && Hkv >= 1, "Tq, Tk, Hq, Hkv must be >= 1");
  RA_REQUIRE(Hq % Hkv == 0, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  RA_REQUIRE(q_pos0 >= 0 && k_pos0 >= 0, "positions must be >= 0");
  if (d != 64 && d != 128) return ra::fail(RA_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", d);
  RA_REQUIRE(q && k && v, "NULL pointer");
  RA_REQUIRE(ra::aligned16(q) && ra::aligned16(k) && ra::aligned16(v), "q, k, v must be 16-byte aligned");
  RA_REQUIRE(static_cast<int64_t>(ra::ceil_div(Tq, BM)) * Hq < (int64_t(1) << 31), "grid too large");
  return RA_OK;
}
}  // namespace

extern "C" ra_status ra_attn_block_fwd(const void* q, const void* k, const void* v, int32_t Tq, int32_t Tk,
                                       int32_t Hq, int32_t Hkv, int32_t d, int64_t q_pos0, int64_t k_pos0,
                                       int32_t causal, float scale, float* o_part, float* lse_part,
                                       ra_stream stream) {
  ra::clear_error();
  ra_status st = check_block_args(q, k, v, Tq, Tk, Hq, Hkv, d, q_pos0, k_pos0);
  if (st != RA_OK) return st;
  RA_REQUIRE(o_part && lse_part && ra::aligned16(o_part) && reinterpret_cast<uintptr_t>(lse_part) % 4 == 0,
             "o_part must be 16-byte aligned, lse_part 4-byte aligned");
  BlockParams bp;
  bp.Tq = Tq; bp.Tk = Tk; bp.Hq = Hq; bp.Hkv = Hkv; bp.group = Hq / Hkv; bp.causal = causal ? 1 : 0;
  bp.q_pos0 = q_pos0; bp.k_pos0 = k_pos0;
  bp.scale_log2 = (scale > 0.f ? scale : 1.f / sqrtf(static_cast<float>(d))) * 1.4426950408889634f;
  bp.o = o_part; bp.lse = lse_part; bp.wait_limit = ra::wait_limit();
  return d == 128 ? launch_block<128>(q, k, v, bp, stream) : launch_block<64>(q, k, v, bp, stream);
}

extern "C" ra_status ra_segmented_prefill_workspace_size(int32_t Tq, int32_t Tk, int32_t Hq, int32_t d,
                                                         int32_t seg_tokens, size_t* bytes) {
  ra::clear_error();
  RA_REQUIRE(bytes != nullptr, "bytes is NULL");
  RA_REQUIRE(Tq >= 1 && Tk >= 1 && Hq >= 1 && d >= 1 && seg_tokens >= 1, "sizes must be >= 1");
  const int64_t P = ra::ceil_div(Tk, seg_tokens);
  const int64_t o_bytes = P * Tq * Hq * d * 4;
  *bytes = static_cast<size_t>(ra::ceil_div(o_bytes, 256) * 256 + P * Tq * Hq * 4);
  return RA_OK;
}

extern "C" ra_status ra_segmented_prefill_fwd(const void* q, const void* k, const void* v, int32_t Tq, int32_t Tk,
                                              int32_t Hq, int32_t Hkv, int32_t d, int64_t q_pos0, int32_t causal,
                                              float scale, int32_t seg_tokens, void* o, ra_dtype out_dt, float* lse,
                                              void* workspace, size_t ws_bytes, ra_stream stream) {
  ra::clear_error();
  ra_status st = check_block_args(q, k, v, Tq, Tk, Hq, Hkv, d, q_pos0, 0);
  if (st != RA_OK) return st;
  RA_REQUIRE(seg_tokens >= 1, "seg_tokens must be >= 1");
  RA_REQUIRE(out_dt == RA_F32 || out_dt == RA_BF16, "unknown out dtype");
  RA_REQUIRE(o && workspace && ra::aligned16(o) && ra::aligned16(workspace), "o/workspace must be 16-byte aligned");
  size_t need = 0;
  if ((st = ra_segmented_prefill_workspace_size(Tq, Tk, Hq, d, seg_tokens, &need)) != RA_OK) return st;
  RA_REQUIRE(ws_bytes >= need, "workspace too small (%zu < %zu bytes)", ws_bytes, need);
  const int64_t P = ra::ceil_div(Tk, seg_tokens);
  float* o_parts = static_cast<float*>(workspace);
  float* lse_parts = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                              ra::ceil_div(P * Tq * Hq * d * 4, 256) * 256);
  const size_t kv_row = static_cast<size_t>(Hkv) * d * 2;
  for (int64_t sgi = 0; sgi < P; ++sgi) {
    const int64_t k0 = sgi * seg_tokens;
    const int32_t tk = static_cast<int32_t>(std::min<int64_t>(seg_tokens, Tk - k0));
    st = ra_attn_block_fwd(q, static_cast<const char*>(k) + k0 * kv_row, static_cast<const char*>(v) + k0 * kv_row,
                           Tq, tk, Hq, Hkv, d, q_pos0, k0, causal, scale, o_parts + sgi * Tq * Hq * d,
                           lse_parts + sgi * Tq * Hq, stream);
    if (st != RA_OK) return st;
  }
  return ra_lse_merge(o_parts, lse_parts, static_cast<int32_t>(P), Tq, Hq, d, o, out_dt, lse, stream);
}
