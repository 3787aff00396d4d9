// Context-parallel KV cache: the interleaved slot mapping and the scatter of
// token K/V rows into the sharded paged cache.
// Source: vLLM-Ascend developer guide "Context Parallel (CP)", section
// "Block table" (virtual blocks of block_size*pcp*dcp tokens, device =
// local_block_index % (pcp*dcp), interleave granularity, and the rule
// block_size % interleave == 0).
#include "ra_common.cuh"

RA_DEFINE_ERROR_FETCH(fetch_error_cache)

namespace {

// Largest q with qsl[q] <= t (qsl non-decreasing, qsl[0] = 0).
__device__ __forceinline__ int request_of(const int32_t* __restrict__ qsl, int R, int64_t t) {
  int lo = 0, hi = R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(qsl[mid]) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void slot_mapping_kernel(const int32_t* __restrict__ qsl, int32_t R,
                                    const int32_t* __restrict__ positions,
                                    const int32_t* __restrict__ block_table, int32_t max_vb,
                                    int64_t T, int32_t block_size, int32_t interleave, int32_t W,
                                    int32_t* __restrict__ slot_out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < T;
       t += stride) {
    const int q = request_of(qsl, R, t);
    const int64_t x = positions[t];
    const int64_t V = static_cast<int64_t>(block_size) * W;  // virtual block size
    const int64_t vb = x / V;
    const int64_t o = x - vb * V;                // offset in the virtual block
    const int64_t lbi = o / interleave;          // local block index
    const int dev = static_cast<int>(lbi % W);   // owning device
    const int64_t off = (lbi / W) * interleave + (o % interleave);
    int32_t slot = -1;
    bool ok = x >= 0 && vb < max_vb;
    if (ok) {
      const int32_t blk = block_table[static_cast<int64_t>(q) * max_vb + vb];
      ok = blk >= 0;
      if (ok) slot = static_cast<int32_t>(static_cast<int64_t>(blk) * block_size + off);
    }
    if (!ok) ra_record_error(RA_ERR_DEVICE_BOUNDS, 10);
    for (int w = 0; w < W; ++w) slot_out[static_cast<int64_t>(w) * T + t] = (ok && w == dev) ? slot : -1;
  }
}

// One warp per token: find the owning device, copy the token's Hkv*d row of
// K and of V into cache[w][slot / bs][g][slot % bs][:] for every head g.
template <typename E>
__global__ void kv_scatter_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                  const int32_t* __restrict__ slot, uint4* __restrict__ kc,
                                  uint4* __restrict__ vc, int64_t T, int32_t W, int32_t Hkv,
                                  int32_t d_words, int32_t block_size, int64_t num_blocks) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t t = warp; t < T; t += nwarps) {
    for (int w = 0; w < W; ++w) {
      const int32_t s = slot[static_cast<int64_t>(w) * T + t];
      if (s < 0) continue;
      const int64_t blk = s / block_size, j = s % block_size;
      if (blk >= num_blocks) {
        if (lane == 0) ra_record_error(RA_ERR_DEVICE_BOUNDS, 11);
        continue;
      }
      const int64_t row_words = static_cast<int64_t>(Hkv) * d_words;
      for (int64_t e = lane; e < row_words; e += 32) {
        const int64_t g = e / d_words, u = e % d_words;
        const int64_t dst = (((static_cast<int64_t>(w) * num_blocks + blk) * Hkv + g) * block_size + j) *
                                d_words + u;
        kc[dst] = k[t * row_words + e];
        vc[dst] = v[t * row_words + e];
      }
    }
  }
}

// One warp per output row: locate token positions[t] of its request in the
// sharded cache with the block-table formula and copy its Hkv*d row of K and
// of V (the reorg that makes each request's KV contiguous again).
__global__ void kv_gather_kernel(const uint4* __restrict__ kc, const uint4* __restrict__ vc,
                                 const int32_t* __restrict__ block_table, int32_t max_vb,
                                 const int32_t* __restrict__ qsl, int32_t R, const int32_t* __restrict__ positions,
                                 int64_t T, int32_t Hkv, int32_t d_words, int32_t block_size, int32_t interleave,
                                 int32_t W, int64_t num_blocks, uint4* __restrict__ k_out, uint4* __restrict__ v_out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t row_words = static_cast<int64_t>(Hkv) * d_words;
  for (int64_t t = warp; t < T; t += nwarps) {
    const int q = request_of(qsl, R, t);
    const int64_t x = positions[t];
    const int64_t V = static_cast<int64_t>(block_size) * W;
    const int64_t vb = x / V;
    const int64_t o = x - vb * V;
    const int64_t lbi = o / interleave;
    const int64_t dev = lbi % W;
    const int64_t off = (lbi / W) * interleave + (o % interleave);
    int64_t blk = -1;
    if (x >= 0 && vb < max_vb) blk = block_table[static_cast<int64_t>(q) * max_vb + vb];
    uint4* kd = k_out + t * row_words;
    uint4* vd = v_out + t * row_words;
    if (blk < 0 || blk >= num_blocks) {
      if (lane == 0) ra_record_error(RA_ERR_DEVICE_BOUNDS, 12);
      for (int64_t e = lane; e < row_words; e += 32) kd[e] = vd[e] = make_uint4(0, 0, 0, 0);
      continue;
    }
    for (int64_t e = lane; e < row_words; e += 32) {
      const int64_t g = e / d_words, u = e % d_words;
      const int64_t src = (((dev * num_blocks + blk) * Hkv + g) * block_size + off) * d_words + u;
      kd[e] = kc[src];
      vd[e] = vc[src];
    }
  }
}

}  // namespace

extern "C" ra_status ra_cp_kv_gather(const void* k_cache, const void* v_cache, const int32_t* block_table,
                                     int32_t max_vblocks, const int32_t* query_start_loc, const int32_t* positions,
                                     int32_t R, int64_t T, int32_t Hkv, int32_t d, int32_t block_size,
                                     int32_t interleave, int32_t pcp, int32_t dcp, int64_t num_blocks, ra_dtype dt,
                                     void* k_out, void* v_out, ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(block_size >= 1 && interleave >= 1 && pcp >= 1 && dcp >= 1,
             "block_size, interleave, pcp and dcp must be >= 1");
  RA_REQUIRE(block_size % interleave == 0,
             "block_size %% cp_kv_cache_interleave_size must be 0 (block_size=%d, interleave=%d)",
             block_size, interleave);
  RA_REQUIRE(R >= 1 && T >= 0 && max_vblocks >= 1 && Hkv >= 1 && d >= 1 && num_blocks >= 1, "sizes must be positive");
  RA_REQUIRE(dt == RA_BF16 || dt == RA_F32, "unknown dtype");
  const int64_t row_bytes = static_cast<int64_t>(d) * (dt == RA_BF16 ? 2 : 4);
  if (row_bytes % 16 != 0) return ra::fail(RA_ERR_UNSUPPORTED, "d*elem_size must be a multiple of 16");
  if (T == 0) return RA_OK;
  RA_REQUIRE(k_cache && v_cache && block_table && query_start_loc && positions && k_out && v_out, "NULL pointer");
  RA_REQUIRE(ra::aligned16(k_cache) && ra::aligned16(v_cache) && ra::aligned16(k_out) && ra::aligned16(v_out),
             "cache and output pointers must be 16-byte aligned");
  const int64_t blocks = std::min<int64_t>(ra::ceil_div(T * 32, 256), 152 * 32);
  kv_gather_kernel<<<blocks, 256, 0, stream>>>(
      static_cast<const uint4*>(k_cache), static_cast<const uint4*>(v_cache), block_table, max_vblocks,
      query_start_loc, R, positions, T, Hkv, static_cast<int32_t>(row_bytes / 16), block_size, interleave, pcp * dcp,
      num_blocks, static_cast<uint4*>(k_out), static_cast<uint4*>(v_out));
  RA_LAUNCH_CHECK("kv_gather_kernel");
  return RA_OK;
}

extern "C" ra_status ra_cp_slot_mapping(const int32_t* query_start_loc, const int32_t* positions,
                                        const int32_t* block_table, int32_t max_vblocks, int32_t R,
                                        int64_t T, int32_t block_size, int32_t interleave,
                                        int32_t pcp, int32_t dcp, int32_t* slot_out,
                                        ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(block_size >= 1 && interleave >= 1 && pcp >= 1 && dcp >= 1,
             "block_size, interleave, pcp and dcp must be >= 1");
  RA_REQUIRE(block_size % interleave == 0,
             "block_size %% cp_kv_cache_interleave_size must be 0 (block_size=%d, interleave=%d)",
             block_size, interleave);
  RA_REQUIRE(R >= 1 && T >= 0 && max_vblocks >= 1, "R >= 1, T >= 0, max_vblocks >= 1 required");
  RA_REQUIRE(static_cast<int64_t>(pcp) * dcp <= 4096, "pcp*dcp too large");
  if (T == 0) return RA_OK;
  RA_REQUIRE(query_start_loc && positions && block_table && slot_out, "NULL pointer");
  const int W = pcp * dcp;
  const int64_t blocks = std::min<int64_t>(ra::ceil_div(T, 256), 152 * 16);
  slot_mapping_kernel<<<blocks, 256, 0, stream>>>(query_start_loc, R, positions, block_table,
                                                  max_vblocks, T, block_size, interleave, W,
                                                  slot_out);
  RA_LAUNCH_CHECK("slot_mapping_kernel");
  return RA_OK;
}

extern "C" ra_status ra_cp_kv_scatter(const void* k, const void* v, const int32_t* slot,
                                      void* k_cache, void* v_cache, int64_t T, int32_t W,
                                      int32_t Hkv, int32_t d, int32_t block_size,
                                      int64_t num_blocks, ra_dtype dt, ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(T >= 0 && W >= 1 && Hkv >= 1 && d >= 1 && block_size >= 1 && num_blocks >= 1,
             "sizes must be positive");
  RA_REQUIRE(dt == RA_BF16 || dt == RA_F32, "unknown dtype");
  const int64_t row_bytes = static_cast<int64_t>(d) * (dt == RA_BF16 ? 2 : 4);
  if (row_bytes % 16 != 0) return ra::fail(RA_ERR_UNSUPPORTED, "d*elem_size must be a multiple of 16");
  if (T == 0) return RA_OK;
  RA_REQUIRE(k && v && slot && k_cache && v_cache, "NULL pointer");
  RA_REQUIRE(ra::aligned16(k) && ra::aligned16(v) && ra::aligned16(k_cache) && ra::aligned16(v_cache),
             "K/V and cache pointers must be 16-byte aligned");
  const int64_t blocks = std::min<int64_t>(ra::ceil_div(T * 32, 256), 152 * 32);
  kv_scatter_kernel<uint4><<<blocks, 256, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), T, W, Hkv,
      static_cast<int32_t>(row_bytes / 16), block_size, num_blocks);
  RA_LAUNCH_CHECK("kv_scatter_kernel");
  return RA_OK;
}
