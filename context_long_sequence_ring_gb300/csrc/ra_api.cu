// Error handling, device status, the zigzag (head-tail) partition, row
// gathers for permute/restore, the synthetic-input generator and the
// bounded-wait self test.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "ra_common.cuh"
#include "ra_sm100.cuh"
#include "ringattn_synth.h"

namespace ra {

static thread_local std::string t_last_error;

void clear_error() { t_last_error.clear(); }

ra_status fail(ra_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (t_last_error.empty()) t_last_error = buf;
  return s;
}

ra_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return RA_OK;
  return fail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace ra

RA_DEFINE_ERROR_FETCH(fetch_error_api)

extern "C" const char* ra_last_error(void) { return ra::t_last_error.c_str(); }

extern "C" const char* ra_version(void) { return "ringattn 0.1 (sm_103a)"; }

extern "C" ra_status ra_device_status(ra_stream stream) {
  ra::clear_error();
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return ra::cuda_status(e, "cudaStreamSynchronize");
  int (*fetch[])(int*) = {ra::fetch_error_api, ra::fetch_error_cache, ra::fetch_error_decode,
                          ra::fetch_error_attn_f32, ra::fetch_error_attn_bf16, ra::fetch_error_attn_block,
                          ra::fetch_error_rope, ra::fetch_error_ring_step};
  const char* names[] = {"partition/gather", "kv cache", "decode/merge", "attention fp32",
                         "ring attention bf16", "block attention bf16", "rope gather", "ring step"};
  static_assert(sizeof(fetch) / sizeof(fetch[0]) == sizeof(names) / sizeof(names[0]),
                "one name per module error word");
  ra_status first = RA_OK;
  for (size_t i = 0; i < sizeof(fetch) / sizeof(fetch[0]); ++i) {
    int where = 0;
    int s = fetch[i](&where);
    if (s < 0) return ra::fail(RA_ERR_CUDA, "reading the device error word failed");
    if (s != 0 && first == RA_OK) {
      first = static_cast<ra_status>(s);
      ra::fail(first, "device error %d in %s kernels (site %d)", s, names[i], where);
    }
  }
  return first;
}

// ===========================================================================
// Zigzag partition (vLLM-Ascend "Context Parallel (CP)", PCP head-tail
// partition).  One thread per padded position p of one sequence:
//   chunk = p / c, offset = p % c, rank = chunk < N ? chunk : 2N-1-chunk,
//   half = chunk < N ? 0 : 1,
//   gathered g = rank * (tokens per rank region) + (this request's start in
//   the rank region) + half * c + offset.
// Sequences are handed to the kernel in batches through the parameter block.
// ===========================================================================
namespace {

constexpr int kZigzagBatch = 256;

struct ZigzagBatch {
  int64_t len[kZigzagBatch];         // L_q
  int64_t orig_start[kZigzagBatch];  // first original index of the request
  int64_t rank_off[kZigzagBatch];    // start of the request inside a rank region
  int64_t region;                    // tokens per rank region = sum_q 2*c_q
  int32_t n;                         // sequences in this batch
  int32_t N;                         // ranks
};

__global__ void zigzag_kernel(const __grid_constant__ ZigzagBatch zb, int32_t* perm,
                              int32_t* restore) {
  const int q = blockIdx.y;
  const int64_t L = zb.len[q];
  const int64_t N2 = 2 * static_cast<int64_t>(zb.N);
  const int64_t c = (L + N2 - 1) / N2;
  const int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (p >= c * N2) return;
  const int64_t chunk = p / c;
  const int64_t off = p - chunk * c;
  const int64_t rank = chunk < zb.N ? chunk : N2 - 1 - chunk;
  const int64_t half = chunk < zb.N ? 0 : 1;
  const int64_t g = rank * zb.region + zb.rank_off[q] + half * c + off;
  if (p < L) {
    perm[g] = static_cast<int32_t>(zb.orig_start[q] + p);
    restore[zb.orig_start[q] + p] = static_cast<int32_t>(g);
  } else {
    perm[g] = -1;
  }
}

// dst[i] = src[idx[i]] (zero row when idx < 0).  One warp per row, 16-byte
// (or 4-/1-byte) words, grid-stride over rows.
template <typename W>
__global__ void gather_rows_kernel(const W* __restrict__ src, int64_t src_rows,
                                   const int32_t* __restrict__ idx, W* __restrict__ dst,
                                   int64_t rows, int64_t words) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t r = warp; r < rows; r += nwarps) {
    const int32_t s = idx[r];
    W* d = dst + r * words;
    if (s >= 0 && s < src_rows) {
      const W* a = src + static_cast<int64_t>(s) * words;
      for (int64_t w = lane; w < words; w += 32) d[w] = a[w];
    } else {
      if (s >= src_rows && lane == 0) ra_record_error(RA_ERR_DEVICE_BOUNDS, 1);
      const W z{};
      for (int64_t w = lane; w < words; w += 32) d[w] = z;
    }
  }
}

// ---------------------------------------------------------------- synth fill
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

template <typename T>
__global__ void synth_fill_kernel(uint64_t key, int64_t n, const T* __restrict__ table,
                                  T* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const uint64_t u = mix64(key + static_cast<uint64_t>(i + 1) * 0x9E3779B97F4A7C15ull);
    out[i] = table[u >> 48];
  }
}

// ---------------------------------------------------------------- self test
__global__ void wait_timeout_kernel(long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = ra::sm100::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ra::sm100::mbar_init(b, 1);
    abort_flag = 0;
    ra::sm100::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nobody arrives: phase 0 never completes, so this wait must expire
    ra::sm100::mbar_wait(b, 0, &abort_flag, limit, 99);
  }
  __syncthreads();
}

}  // namespace

extern "C" ra_status ra_zigzag_partition(const int64_t* seq_lens, int32_t num_seqs,
                                         int32_t n_ranks, int32_t* perm, int32_t* restore,
                                         int64_t* padded_total, int64_t* total,
                                         ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(num_seqs >= 0, "num_seqs must be >= 0 (got %d)", num_seqs);
  RA_REQUIRE(n_ranks >= 1, "n_ranks must be >= 1 (got %d)", n_ranks);
  RA_REQUIRE(num_seqs == 0 || seq_lens != nullptr, "seq_lens is NULL");
  const int64_t N2 = 2 * static_cast<int64_t>(n_ranks);
  int64_t G = 0, T = 0;
  std::vector<int64_t> rank_off(num_seqs), orig(num_seqs);
  for (int32_t q = 0; q < num_seqs; ++q) {
    RA_REQUIRE(seq_lens[q] >= 0, "seq_lens[%d] is negative", q);
    const int64_t c = ra::ceil_div(seq_lens[q], N2);
    rank_off[q] = G / n_ranks;  // every request adds 2c to each rank region
    orig[q] = T;
    G += c * N2;
    T += seq_lens[q];
    RA_REQUIRE(G < (int64_t(1) << 31), "padded total exceeds int32 indexing");
  }
  if (padded_total) *padded_total = G;
  if (total) *total = T;
  if (perm == nullptr || restore == nullptr || G == 0) return RA_OK;
  RA_REQUIRE(reinterpret_cast<uintptr_t>(perm) % 4 == 0 &&
                 reinterpret_cast<uintptr_t>(restore) % 4 == 0,
             "perm/restore must be 4-byte aligned");
  const int64_t region = G / n_ranks;
  for (int32_t q0 = 0; q0 < num_seqs; q0 += kZigzagBatch) {
    ZigzagBatch zb;
    memset(&zb, 0, sizeof(zb));
    zb.n = std::min(kZigzagBatch, num_seqs - q0);
    zb.N = n_ranks;
    zb.region = region;
    int64_t maxp = 0;
    for (int i = 0; i < zb.n; ++i) {
      zb.len[i] = seq_lens[q0 + i];
      zb.orig_start[i] = orig[q0 + i];
      zb.rank_off[i] = rank_off[q0 + i];
      maxp = std::max(maxp, ra::ceil_div(zb.len[i], N2) * N2);
    }
    if (maxp == 0) continue;
    dim3 grid(static_cast<unsigned>(ra::ceil_div(maxp, 256)), zb.n);
    zigzag_kernel<<<grid, 256, 0, stream>>>(zb, perm, restore);
    RA_LAUNCH_CHECK("zigzag_kernel");
  }
  return RA_OK;
}

extern "C" ra_status ra_gather_rows(const void* src, int64_t src_rows, const int32_t* idx,
                                    void* dst, int64_t rows, int64_t row_bytes,
                                    ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(rows >= 0 && src_rows >= 0 && row_bytes >= 0, "negative size");
  if (rows == 0 || row_bytes == 0) return RA_OK;
  RA_REQUIRE(src && idx && dst, "NULL pointer");
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
  const int64_t total_warps = rows;
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>(ra::ceil_div(total_warps * 32, threads), 152 * 64);
  if (row_bytes % 16 == 0 && (a & 15) == 0) {
    gather_rows_kernel<uint4><<<blocks, threads, 0, stream>>>(
        static_cast<const uint4*>(src), src_rows, idx, static_cast<uint4*>(dst), rows,
        row_bytes / 16);
  } else if (row_bytes % 4 == 0 && (a & 3) == 0) {
    gather_rows_kernel<uint32_t><<<blocks, threads, 0, stream>>>(
        static_cast<const uint32_t*>(src), src_rows, idx, static_cast<uint32_t*>(dst), rows,
        row_bytes / 4);
  } else {
    gather_rows_kernel<uint8_t><<<blocks, threads, 0, stream>>>(
        static_cast<const uint8_t*>(src), src_rows, idx, static_cast<uint8_t*>(dst), rows,
        row_bytes);
  }
  RA_LAUNCH_CHECK("gather_rows_kernel");
  return RA_OK;
}

extern "C" ra_status ra_synth_fill(uint64_t key, int64_t n, const void* table,
                                   int32_t elem_bytes, void* out, ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(n >= 0, "n must be >= 0");
  RA_REQUIRE(elem_bytes == 2 || elem_bytes == 4, "elem_bytes must be 2 or 4");
  if (n == 0) return RA_OK;
  RA_REQUIRE(table && out, "NULL pointer");
  const int64_t blocks = std::min<int64_t>(ra::ceil_div(n, 256), 152 * 32);
  if (elem_bytes == 2)
    synth_fill_kernel<uint16_t><<<blocks, 256, 0, stream>>>(
        key, n, static_cast<const uint16_t*>(table), static_cast<uint16_t*>(out));
  else
    synth_fill_kernel<uint32_t><<<blocks, 256, 0, stream>>>(
        key, n, static_cast<const uint32_t*>(table), static_cast<uint32_t*>(out));
  RA_LAUNCH_CHECK("synth_fill_kernel");
  return RA_OK;
}

extern "C" ra_status ra_selftest_wait_timeout(int64_t limit_cycles, ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(limit_cycles > 0 && limit_cycles <= (int64_t(1) << 34),
             "limit_cycles must be in (0, 2^34]");
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_cycles);
  RA_LAUNCH_CHECK("wait_timeout_kernel");
  return RA_OK;
}
