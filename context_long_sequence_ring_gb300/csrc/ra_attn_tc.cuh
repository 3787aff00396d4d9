// Shared pieces of the tcgen05 attention kernels (ring-order and block
// partial): tile constants, the shared-memory layout of a one-head pipeline,
// the online-softmax step of one score row held in tensor memory, and the
// host-side TMA tensor-map encoding.  Included by each attention translation
// unit; everything here has internal linkage.
#pragma once

#include <cuda.h>
#include <math_constants.h>

#include <cstdlib>

#include "ra_common.cuh"
#include "ra_sm100.cuh"

namespace {

using namespace ra::sm100;

constexpr int BM = 128;       // query rows per tile
constexpr int BN = 128;       // keys per K/V tile
constexpr int STAGES = 2;     // K/V shared-memory ring depth
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColO = 2 * BN;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct __align__(1024) Smem {
  uint8_t q[BM * D * 2];
  uint8_t k[STAGES][BN * D * 2];
  uint8_t v[STAGES][BN * D * 2];
  uint8_t p[BM * BN * 2];
  uint64_t q_full, q_empty, k_full[STAGES], k_empty[STAGES], v_full[STAGES], v_empty[STAGES];
  uint64_t s_full[2], s_empty[2], p_full, pv_done, o_empty, drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ uint32_t f2_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 2^x with the SFU instruction (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ softmax of one row
__device__ __forceinline__ uint64_t f2pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Columns [c0, c0+32) of a score row: mask (when asked) and return the max.
__device__ __forceinline__ float chunk_mask_max(uint32_t (&x)[32], int c0, bool masked, int col_lim) {
  if (masked) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (c0 + i >= col_lim) x[i] = __float_as_uint(-CUDART_INF_F);
  }
  float mx[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) mx[k] = __uint_as_float(x[k]);
#pragma unroll
  for (int i = 4; i < 32; i += 8)
#pragma unroll
    for (int k = 0; k < 4; ++k) mx[k] = fmax3(mx[k], __uint_as_float(x[i + k]), __uint_as_float(x[i + 4 + k]));
  return fmax3(fmax3(mx[0], mx[1], mx[2]), mx[3], mx[3]);
}

// p = 2^(s*scale - m_ref) for 32 columns, packed to bf16 pairs into pk[0..16); adds the
// fp32 sums into two packed accumulators.
__device__ __forceinline__ void chunk_exp_pack(const uint32_t (&x)[32], uint64_t sc2, uint64_t negm2,
                                               uint64_t& acc0, uint64_t& acc1, uint32_t* pk) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    float t0, t1;
    f2unpack(ffma2(f2pack(__uint_as_float(x[i]), __uint_as_float(x[i + 1])), sc2, negm2), t0, t1);
    const float p0 = ex2(t0), p1 = ex2(t1);
    if ((i >> 1) & 1) acc1 = fadd2(acc1, f2pack(p0, p1)); else acc0 = fadd2(acc0, f2pack(p0, p1));
    pk[i >> 1] = f2_bf16x2(p0, p1);
  }
}

// Columns [c0, c0+32) of a score row at or past col_lim become -inf (masked).
__device__ __forceinline__ void chunk_mask(uint32_t (&x)[32], int c0, int col_lim) {
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (c0 + i >= col_lim) x[i] = __float_as_uint(-CUDART_INF_F);
}

// Largest sum of one 32-column chunk of p = 2^(s*scale - m) that keeps the
// stale reference m: every p of the chunk is then at most 2^8, the bound the
// row-max test held P to (a looser 2^12 measured larger O errors on sharp
// softmaxes for half a percent of speed).
constexpr float kChunkSumLimit = 256.f;

// One online-softmax step for the score row at tensor-memory address s_addr
// (BN fp32 columns, raw Q.K^T): fills pk with P in bf16 pairs and updates the
// running max m (log2 units) and sum l.  Returns the factor O must be scaled by
// (1 when unchanged).
//
// After the first K/V tile the row is read once, 32 columns at a time, and the
// exps are taken at once against the running max, before the whole row is
// seen.  The chunk's own sum of p then decides whether that reference still
// holds: while it stays at most 2^8 every p is bounded by 2^8 and nothing
// needs rescaling (the stale reference is exact because l and O always share
// it).  This test costs three adds per chunk where a row max would cost a
// reduction over all 32 scores.  If any row of the warp exceeds it (or has no
// reference yet), the warp falls back to two passes (max, then exps) over the
// scores, which are still in tensor memory, and rows whose max grew by more
// than 2^8 move their reference.
template <int NP>
__device__ __forceinline__ float softmax_row(uint32_t s_addr, int j, bool masked, int col_lim, float scale,
                                             float& m, float& l, uint32_t (&pk)[NP]) {
  constexpr int NCOL = 2 * NP;
  const uint64_t sc2 = f2pack(scale, scale);
  if (j > 0) {
    const uint64_t negm2 = f2pack(-m, -m);
    bool grow = __any_sync(0xffffffffu, m == -CUDART_INF_F);   // no reference yet: -inf - -inf is NaN
    float lsum = 0.f;
    // the load of chunk c+1 is in flight while chunk c is processed
    uint32_t xa[32], xb[32];
    tmem_ld32(s_addr, xa);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < NCOL / 32; ++c) {
      if (grow) break;
      uint32_t (&x)[32] = (c & 1) ? xb : xa;
      uint32_t (&y)[32] = (c & 1) ? xa : xb;
      if (c + 1 < NCOL / 32) tmem_ld32(s_addr + 32 * (c + 1), y);
      if (masked) chunk_mask(x, 32 * c, col_lim);
      uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
      chunk_exp_pack(x, sc2, negm2, acc0, acc1, &pk[16 * c]);
      float a0, a1, b0, b1;
      f2unpack(acc0, a0, a1);
      f2unpack(acc1, b0, b1);
      const float cs = (a0 + a1) + (b0 + b1);
      if (__any_sync(0xffffffffu, !(cs <= kChunkSumLimit))) { grow = true; tmem_wait_ld(); break; }
      lsum += cs;
      if (c + 1 < NCOL / 32) tmem_wait_ld();
    }
    if (!grow) {
      l += lsum;
      return 1.f;
    }
  }
  // two passes: the row max, then the exps against the (possibly new) reference
  float mx = -CUDART_INF_F;
#pragma unroll
  for (int c = 0; c < NCOL / 32; ++c) {
    uint32_t x[32];
    tmem_ld32(s_addr + 32 * c, x);
    tmem_wait_ld();
    mx = fmaxf(mx, chunk_mask_max(x, 32 * c, masked, col_lim));
  }
  const float m_tile = mx * scale;
  const bool need = (j == 0) || (m_tile > m + 8.f);
  const float m_use = need ? fmaxf(m, m_tile) : m;
  const float m_ref = (m_use == -CUDART_INF_F) ? 0.f : m_use;
  const float alpha = (j == 0) ? 0.f : ex2(m - m_ref);
  const uint64_t negm2 = f2pack(-m_ref, -m_ref);
  uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
  for (int c = 0; c < NCOL / 32; ++c) {
    uint32_t x[32];
    tmem_ld32(s_addr + 32 * c, x);
    tmem_wait_ld();
    if (masked) chunk_mask(x, 32 * c, col_lim);
    chunk_exp_pack(x, sc2, negm2, acc0, acc1, &pk[16 * c]);
  }
  float a0, a1, b0, b1;
  f2unpack(acc0, a0, a1);
  f2unpack(acc1, b0, b1);
  const float rs = (a0 + a1) + (b0 + b1);
  l = (j == 0) ? rs : l * alpha + rs;
  m = m_use;
  return (j == 0) ? 1.f : alpha;
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = decltype(&cuTensorMapEncodeTiled);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Token-major [rows, H, D] bf16 tensor; box = 64 columns x 1 head x 128 rows,
// 128-byte swizzle (the layout the MMA descriptors expect).
ra_status make_map(CUtensorMap* map, const void* base, int D, int H, int64_t rows, uint32_t box_rows = 128) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return ra::fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return ra::fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return RA_OK;
}

}  // namespace

namespace ra {
// Bound of every device-side wait, in SM clock cycles: ~0.5 s by default,
// overridable with the environment variable RA_WAIT_LIMIT_CYCLES.
static inline long long wait_limit() {
  static long long lim = [] {
    const char* e = getenv("RA_WAIT_LIMIT_CYCLES");
    long long v = e ? atoll(e) : 0;
    return v > 0 ? v : (1ll << 30);
  }();
  return lim;
}
}  // namespace ra
