// Context-parallel decode: split-KV partial attention over the sharded paged
// cache, and the LSE merge of partial results.
//
// Sources: vLLM-Ascend developer guide "Context Parallel (CP)" -- section
// "Block table" (which device holds which token), sections on DCP/PCP decode
// (each device attends over its local KV shard; partial outputs and LSEs are
// merged by a cp_lse_ag_out_rs-style update).  The merge weights follow the
// blockwise decomposition on the guijiagi.com "Ring Attention" tag page:
// a partial with LSE_p = ln sum_j e^{s_j} contributes e^{LSE_p - LSE} O_p.
//
// Decode kernel layout: one CTA per (split, device w, request r), one warp per
// K/V head.  The 2..8 query heads of a GQA group share each K/V load.  Scores
// and P.V are warp-level bf16 tensor-core products (mma.sync m16n8k16 with
// fp32 accumulation): per 16-token tile a warp issues D/16 MMAs for Q.K^T and
// D/16 for P.V, which keeps the instruction count per HBM byte far below
// what scalar FMAs (about 3.6 issued instructions per byte) would need, so
// the kernel is bound by HBM.  Softmax runs in fp32 in the log2 domain.
#include <math_constants.h>

#include <mutex>

#include "ra_common.cuh"

RA_DEFINE_ERROR_FETCH(fetch_error_decode)

namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_nc(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

struct DecodeParams {
  const __nv_bfloat16* q;   // [R, Hq, D]
  const __nv_bfloat16* kc;  // [W, NB, Hkv, bs, D]
  const __nv_bfloat16* vc;
  const int32_t* block_table;  // [R, max_vb]
  const int32_t* ctx;          // [R]
  float* o_parts;              // [P, R, Hq, D]
  float* lse_parts;            // [P, R, Hq]
  int R, Hq, Hkv, G, bs, interleave, W, max_vb, split_blocks, n_splits;
  int dev0;                    // the cache holds devices dev0, dev0+1, ... (blockIdx.y counts from dev0)
  long long num_blocks;
  float scale_log2;
};

// Thread (g = lane/4, t = lane%4) of the warp.  Token tile = 16 slots.
//  Q.K^T: A = K tile [16 slots x D] (rows g, g+8), B = Q^T [D x 8 heads];
//    the thread holds K/Q d-pieces of 8 elements at d = 8*(t + 4*i); MMA
//    k-step ks uses words 2*(ks&1), 2*(ks&1)+1 of piece ks>>1 (the same
//    bijection of d for A and B, so the contraction covers every d once).
//  P.V: O^T [D x 8] += V^T [D x 16 slots] . P^T [16 x 8]; rows of M-block mb
//    are d = 8*g + 64*(mb/4) + 2*(mb%4) + {0 (row g), 1 (row g+8)}; the
//    thread loads V pieces at d = 8*g and 8*g + 64 of slots 2t, 2t+1, 2t+8,
//    2t+9 and pairs tokens with byte permutes.
template <int D>
__global__ void __launch_bounds__(kWarps * 32, 1)
    cp_decode_kernel(const DecodeParams p) {
  constexpr int KP = D / 32;  // K/Q pieces (16 B) per thread per row
  constexpr int VP = D / 64;  // V pieces per thread per token
  constexpr int MB = D / 16;  // M-blocks of the P.V product
  constexpr int KS = D / 16;  // k-steps of the Q.K^T product
  __shared__ __align__(16) uint16_t p_smem[kWarps][8][16];  // P^T [head][slot] bf16 per warp

  const int sp = blockIdx.x, wl = blockIdx.y, r = blockIdx.z;
  const int w = p.dev0 + wl;  // the device's number among all W (token ownership)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int L = p.ctx[r];
  const int64_t Vsz = static_cast<int64_t>(p.bs) * p.W;
  const int nvb = static_cast<int>((L + Vsz - 1) / Vsz);
  const int vb0 = sp * p.split_blocks;
  const int vb1 = min(nvb, vb0 + p.split_blocks);
  const int part = wl * p.n_splits + sp;

  for (int kvh = warp; kvh < p.Hkv; kvh += kWarps) {
    // ---- Q fragments (bf16 pairs), heads >= G are zero
    uint4 qf[KP];
    const int hq = kvh * p.G + g;
#pragma unroll
    for (int i = 0; i < KP; ++i) {
      if (g < p.G)
        qf[i] = *reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(r) * p.Hq + hq) * D +
                                                8 * (t + 4 * i));
      else
        qf[i] = make_uint4(0, 0, 0, 0);
    }
    float acc[MB][4];
#pragma unroll
    for (int mb = 0; mb < MB; ++mb) acc[mb][0] = acc[mb][1] = acc[mb][2] = acc[mb][3] = 0.f;
    float m_run[2] = {-CUDART_INF_F, -CUDART_INF_F};  // heads 2t, 2t+1 (log2 units)
    float l_part[2] = {0.f, 0.f};

    for (int vb = vb0; vb < vb1; ++vb) {
      const int32_t blk = p.block_table[static_cast<int64_t>(r) * p.max_vb + vb];
      if (blk < 0 || blk >= p.num_blocks) {
        if (lane == 0) ra_record_error(RA_ERR_DEVICE_BOUNDS, 20);
        continue;
      }
      const int64_t head_base =
          ((static_cast<int64_t>(wl) * p.num_blocks + blk) * p.Hkv + kvh) * p.bs * D;
      const __nv_bfloat16* kb = p.kc + head_base;
      const __nv_bfloat16* vbp = p.vc + head_base;
      const bool block_full = static_cast<int64_t>(vb + 1) * Vsz <= L;
      for (int s0 = 0; s0 < p.bs; s0 += 16) {
        // ---- loads
        uint4 ka[KP], kb8[KP];
#pragma unroll
        for (int i = 0; i < KP; ++i) {
          ka[i] = ldg_nc(reinterpret_cast<const uint4*>(kb + (s0 + g) * D + 8 * (t + 4 * i)));
          kb8[i] = ldg_nc(reinterpret_cast<const uint4*>(kb + (s0 + g + 8) * D + 8 * (t + 4 * i)));
        }
        uint4 vv[4][VP];  // slots 2t, 2t+1, 2t+8, 2t+9
        const int vs[4] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9};
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int j = 0; j < VP; ++j)
            vv[u][j] = ldg_nc(reinterpret_cast<const uint4*>(vbp + (s0 + vs[u]) * D + 8 * g + 64 * j));

        // ---- validity of the slots this thread touches
        bool ok_s[2] = {true, true};   // score rows: slots s0+g, s0+g+8
        bool ok_v[4] = {true, true, true, true};
        if (!block_full) {
          const int Wd = p.W, I = p.interleave;
          auto tok = [&](int s) -> int64_t {
            return static_cast<int64_t>(vb) * Vsz + (static_cast<int64_t>(s / I) * Wd + w) * I + s % I;
          };
          ok_s[0] = tok(s0 + g) < L;
          ok_s[1] = tok(s0 + g + 8) < L;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            ok_v[u] = tok(s0 + vs[u]) < L;
            if (!ok_v[u]) {
#pragma unroll
              for (int j = 0; j < VP; ++j) vv[u][j] = make_uint4(0, 0, 0, 0);
            }
          }
        }

        // ---- S^T [16 slots x 8 heads] = K . Q^T
        float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int i = ks >> 1, wsel = 2 * (ks & 1);
          mma_16816(s, word(ka[i], wsel), word(kb8[i], wsel), word(ka[i], wsel + 1),
                    word(kb8[i], wsel + 1), word(qf[i], wsel), word(qf[i], wsel + 1));
        }
        // s[0]: slot g head 2t; s[1]: slot g head 2t+1; s[2], s[3]: slot g+8
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool ok = ok_s[e >> 1] && (2 * t + (e & 1) < p.G);
          s[e] = ok ? s[e] * p.scale_log2 : -CUDART_INF_F;
        }
        // ---- tile max per head over the 16 slots (lanes with equal t)
        float mt[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 4));
          mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 8));
          mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 16));
        }
        // Lazy rescale: keep the running max unless the tile max exceeds it by
        // more than 8 (log2 units); exactness holds because l and acc always
        // share the same reference.
        float alpha[2];
        bool resc = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          alpha[h] = 1.f;
          if (mt[h] > m_run[h] + 8.f) {
            alpha[h] = (m_run[h] == -CUDART_INF_F) ? 0.f : exp2f(m_run[h] - mt[h]);
            m_run[h] = mt[h];
            resc = true;
          }
        }
        if (resc) {
#pragma unroll
          for (int mb = 0; mb < MB; ++mb) {
            acc[mb][0] *= alpha[0]; acc[mb][1] *= alpha[1];
            acc[mb][2] *= alpha[0]; acc[mb][3] *= alpha[1];
          }
          l_part[0] *= alpha[0];
          l_part[1] *= alpha[1];
        }
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float m = m_run[e & 1];
          pv[e] = (m == -CUDART_INF_F) ? 0.f : exp2f(s[e] - m);
        }
        l_part[0] += pv[0] + pv[2];
        l_part[1] += pv[1] + pv[3];
        // ---- P^T to shared memory (bf16), then the B fragments
        __nv_bfloat16 pb[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pb[e] = __float2bfloat16_rn(pv[e]);
        p_smem[warp][2 * t][g] = *reinterpret_cast<uint16_t*>(&pb[0]);
        p_smem[warp][2 * t + 1][g] = *reinterpret_cast<uint16_t*>(&pb[1]);
        p_smem[warp][2 * t][g + 8] = *reinterpret_cast<uint16_t*>(&pb[2]);
        p_smem[warp][2 * t + 1][g + 8] = *reinterpret_cast<uint16_t*>(&pb[3]);
        __syncwarp();
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&p_smem[warp][g][2 * t]);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&p_smem[warp][g][2 * t + 8]);
        __syncwarp();
        // ---- O^T += V^T . P^T
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
          const int j = mb >> 2, wi = mb & 3;
          const uint32_t w0 = word(vv[0][j], wi), w1 = word(vv[1][j], wi);
          const uint32_t w8 = word(vv[2][j], wi), w9 = word(vv[3][j], wi);
          mma_16816(acc[mb], __byte_perm(w0, w1, 0x5410), __byte_perm(w0, w1, 0x7632),
                    __byte_perm(w8, w9, 0x5410), __byte_perm(w8, w9, 0x7632), b0, b1);
        }
      }
    }
    // ---- finish: l over the 16 slot rows (lanes with equal t)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      l_part[h] += __shfl_xor_sync(0xffffffffu, l_part[h], 4);
      l_part[h] += __shfl_xor_sync(0xffffffffu, l_part[h], 8);
      l_part[h] += __shfl_xor_sync(0xffffffffu, l_part[h], 16);
    }
    const int64_t prow = (static_cast<int64_t>(part) * p.R + r) * p.Hq + kvh * p.G;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int head = 2 * t + h;
      if (head >= p.G) continue;
      const bool live = l_part[h] > 0.f;
      if (g == 0)
        p.lse_parts[prow + head] = live ? (m_run[h] + log2f(l_part[h])) * kLn2 : -CUDART_INF_F;
      if (!live) continue;
      const float inv = 1.f / l_part[h];
      float* orow = p.o_parts + (prow + head) * D;
#pragma unroll
      for (int mb = 0; mb < MB; ++mb) {
        const int d0 = 8 * g + 64 * (mb >> 2) + 2 * (mb & 3);
        orow[d0] = acc[mb][h] * inv;
        orow[d0 + 1] = acc[mb][2 + h] * inv;
      }
    }
  }
}

// One warp per (token, head) row: LSE = M + ln sum_p e^{LSE_p - M},
// O = sum_p e^{LSE_p - LSE} O_p (partials with LSE_p = -inf skipped).
template <bool OUT_BF16>
__device__ __forceinline__ void store_merged(void* o_out, int64_t at, const float4& a) {
  if (OUT_BF16) {
    uint2 pk = make_uint2(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w));
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + at) = pk;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(o_out) + at) = a;
  }
}

// MODE 1: at most 8 partials, d = 128; MODE 0: any P and d.  Separate
// instances keep the fast path's register count (and so its occupancy).
template <bool OUT_BF16, int MODE>
__global__ void lse_merge_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts,
                                 int P, int64_t rows, int d, void* __restrict__ o_out,
                                 float* __restrict__ lse_out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  if (MODE == 1) {
    // Few partials (segmented prefill, stand-alone merges): lane p holds partial p's
    // LSE and weight, and the warp's loads of all P partial rows are issued together,
    // independent of the LSE arithmetic, so a row costs one memory latency.
    for (int64_t row = warp; row < rows; row += nwarps) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (u < P) v[u] = *reinterpret_cast<const float4*>(o_parts + (static_cast<int64_t>(u) * rows + row) * 128 + 4 * lane);
      const float x = lane < P ? lse_parts[static_cast<int64_t>(lane) * rows + row] : -CUDART_INF_F;
      float M = x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float wu = (x == -CUDART_INF_F) ? 0.f : expf(x - M);
      float tot = wu;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
      const float w = tot > 0.f ? wu / tot : 0.f;   // e^{LSE_p - LSE}
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (u >= P) break;
        const float wp = __shfl_sync(0xffffffffu, w, u);
        if (wp != 0.f) {   // an empty partial's O is never read
          a.x += wp * v[u].x; a.y += wp * v[u].y; a.z += wp * v[u].z; a.w += wp * v[u].w;
        }
      }
      store_merged<OUT_BF16>(o_out, row * 128 + 4 * lane, a);
      if (lse_out && lane == 0) lse_out[row] = (M == -CUDART_INF_F) ? -CUDART_INF_F : M + logf(tot);
    }
    return;
  }
  for (int64_t row = warp; row < rows; row += nwarps) {
    float M = -CUDART_INF_F;
    for (int pp = lane; pp < P; pp += 32) M = fmaxf(M, lse_parts[static_cast<int64_t>(pp) * rows + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float tot = 0.f;
    if (M != -CUDART_INF_F)
      for (int pp = lane; pp < P; pp += 32) {
        const float x = lse_parts[static_cast<int64_t>(pp) * rows + row];
        tot += (x == -CUDART_INF_F) ? 0.f : expf(x - M);
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    const float lse = (M == -CUDART_INF_F) ? -CUDART_INF_F : M + logf(tot);
    for (int e0 = 4 * lane; e0 < d; e0 += 128) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (M != -CUDART_INF_F) {
        for (int pp = 0; pp < P; ++pp) {
          const float x = lse_parts[static_cast<int64_t>(pp) * rows + row];
          if (x == -CUDART_INF_F) continue;
          const float wgt = expf(x - lse);
          const float4 v = *reinterpret_cast<const float4*>(o_parts + (static_cast<int64_t>(pp) * rows + row) * d + e0);
          a.x += wgt * v.x; a.y += wgt * v.y; a.z += wgt * v.z; a.w += wgt * v.w;
        }
      }
      store_merged<OUT_BF16>(o_out, row * d + e0, a);
    }
    if (lse_out && lane == 0) lse_out[row] = lse;
  }
}

ra_status launch_merge(const float* o_parts, const float* lse_parts, int P, int64_t rows, int d,
                       void* o_out, ra_dtype out_dt, float* lse_out, cudaStream_t stream) {
  const int64_t blocks = std::min<int64_t>(ra::ceil_div(rows * 32, 256), 152 * 16);
  const int mode = (d == 128 && P <= 8) ? 1 : 0;
  const bool bf = out_dt == RA_BF16;
#define RA_MERGE(B, M) lse_merge_kernel<B, M><<<blocks, 256, 0, stream>>>(o_parts, lse_parts, P, rows, d, o_out, lse_out)
  if (mode == 1) { if (bf) RA_MERGE(true, 1); else RA_MERGE(false, 1); }
  else { if (bf) RA_MERGE(true, 0); else RA_MERGE(false, 0); }
#undef RA_MERGE
  RA_LAUNCH_CHECK("lse_merge_kernel");
  return RA_OK;
}

int32_t n_splits_of(int32_t max_vblocks, int32_t split_blocks) {
  return static_cast<int32_t>(ra::ceil_div(max_vblocks, split_blocks));
}

}  // namespace

extern "C" ra_status ra_lse_merge(const float* o_parts, const float* lse_parts, int32_t P, int64_t T,
                                  int32_t H, int32_t d, void* o_out, ra_dtype out_dt, float* lse_out,
                                  ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(P >= 1 && T >= 0 && H >= 1 && d >= 1, "P, H, d must be >= 1 and T >= 0");
  RA_REQUIRE(out_dt == RA_F32 || out_dt == RA_BF16, "unknown out dtype");
  if (d % 4 != 0) return ra::fail(RA_ERR_UNSUPPORTED, "d must be a multiple of 4 (got %d)", d);
  if (T == 0) return RA_OK;
  RA_REQUIRE(o_parts && lse_parts && o_out, "NULL pointer");
  RA_REQUIRE(ra::aligned16(o_parts) && ra::aligned16(o_out), "o_parts/o_out must be 16-byte aligned");
  return launch_merge(o_parts, lse_parts, P, T * H, d, o_out, out_dt, lse_out, stream);
}

extern "C" ra_status ra_cp_decode_workspace_size(int32_t R, int32_t Hq, int32_t d, int32_t max_vblocks,
                                                 int32_t pcp, int32_t dcp, int32_t split_blocks,
                                                 size_t* bytes) {
  ra::clear_error();
  RA_REQUIRE(bytes != nullptr, "bytes is NULL");
  RA_REQUIRE(R >= 1 && Hq >= 1 && d >= 1 && max_vblocks >= 1 && pcp >= 1 && dcp >= 1 && split_blocks >= 1,
             "sizes must be >= 1");
  const int64_t P = static_cast<int64_t>(pcp) * dcp * n_splits_of(max_vblocks, split_blocks);
  const int64_t o_bytes = P * R * Hq * d * 4;
  const int64_t l_bytes = P * R * Hq * 4;
  *bytes = static_cast<size_t>(ra::ceil_div(o_bytes, 256) * 256 + l_bytes);
  return RA_OK;
}

namespace {
// Checks shared by the decode entry points; fills the kernel parameters.
ra_status decode_params(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                        const int32_t* ctx_lens, int32_t R, int32_t Hq, int32_t Hkv, int32_t d, int32_t block_size,
                        int32_t interleave, int32_t pcp, int32_t dcp, int32_t dev0, int32_t n_dev,
                        int32_t max_vblocks, int64_t num_blocks, float scale, int32_t split_blocks,
                        DecodeParams& prm) {
  RA_REQUIRE(R >= 1 && Hq >= 1 && Hkv >= 1 && block_size >= 1 && interleave >= 1 && pcp >= 1 &&
                 dcp >= 1 && max_vblocks >= 1 && num_blocks >= 1 && split_blocks >= 1,
             "sizes must be >= 1");
  RA_REQUIRE(block_size % interleave == 0,
             "block_size %% cp_kv_cache_interleave_size must be 0 (block_size=%d, interleave=%d)",
             block_size, interleave);
  RA_REQUIRE(Hq % Hkv == 0, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  const int W = pcp * dcp;
  RA_REQUIRE(dev0 >= 0 && n_dev >= 1 && dev0 + n_dev <= W, "devices [%d, %d) must lie in [0, pcp*dcp = %d)", dev0,
             dev0 + n_dev, W);
  if (d != 64 && d != 128) return ra::fail(RA_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", d);
  if (Hq / Hkv > 8) return ra::fail(RA_ERR_UNSUPPORTED, "GQA group %d > 8 not supported", Hq / Hkv);
  if (block_size % 16 != 0) return ra::fail(RA_ERR_UNSUPPORTED, "block_size must be a multiple of 16");
  RA_REQUIRE(q && k_cache && v_cache && block_table && ctx_lens, "NULL pointer");
  RA_REQUIRE(ra::aligned16(q) && ra::aligned16(k_cache) && ra::aligned16(v_cache),
             "q and the caches must be 16-byte aligned");
  const int n_splits = n_splits_of(max_vblocks, split_blocks);
  RA_REQUIRE(n_splits <= 65535 && n_dev <= 65535 && R <= 65535, "grid too large");
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.kc = static_cast<const __nv_bfloat16*>(k_cache);
  prm.vc = static_cast<const __nv_bfloat16*>(v_cache);
  prm.block_table = block_table;
  prm.ctx = ctx_lens;
  prm.R = R; prm.Hq = Hq; prm.Hkv = Hkv; prm.G = Hq / Hkv; prm.bs = block_size;
  prm.interleave = interleave; prm.W = W; prm.max_vb = max_vblocks;
  prm.split_blocks = split_blocks; prm.n_splits = n_splits; prm.num_blocks = num_blocks;
  prm.dev0 = dev0;
  prm.scale_log2 = (scale > 0.f ? scale : 1.f / sqrtf(static_cast<float>(d))) * kLog2e;
  return RA_OK;
}

ra_status launch_decode(const DecodeParams& prm, int n_dev, int d, cudaStream_t stream) {
  dim3 grid(prm.n_splits, n_dev, prm.R);
  if (d == 128)
    cp_decode_kernel<128><<<grid, kWarps * 32, 0, stream>>>(prm);
  else
    cp_decode_kernel<64><<<grid, kWarps * 32, 0, stream>>>(prm);
  RA_LAUNCH_CHECK("cp_decode_kernel");
  return RA_OK;
}
}  // namespace

extern "C" ra_status ra_cp_decode_partials(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* block_table, const int32_t* ctx_lens, int32_t R,
                                           int32_t Hq, int32_t Hkv, int32_t d, int32_t block_size,
                                           int32_t interleave, int32_t pcp, int32_t dcp, int32_t dev0,
                                           int32_t n_dev, int32_t max_vblocks, int64_t num_blocks, float scale,
                                           int32_t split_blocks, float* o_parts, float* lse_parts,
                                           int32_t* n_parts_out, ra_stream stream) {
  ra::clear_error();
  DecodeParams prm;
  ra_status st = decode_params(q, k_cache, v_cache, block_table, ctx_lens, R, Hq, Hkv, d, block_size, interleave,
                               pcp, dcp, dev0, n_dev, max_vblocks, num_blocks, scale, split_blocks, prm);
  if (st != RA_OK) return st;
  const int64_t P = static_cast<int64_t>(n_dev) * prm.n_splits;
  RA_REQUIRE(P < (int64_t(1) << 31), "too many partials");
  if (n_parts_out) *n_parts_out = static_cast<int32_t>(P);
  if (o_parts == nullptr && lse_parts == nullptr) return RA_OK;  // size query
  RA_REQUIRE(o_parts && lse_parts, "o_parts and lse_parts are given together");
  RA_REQUIRE(ra::aligned16(o_parts) && reinterpret_cast<uintptr_t>(lse_parts) % 4 == 0,
             "o_parts must be 16-byte aligned, lse_parts 4-byte aligned");
  prm.o_parts = o_parts;
  prm.lse_parts = lse_parts;
  return launch_decode(prm, n_dev, d, stream);
}

extern "C" ra_status ra_cp_decode(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, const int32_t* ctx_lens, int32_t R,
                                  int32_t Hq, int32_t Hkv, int32_t d, int32_t block_size,
                                  int32_t interleave, int32_t pcp, int32_t dcp, int32_t max_vblocks,
                                  int64_t num_blocks, float scale, int32_t split_blocks, void* o,
                                  ra_dtype out_dt, float* lse, void* workspace, size_t ws_bytes,
                                  ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(out_dt == RA_F32 || out_dt == RA_BF16, "unknown out dtype");
  DecodeParams prm;
  ra_status st = decode_params(q, k_cache, v_cache, block_table, ctx_lens, R, Hq, Hkv, d, block_size, interleave,
                               pcp, dcp, 0, pcp * dcp, max_vblocks, num_blocks, scale, split_blocks, prm);
  if (st != RA_OK) return st;
  RA_REQUIRE(o && workspace, "NULL pointer");
  RA_REQUIRE(ra::aligned16(o) && ra::aligned16(workspace), "o and workspace must be 16-byte aligned");
  size_t need = 0;
  if ((st = ra_cp_decode_workspace_size(R, Hq, d, max_vblocks, pcp, dcp, split_blocks, &need)) != RA_OK) return st;
  RA_REQUIRE(ws_bytes >= need, "workspace too small (%zu < %zu bytes)", ws_bytes, need);
  const int64_t P = static_cast<int64_t>(prm.W) * prm.n_splits;
  prm.o_parts = static_cast<float*>(workspace);
  prm.lse_parts = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           ra::ceil_div(P * R * Hq * d * 4, 256) * 256);
  if ((st = launch_decode(prm, prm.W, d, stream)) != RA_OK) return st;
  return launch_merge(prm.o_parts, prm.lse_parts, static_cast<int>(P), static_cast<int64_t>(R) * Hq, d, o,
                      out_dt, lse, stream);
}

// ===========================================================================
// Step 2 of cp_lse_ag_out_rs (vLLM-Ascend "Context Parallel (CP)", DCP
// decode): with every device's LSE gathered, device w scales its own partial
// O_w by e^{LSE_w - LSE}, LSE = ln sum_v e^{LSE_v}, and lays it out by the
// device that keeps each head after the reduce-scatter.  One warp per
// (request, head) row.
// ===========================================================================
namespace {
__global__ void lse_rescale_kernel(const float* __restrict__ o_local, const float* __restrict__ lse_all, int W,
                                   int w, int64_t R, int Hq, int d, float* __restrict__ o_scaled,
                                   float* __restrict__ lse_total) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = R * Hq;
  const int hs = Hq / W;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < rows;
       row += nwarps) {
    const int64_t r = row / Hq;
    const int h = static_cast<int>(row % Hq);
    float M = -CUDART_INF_F;
    for (int v = lane; v < W; v += 32) M = fmaxf(M, lse_all[static_cast<int64_t>(v) * rows + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float tot = 0.f;
    if (M != -CUDART_INF_F)
      for (int v = lane; v < W; v += 32) {
        const float x = lse_all[static_cast<int64_t>(v) * rows + row];
        tot += x == -CUDART_INF_F ? 0.f : expf(x - M);
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    const float lse = M == -CUDART_INF_F ? -CUDART_INF_F : M + logf(tot);
    const float mine = lse_all[static_cast<int64_t>(w) * rows + row];
    const float wgt = (mine == -CUDART_INF_F || lse == -CUDART_INF_F) ? 0.f : expf(mine - lse);
    const int v = h / hs, j = h % hs;
    float* dst = o_scaled + ((static_cast<int64_t>(v) * R + r) * hs + j) * d;
    const float* src = o_local + row * d;
    for (int e = 4 * lane; e < d; e += 128) {
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (wgt != 0.f) {   // a partial with no key is not read
        a = *reinterpret_cast<const float4*>(src + e);
        a.x *= wgt; a.y *= wgt; a.z *= wgt; a.w *= wgt;
      }
      *reinterpret_cast<float4*>(dst + e) = a;
    }
    if (lse_total && v == w && lane == 0) lse_total[r * hs + j] = lse;
  }
}
}  // namespace

// The all-to-all form of the same merge: device w lays its output and LSE out by the device that
// keeps each head, so that one all-to-all hands every device the W partials of its own heads
// (merged there by ra_lse_merge).  One warp per (request, head) row.
namespace {
__global__ void head_split_kernel(const float* __restrict__ o_local, const float* __restrict__ lse_local, int W,
                                  int64_t R, int Hq, int d, float* __restrict__ o_split,
                                  float* __restrict__ lse_split) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = R * Hq;
  const int hs = Hq / W;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < rows;
       row += nwarps) {
    const int64_t r = row / Hq;
    const int h = static_cast<int>(row % Hq);
    const int v = h / hs, j = h % hs;
    const int64_t at = (static_cast<int64_t>(v) * R + r) * hs + j;
    const float lse = lse_local[row];
    const bool live = lse != -CUDART_INF_F;
    for (int e = 4 * lane; e < d; e += 128) {
      const float4 a = live ? *reinterpret_cast<const float4*>(o_local + row * d + e) : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(o_split + at * d + e) = a;
    }
    if (lane == 0) lse_split[at] = lse;
  }
}
}  // namespace

extern "C" ra_status ra_cp_head_split(const float* o_local, const float* lse_local, int32_t W, int64_t R, int32_t Hq,
                                      int32_t d, float* o_split, float* lse_split, ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(W >= 1 && R >= 0 && Hq >= 1 && d >= 1, "W, Hq, d >= 1 and R >= 0");
  RA_REQUIRE(Hq % W == 0, "Hq (%d) must be a multiple of W (%d)", Hq, W);
  if (d % 4 != 0) return ra::fail(RA_ERR_UNSUPPORTED, "d must be a multiple of 4 (got %d)", d);
  if (R == 0) return RA_OK;
  RA_REQUIRE(o_local && lse_local && o_split && lse_split, "NULL pointer");
  RA_REQUIRE(ra::aligned16(o_local) && ra::aligned16(o_split), "o_local and o_split must be 16-byte aligned");
  const int64_t blocks = std::min<int64_t>(ra::ceil_div(R * Hq * 32, 256), 152 * 16);
  head_split_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_local, lse_local, W, R, Hq, d, o_split,
                                                                       lse_split);
  RA_LAUNCH_CHECK("head_split_kernel");
  return RA_OK;
}

extern "C" ra_status ra_cp_lse_rescale(const float* o_local, const float* lse_all, int32_t W, int32_t w, int64_t R,
                                       int32_t Hq, int32_t d, float* o_scaled, float* lse_total,
                                       ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(W >= 1 && w >= 0 && w < W, "w (%d) must be in [0, W = %d)", w, W);
  RA_REQUIRE(R >= 0 && Hq >= 1 && d >= 1, "R >= 0, Hq and d >= 1");
  RA_REQUIRE(Hq % W == 0, "Hq (%d) must be a multiple of W (%d)", Hq, W);
  if (d % 4 != 0) return ra::fail(RA_ERR_UNSUPPORTED, "d must be a multiple of 4 (got %d)", d);
  if (R == 0) return RA_OK;
  RA_REQUIRE(o_local && lse_all && o_scaled, "NULL pointer");
  RA_REQUIRE(ra::aligned16(o_local) && ra::aligned16(o_scaled), "o_local and o_scaled must be 16-byte aligned");
  const int64_t blocks = std::min<int64_t>(ra::ceil_div(R * Hq * 32, 256), 152 * 16);
  lse_rescale_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_local, lse_all, W, w, R, Hq, d, o_scaled,
                                                                         lse_total);
  RA_LAUNCH_CHECK("lse_rescale_kernel");
  return RA_OK;
}

// ===========================================================================
// Allocation-free decode.
//
// Some callers cannot call cudaMalloc on the path where decode runs: an
// inference runtime that reserves all device memory at start-up and forbids
// allocation afterwards, code running under an allocator that cannot hand out
// raw scratch, or a host process that must keep its device footprint fixed.
// ra_cp_decode_noalloc gives them the same decode with the fp32 partials kept
// in a fixed scratch array that lives in this library's device memory instead
// of a caller-provided workspace.  Every GPU that loads the library holds the
// array (kNoAllocScratchBytes) until the process exits.
//
// The array's name is a host-side stand-in in host code, not a device
// address; its device address is looked up with cudaGetSymbolAddress (with the
// device current) the first time the entry point runs on a device, and reused
// while that device's CUDA context stays the same.  A context that was torn
// down and created again (cudaDeviceReset, for one) reloads this module, which
// may place the array elsewhere, so the address is looked up again then.
//
// Under lazy module loading (CUDA's default) this module, and with it the
// array, is loaded by the first call on each device: that call commits the
// array's device memory.  Callers that must not allocate after start-up make
// one warm-up call per device at start-up (the same call that must precede any
// stream capture), or load modules eagerly (CUDA_MODULE_LOADING=EAGER).
//
// All calls share the array and it keeps the last call's contents.  Nothing in
// it has to start at zero: each call writes the LSE of every partial before the
// merge reads it, and the merge reads a partial's O only when that LSE is
// finite, i.e. when the same call wrote that O.  Calls whose work overlaps on
// the GPU (for example on two streams at once) race on the array.
// ===========================================================================
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx_id[kMaxDevices] = {};  // id of the context the address belongs to

// cuCtxGetCurrent and cuCtxGetId from the driver (the library links the
// runtime only).  A context id is unique for the life of the process, so a
// context created again after a reset has a new one.
using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);
template <class Fn>
Fn driver_fn(const char* name) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(ptr);
  return nullptr;
}

// Id of the calling thread's current context, 0 if none is current yet.
unsigned long long current_ctx_id() {
  static const CtxGetCurrentFn get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (!get_ctx || !get_id || get_ctx(&ctx) != 0 || ctx == nullptr || get_id(ctx, &id) != 0) return 0;
  return id;
}

// Device address of g_decode_scratch in the current device's context: looked
// up (with that device current) the first time on a device, and again
// whenever the device's context has changed since.
ra_status scratch_address(void** out) {
  int dev = 0;
  RA_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return ra::fail(RA_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  const unsigned long long id = current_ctx_id();
  if (g_scratch_ptr[dev] == nullptr || id == 0 || id != g_scratch_ctx_id[dev]) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) return ra::cuda_status(e, "cudaGetSymbolAddress(decode scratch)");
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx_id[dev] = current_ctx_id();  // the lookup made the primary context current
  }
  *out = g_scratch_ptr[dev];
  return RA_OK;
}
}  // namespace

extern "C" ra_status ra_cp_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_table, const int32_t* ctx_lens, int32_t R,
                                          int32_t Hq, int32_t Hkv, int32_t d, int32_t block_size,
                                          int32_t interleave, int32_t pcp, int32_t dcp, int32_t max_vblocks,
                                          int64_t num_blocks, float scale, int32_t split_blocks, void* o,
                                          ra_dtype out_dt, float* lse, ra_stream stream) {
  ra::clear_error();
  size_t need = 0;
  ra_status st = ra_cp_decode_workspace_size(R, Hq, d, max_vblocks, pcp, dcp, split_blocks, &need);
  if (st != RA_OK) return st;
  if (need > kNoAllocScratchBytes)
    return ra::fail(RA_ERR_INVALID_ARG,
                    "this decode needs %zu bytes of scratch, but the allocation-free entry point holds at most "
                    "%zu bytes; raise split_blocks or call ra_cp_decode with a workspace",
                    need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != RA_OK) return st;
  return ra_cp_decode(q, k_cache, v_cache, block_table, ctx_lens, R, Hq, Hkv, d, block_size, interleave, pcp,
                      dcp, max_vblocks, num_blocks, scale, split_blocks, o, out_dt, lse, scratch,
                      kNoAllocScratchBytes, stream);
}
