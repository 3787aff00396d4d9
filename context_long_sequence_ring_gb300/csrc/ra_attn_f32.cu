// Ring-order attention forward in exact fp32 on the CUDA cores (no tensor
// cores: tf32 would not meet a 1e-4 tolerance).
//
// Sources: "Parallelism-CP" diagram (Q/K/V split along the sequence, K/V
// rotating on a ring until every Q block has met every K/V block);
// guijiagi.com "Ring Attention" tag page (ring step t: rank i works on the K/V
// block of rank (i - t) mod N; the blockwise decomposition with a running max
// and running sum); vLLM-Ascend "Context Parallel (CP)" head-tail partition
// (rank r owns chunks r and 2N-1-r of the 2N equal chunks).
//
// Grid: (row tiles of 8 queries per chunk, 2N chunks, B*Hq).  A CTA holds 8
// query rows of one chunk (one warp per row) and walks the K/V of the ring in
// rank order s = r, r-1, ..., each rank's two chunks in turn, 32 keys per
// shared-memory tile; every lane scores one key, the warp updates
// (m, l, acc) and each lane accumulates D/32 output columns.
#include <math_constants.h>

#include "ra_common.cuh"

RA_DEFINE_ERROR_FETCH(fetch_error_attn_f32)

namespace {

constexpr int kRows = 8;   // query rows per CTA (one warp each)
constexpr int kKeys = 32;  // keys per shared-memory tile

struct F32Params {
  const float* q; const float* k; const float* v; float* o; float* lse;
  int B, Hq, Hkv, S, N, c, causal, layout;
  float scale_log2;
};

// Token row of (sequence b, global chunk ch, offset off) in the tensor.
__device__ __forceinline__ int64_t token_row(const F32Params& p, int b, int ch, int off) {
  if (p.layout == RA_LAYOUT_NATURAL) return static_cast<int64_t>(b) * p.S + static_cast<int64_t>(ch) * p.c + off;
  const int rank = ch < p.N ? ch : 2 * p.N - 1 - ch;
  const int half = ch < p.N ? 0 : 1;
  return ((static_cast<int64_t>(rank) * p.B + b) * 2 + half) * p.c + off;
}

template <int D>
__global__ void __launch_bounds__(kRows * 32) ring_attn_f32_kernel(const F32Params p) {
  constexpr int E = D / 32;  // output columns per lane
  __shared__ float ks[kKeys][D + 1];
  __shared__ float vs[kKeys][D];
  __shared__ float qs[kRows][D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qc = blockIdx.y;                  // global chunk of these queries
  const int bh = blockIdx.z;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int g = hq / (p.Hq / p.Hkv);
  const int r = qc < p.N ? qc : 2 * p.N - 1 - qc;  // owning rank
  const int row0 = blockIdx.x * kRows;
  const int row = row0 + warp;                 // offset inside the chunk
  const bool row_ok = row < p.c;
  const int qpos = qc * p.c + row;             // original position

  for (int i = threadIdx.x; i < kRows * D; i += blockDim.x) {
    const int rr = i / D, e = i % D;
    float x = 0.f;
    if (row0 + rr < p.c) x = p.q[(token_row(p, b, qc, row0 + rr) * p.Hq + hq) * D + e];
    qs[rr][e] = x;
  }

  float m = -CUDART_INF_F, l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  const int last_row = min(row0 + kRows, p.c) - 1;

  for (int t = 0; t < p.N; ++t) {
    const int s = (r - t + p.N) % p.N;  // rank whose K/V block is held at step t
    for (int h2 = 0; h2 < 2; ++h2) {
      const int kc = h2 == 0 ? s : 2 * p.N - 1 - s;
      if (p.causal && kc > qc) continue;
      for (int k0 = 0; k0 < p.c; k0 += kKeys) {
        if (p.causal && kc == qc && k0 > last_row) break;  // no key visible to any row
        __syncthreads();
        for (int i = threadIdx.x; i < kKeys * D; i += blockDim.x) {
          const int j = i / D, e = i % D;
          float kx = 0.f, vx = 0.f;
          if (k0 + j < p.c) {
            const int64_t tr = token_row(p, b, kc, k0 + j);
            kx = p.k[(tr * p.Hkv + g) * D + e];
            vx = p.v[(tr * p.Hkv + g) * D + e];
          }
          ks[j][e] = kx;
          vs[j][e] = vx;
        }
        __syncthreads();
        const int kpos = kc * p.c + k0 + lane;
        bool vis = row_ok && (k0 + lane < p.c) && (!p.causal || kpos <= qpos);
        float sc = 0.f;
#pragma unroll 8
        for (int e = 0; e < D; ++e) sc = fmaf(qs[warp][e], ks[lane][e], sc);
        sc = vis ? sc * p.scale_log2 : -CUDART_INF_F;
        float mx = sc;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m, mx);
        if (m_new == -CUDART_INF_F) continue;  // nothing visible yet (warp-uniform)
        const float alpha = exp2f(m - m_new);  // 0 when m = -inf
        const float pj = exp2f(sc - m_new);
        float ps = pj;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l = l * alpha + ps;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] *= alpha;
        for (int j = 0; j < kKeys; ++j) {
          const float pjj = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] = fmaf(pjj, vs[j][lane + 32 * e], acc[e]);
        }
        m = m_new;
      }
    }
  }
  if (!row_ok) return;
  const int64_t tr = token_row(p, b, qc, row);
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) p.o[(tr * p.Hq + hq) * D + lane + 32 * e] = acc[e] * inv;
  if (lane == 0)
    p.lse[tr * p.Hq + hq] = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
}

}  // namespace

namespace ra {
ra_status ring_attn_fwd_f32(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                            int Hkv, int S, int d, int causal, int N, float scale, int layout,
                            cudaStream_t stream) {
  F32Params p;
  p.q = static_cast<const float*>(q); p.k = static_cast<const float*>(k); p.v = static_cast<const float*>(v);
  p.o = static_cast<float*>(o); p.lse = lse;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.S = S; p.N = N; p.c = S / (2 * N); p.causal = causal; p.layout = layout;
  p.scale_log2 = scale * 1.4426950408889634f;
  const int64_t by = 2 * N, bz = static_cast<int64_t>(B) * Hq;
  if (by > 65535 || bz > 65535) return fail(RA_ERR_UNSUPPORTED, "grid too large for the fp32 kernel");
  dim3 grid(static_cast<unsigned>(ceil_div(p.c, kRows)), static_cast<unsigned>(by), static_cast<unsigned>(bz));
  if (d == 128)
    ring_attn_f32_kernel<128><<<grid, kRows * 32, 0, stream>>>(p);
  else
    ring_attn_f32_kernel<64><<<grid, kRows * 32, 0, stream>>>(p);
  RA_LAUNCH_CHECK("ring_attn_f32_kernel");
  return RA_OK;
}
}  // namespace ra
