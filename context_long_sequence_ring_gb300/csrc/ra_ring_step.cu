// One step of a ring across devices: a rank's queries against the K/V block it
// holds at that step, folded into the rank's running (O, LSE) result, on the
// tcgen05 two-slot pipeline.
//
// Sources: "Parallelism-CP" diagram (each card computes its own Q against the
// K/V blocks that rotate around the ring; every Q block meets every block);
// guijiagi.com "Ring Attention" tag page (at step t rank i holds the block of
// rank (i - t) mod N; blockwise decomposition, a partial over a key subset is
// carried by its log-sum-exp); vLLM-Ascend "Context Parallel (CP)" head-tail
// partition (rank r holds chunks r and 2N-1-r; the causal mask compares
// original positions).
//
// A rank's local buffers hold, per sequence, chunk `rank` then chunk
// 2N-1-rank (queries) and chunk `src` then chunk 2N-1-src (the held K/V), each
// c rows.  Work item = a mirrored pair of query tiles of the rank -- tile j of
// its first chunk and tile nt-1-j of its second -- for two query heads of one
// GQA group (even groups) or for one head with two adjacent tiles per slot
// pair (odd groups), as in the single-device ring kernel; so the causal work
// of every CTA is the same within a step.  A query tile that sees no key of
// the held block (its chunk precedes both held chunks) is not run; its rows
// keep their running result.  The epilogue merges the step's partial into the
// running result with the LSE weights: O = w_in O_in + w_p O_p,
// LSE = ln(e^{LSE_in} + e^{LSE_p}), w = e^{LSE_x - LSE}.
#include "ra_attn_pair.cuh"
#include "ra_ring_sched.cuh"

RA_DEFINE_ERROR_FETCH(fetch_error_ring_step)

namespace {
using namespace ra::sm100;

struct StepParams {
  int B, Hq, Hkv, group, N, r, s, c, nt, ntp, causal;
  float scale_log2;
  const float* o_in;    // [B*2c, Hq, D] fp32 running output, or null at a rank's first step
  const float* lse_in;  // [B*2c, Hq]
  void* o_out;          // [B*2c, Hq, D], fp32 or bf16 (may be o_in when fp32)
  int out_bf16;
  float* lse_out;       // [B*2c, Hq] (may be lse_in)
  long long wait_limit;
};

// Step schedule.  PAIR: slots = two query heads of a GQA group at one query
// tile.  !PAIR: slots = adjacent query tiles 2i, 2i+1 of one head, which walk
// the K/V tiles of the later one (under the causal mask a superset of the
// earlier tile's).  A CTA has two candidate units (one per local query chunk);
// units that see no key of the held block are skipped.
template <int D, bool PAIR>
struct StepPolicy : PolicyDefaults {
  using Args = StepParams;
  struct KvPos {
    int kh, kt, lim0, lim1;
    int32_t row;
  };
  const StepParams& p;
  int b, g, hq0, idx0, idx1;  // idx_u: tile index (PAIR) or tile-pair index (!PAIR) of unit u
  int n_units, first;         // units that run (a unit meeting no K/V tile is skipped), the first
  int u;                      // the selected unit
  float f_in, f_p, lse_new;   // merge weights of the row being stored (per thread)
  int64_t at_row;             // its output row index (token row * Hq + head)

  __device__ int qchunk(int half) const { return half == 0 ? p.r : 2 * p.N - 1 - p.r; }
  __device__ int kchunk(int half) const { return half == 0 ? p.s : 2 * p.N - 1 - p.s; }
  // query tile of slot h in unit uu; the tile whose K/V tiles the unit walks
  __device__ int qtile(int uu, int h) const { return PAIR ? (uu == 0 ? idx0 : idx1) : 2 * (uu == 0 ? idx0 : idx1) + h; }
  __device__ int walk_tile(int uu) const { return PAIR ? qtile(uu, 0) : min(qtile(uu, 1), p.nt - 1); }
  __device__ int valid(int qi) const { return max(0, min(BM, p.c - qi * BM)); }
  __device__ int head(int h) const { return PAIR ? hq0 + h : hq0; }

  __device__ Sched sched() const { return Sched{p.N, p.c, p.nt, p.causal, BN, p.nt}; }
  __device__ StepPolicy(const StepParams& a, int idx) : p(a) {
    if (PAIR) {
      const int pairs = a.group / 2;
      const int hp = idx % pairs; idx /= pairs;
      const int j = idx % a.nt; idx /= a.nt;
      g = idx % a.Hkv; idx /= a.Hkv;
      b = idx;
      hq0 = g * a.group + 2 * hp;
      idx0 = j;
      idx1 = a.nt - 1 - j;
    } else {
      const int hg = idx % a.group; idx /= a.group;
      const int jp = idx % a.ntp; idx /= a.ntp;
      g = idx % a.Hkv; idx /= a.Hkv;
      b = idx;
      hq0 = g * a.group + hg;
      idx0 = jp;
      idx1 = a.ntp - 1 - jp;
    }
    n_units = (nkv(0) > 0 ? 1 : 0) + (nkv(1) > 0 ? 1 : 0);
    first = nkv(0) > 0 ? 0 : 1;
    u = first;
  }
  // K/V tiles of held chunk kh that unit uu's walk tile meets
  __device__ int lim(int uu, int kh) const {
    const int qc = qchunk(uu), qi = walk_tile(uu);
    const int kc = kchunk(kh);
    if (!p.causal || kc < qc) return p.nt;
    if (kc > qc) return 0;
    return min(p.nt, (qi * BM + max(1, valid(qi)) - 1) / BN + 1);   // the diagonal chunk
  }
  __device__ int nkv(int uu) const { return lim(uu, 0) + lim(uu, 1); }
  __device__ int tiles() const { return n_units; }
  __device__ int kvh() const { return g; }
  __device__ void set_tile(int ti) { u = ti == 0 ? first : 1; }
  __device__ int32_t row_of(int uu, int qi, int off) const { return (b * 2 + uu) * p.c + qi * BM + off; }
  __device__ int q_head(int h) const { return head(h); }
  __device__ int32_t q_row(int h) const { return row_of(u, qtile(u, h), 0); }
  __device__ int q_valid(int h) const { return valid(qtile(u, h)); }
  __device__ int n_kv() const { return nkv(u); }
  __device__ void kv_begin(KvPos& k) const {
    k.kh = 0; k.kt = -1; k.lim0 = lim(u, 0); k.lim1 = lim(u, 1);
  }
  __device__ bool kv_next(KvPos& k) const {
    ++k.kt;
    if (k.kh == 0 && k.kt >= k.lim0) { k.kh = 1; k.kt = 0; }
    if (k.kh == 1 && k.kt >= k.lim1) return false;
    k.row = (b * 2 + k.kh) * p.c + k.kt * BN;
    return true;
  }
  __device__ void mask(const KvPos& k, int h, int row, int& col_lim, bool& masked) const {
    tile_mask(sched(), qchunk(u), qtile(u, h), kchunk(k.kh), k.kt, row, col_lim, masked);
  }

  // ---------------------------------------------------------------- epilogue: merge with the running result
  __device__ void prepare_row(int h, int row, float lse2, float inv_l) {
    at_row = static_cast<int64_t>(row_of(u, qtile(u, h), row)) * p.Hq + head(h);
    const float lp = lse2 * kLn2;  // natural log
    if (p.o_in == nullptr) {
      f_in = 0.f; f_p = inv_l; lse_new = lp;
      return;
    }
    const float li = p.lse_in[at_row];
    const float M = fmaxf(li, lp);
    if (M == -CUDART_INF_F) {
      f_in = 0.f; f_p = 0.f; lse_new = -CUDART_INF_F;
      return;
    }
    const float wi = li == -CUDART_INF_F ? 0.f : expf(li - M);
    const float wp = lp == -CUDART_INF_F ? 0.f : expf(lp - M);
    const float tot = wi + wp;
    f_in = wi / tot;
    f_p = wp / tot * inv_l;
    lse_new = M + logf(tot);
  }
  __device__ void store_o(int, int, int col0, const uint32_t (&o)[32], float) const {
    const int64_t at = at_row * D + col0;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(o[i + e]) * f_p;
      if (f_in != 0.f) {
        const float4 a = *reinterpret_cast<const float4*>(p.o_in + at + i);
        const float4 c = *reinterpret_cast<const float4*>(p.o_in + at + i + 4);
        x[0] += f_in * a.x; x[1] += f_in * a.y; x[2] += f_in * a.z; x[3] += f_in * a.w;
        x[4] += f_in * c.x; x[5] += f_in * c.y; x[6] += f_in * c.z; x[7] += f_in * c.w;
      }
      store8(at + i, x);
    }
  }
  __device__ void store_lse(int, int, float) const { p.lse_out[at_row] = lse_new; }

  __device__ void store8(int64_t at, const float (&x)[8]) const {
    if (p.out_bf16) {
      uint4 pk;
      pk.x = f2_bf16x2(x[0], x[1]);
      pk.y = f2_bf16x2(x[2], x[3]);
      pk.z = f2_bf16x2(x[4], x[5]);
      pk.w = f2_bf16x2(x[6], x[7]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o_out) + at) = pk;
    } else {
      float* dst = static_cast<float*>(p.o_out) + at;
      *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(x[4], x[5], x[6], x[7]);
    }
  }

  // A row the step does not touch keeps its running result: copied (or converted) when the output
  // is not the running buffer itself; O 0 and LSE -inf at a first step.
  __device__ void pass_row(int64_t at) const {
    const bool in_place = p.o_in != nullptr && static_cast<const void*>(p.o_in) == p.o_out && !p.out_bf16;
    if (!in_place) {
      for (int c0 = 0; c0 < D; c0 += 8) {
        float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (p.o_in) {
          const float4 a = *reinterpret_cast<const float4*>(p.o_in + at * D + c0);
          const float4 c = *reinterpret_cast<const float4*>(p.o_in + at * D + c0 + 4);
          x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
        }
        store8(at * D + c0, x);
      }
    }
    if (p.lse_in != p.lse_out || p.lse_in == nullptr) p.lse_out[at] = p.lse_in ? p.lse_in[at] : -CUDART_INF_F;
  }
  __device__ void skipped_rows(int h, int row) const {
    for (int uu = 0; uu < 2; ++uu) {
      if (nkv(uu) > 0) continue;
      const int qi = qtile(uu, h);
      if (row < valid(qi)) pass_row(static_cast<int64_t>(row_of(uu, qi, row)) * p.Hq + head(h));
    }
  }
  __device__ void write_empty(int tid, int nthreads) const {
    for (int i = tid; i < 2 * 2 * BM; i += nthreads) {
      const int uu = i / (2 * BM), h = (i / BM) % 2, row = i % BM;
      const int qi = qtile(uu, h);
      if (row < valid(qi)) pass_row(static_cast<int64_t>(row_of(uu, qi, row)) * p.Hq + head(h));
    }
  }
};

template <int D, bool PAIR>
ra_status launch_step(const void* q, const void* k, const void* v, const StepParams& prm, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  const int64_t rows = static_cast<int64_t>(prm.B) * 2 * prm.c;
  ra_status st;
  if ((st = make_map(&mq, q, D, prm.Hq, rows)) != RA_OK) return st;
  if ((st = make_map(&mk, k, D, prm.Hkv, rows)) != RA_OK) return st;
  if ((st = make_map(&mv, v, D, prm.Hkv, rows)) != RA_OK) return st;
  const int64_t items = PAIR ? static_cast<int64_t>(prm.B) * prm.Hkv * (prm.group / 2) * prm.nt
                             : static_cast<int64_t>(prm.B) * prm.Hq * prm.ntp;
  const size_t smem = sizeof(Smem2<D>) + 1024;
  RA_CUDA_TRY(cudaFuncSetAttribute(attn_pair_kernel<D, StepPolicy<D, PAIR>>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
  attn_pair_kernel<D, StepPolicy<D, PAIR>><<<static_cast<unsigned>(items), kThreads2, smem, stream>>>(mq, mk, mv,
                                                                                                     prm);
  RA_LAUNCH_CHECK("attn_pair_kernel<StepPolicy>");
  return RA_OK;
}

}  // namespace

extern "C" ra_status ra_ring_step_fwd(const void* q, const void* k, const void* v, int32_t B, int32_t Hq,
                                      int32_t Hkv, int32_t c, int32_t d, int32_t n_ranks, int32_t rank,
                                      int32_t src, int32_t causal, float scale, const float* o_in,
                                      const float* lse_in, void* o_out, ra_dtype out_dt, float* lse_out,
                                      ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(B >= 1 && Hq >= 1 && Hkv >= 1 && c >= 1, "B, Hq, Hkv and c must be >= 1");
  RA_REQUIRE(Hq % Hkv == 0, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  RA_REQUIRE(n_ranks >= 1, "n_ranks must be >= 1 (got %d)", n_ranks);
  RA_REQUIRE(rank >= 0 && rank < n_ranks && src >= 0 && src < n_ranks, "rank (%d) and src (%d) must be in [0, %d)",
             rank, src, n_ranks);
  RA_REQUIRE(static_cast<int64_t>(B) * 2 * c < (int64_t(1) << 31), "B*2c must be < 2^31");
  RA_REQUIRE(out_dt == RA_F32 || out_dt == RA_BF16, "unknown out dtype");
  if (d != 64 && d != 128) return ra::fail(RA_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", d);
  RA_REQUIRE(q && k && v && o_out && lse_out, "NULL pointer");
  RA_REQUIRE((o_in == nullptr) == (lse_in == nullptr), "o_in and lse_in are given together or not at all");
  RA_REQUIRE(ra::aligned16(q) && ra::aligned16(k) && ra::aligned16(v) && ra::aligned16(o_out) &&
                 (o_in == nullptr || ra::aligned16(o_in)) && reinterpret_cast<uintptr_t>(lse_out) % 4 == 0 &&
                 reinterpret_cast<uintptr_t>(lse_in) % 4 == 0,
             "q, k, v, o_in and o_out must be 16-byte aligned");
  RA_REQUIRE(!(o_in != nullptr && static_cast<const void*>(o_in) == o_out && out_dt == RA_BF16),
             "a bf16 output cannot overwrite the fp32 running output in place");
  StepParams prm;
  prm.B = B; prm.Hq = Hq; prm.Hkv = Hkv; prm.group = Hq / Hkv; prm.N = n_ranks; prm.r = rank; prm.s = src;
  prm.c = c; prm.nt = static_cast<int>(ra::ceil_div(c, BM)); prm.ntp = (prm.nt + 1) / 2;
  prm.causal = causal ? 1 : 0;
  prm.scale_log2 = (scale > 0.f ? scale : 1.f / sqrtf(static_cast<float>(d))) * 1.4426950408889634f;
  prm.o_in = o_in; prm.lse_in = lse_in; prm.o_out = o_out; prm.out_bf16 = out_dt == RA_BF16 ? 1 : 0;
  prm.lse_out = lse_out; prm.wait_limit = ra::wait_limit();
  const bool pair = prm.group % 2 == 0;
  const int64_t items = pair ? static_cast<int64_t>(B) * Hkv * (prm.group / 2) * prm.nt
                             : static_cast<int64_t>(B) * Hq * prm.ntp;
  RA_REQUIRE(items < (int64_t(1) << 31), "too many work items");
  if (d == 128) return pair ? launch_step<128, true>(q, k, v, prm, stream) : launch_step<128, false>(q, k, v, prm, stream);
  return pair ? launch_step<64, true>(q, k, v, prm, stream) : launch_step<64, false>(q, k, v, prm, stream);
}
