// Rotary position embedding fused with the row gather of the zigzag
// partition.
//
// Source: guijiagi.com tag page "Ring Attention", article on the evolution of
// long-context techniques, section 1.2 "RoPE": the vector at position m is
// rotated as x e^{i m theta_i}, theta_i = base^(-2i/d), which in real form is
// x*cos + rotate_half(x)*sin; component j < d/2 and component j + d/2 are the
// real and imaginary parts of the j-th complex number.
//
// The gather to the zigzag layout already reads and writes every Q and K row
// once, so rotating there costs no extra HBM traffic; rotating inside the
// attention kernel instead would redo it for every query tile that visits a
// K tile.
//
// Angles.  m * theta_i reaches 1.3e5 rad at 131072 tokens, where a float
// product alone is off by up to 4e-3 rad.  The angle is therefore taken in
// turns, m * phi_i with phi_i = theta_i / (2 pi) held as an unevaluated sum of
// two floats (hi + lo, computed in double on the host).  The product m * hi is
// split exactly into p + e with one FMA (Dekker's error-free product), the
// integer turns rint(p) drop out exactly, and the remaining fraction in
// [-1/2, 1/2] goes to sincospif.  The angle error is then about 1e-7 turns,
// independent of the position.
#include <algorithm>
#include <cmath>

#include "ra_common.cuh"

RA_DEFINE_ERROR_FETCH(fetch_error_rope)

namespace {

constexpr int kRopeThreads = 256;
constexpr int kMaxHalf = 128;            // d <= 256
constexpr int kHeadsInFlight = 4;        // heads whose loads a thread issues before it rotates them
constexpr int kPositionLimit = 1 << 24;  // positions are exact in a float below this

struct RopeParams {
  float2 phase[kMaxHalf];  // phi_i = theta_i / 2pi as hi + lo
};

// ---------------------------------------------------------------- packed fp32 pairs
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// 16 bytes of T as VEC/2 packed fp32 pairs, and back (rounded to nearest even).
template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4& u, uint64_t (&f)[4]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = pk2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  }
  __device__ static uint4 pack(const uint64_t (&f)[4]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo, hi;
      asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(f[i]));
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[i]) : "f"(hi), "f"(lo));
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <> struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& u, uint64_t (&f)[2]) {
    f[0] = (static_cast<uint64_t>(u.y) << 32) | u.x;
    f[1] = (static_cast<uint64_t>(u.w) << 32) | u.z;
  }
  __device__ static uint4 pack(const uint64_t (&f)[2]) {
    return make_uint4(static_cast<uint32_t>(f[0]), static_cast<uint32_t>(f[0] >> 32), static_cast<uint32_t>(f[1]),
                      static_cast<uint32_t>(f[1] >> 32));
  }
};

// Source row of output row r (identity when idx is NULL); -1 for a pad row.
__device__ __forceinline__ int64_t source_row(const int32_t* idx, int64_t r, int64_t src_rows) {
  if (!idx) return r;
  const int32_t s = idx[r];
  if (s >= src_rows) {
    ra_record_error(RA_ERR_DEVICE_BOUNDS, 40);
    return -1;
  }
  return s;
}

// Work layout.  A token's row is H heads of d = 2 * vh vectors of 16 bytes.
// One thread owns one (token, chunk k) pair for all H heads: it computes the
// VEC angles of chunk k once, in registers, and applies them to every head's
// vector at chunk k of the first half (real parts) and its partner at chunk k
// of the second half (imaginary parts).  vh threads thus cover a token and
// compute exactly its d/2 angles, with no shared memory and no barrier.
// Consecutive threads take consecutive chunks of a token, so each load or
// store of a warp covers whole 128-byte segments of 32 / vh tokens.
// Heads go in groups of kHeadsInFlight: the group's loads are issued before
// its rotations (for the first group, before the angles are computed).  src
// and dst may be the same buffer (in place, identity gather): every vector is
// read and then written by the same thread only, so they carry no __restrict__.
template <typename T>
__global__ void __launch_bounds__(kRopeThreads)
    rope_gather_kernel(const uint4* src, int64_t src_rows, const int32_t* __restrict__ idx, int64_t rows,
                       const int32_t* __restrict__ positions, int32_t H, int32_t vh,
                       const __grid_constant__ RopeParams prm, uint4* dst) {
  constexpr int VEC = Vec<T>::N;
  constexpr int NP = VEC / 2;                    // packed pairs per vector
  const int64_t row_vecs = static_cast<int64_t>(H) * 2 * vh;
  const int64_t head_vecs = 2 * vh;
  const int64_t total = rows * vh;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kRopeThreads;

  for (int64_t w = static_cast<int64_t>(blockIdx.x) * kRopeThreads + threadIdx.x; w < total; w += stride) {
    const int64_t r = w / vh;
    const int k = static_cast<int>(w - r * vh);
    const int64_t s = source_row(idx, r, src_rows);
    uint4* y = dst + r * row_vecs + k;
    if (s < 0) {
      for (int h = 0; h < H; ++h) {
        y[h * head_vecs] = make_uint4(0, 0, 0, 0);
        y[h * head_vecs + vh] = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    const uint4* x = src + s * row_vecs + k;
    int32_t pos = positions[s];

    uint4 a[kHeadsInFlight], b[kHeadsInFlight];
#pragma unroll
    for (int j = 0; j < kHeadsInFlight; ++j) {
      if (j < H) {
        a[j] = x[j * head_vecs];
        b[j] = x[j * head_vecs + vh];
      }
    }

    // the VEC angles m * theta_i, i = k*VEC .. k*VEC + VEC-1, as packed cos, sin, -sin
    if (pos < 0 || pos >= kPositionLimit) {
      ra_record_error(RA_ERR_DEVICE_BOUNDS, 41);
      pos = 0;
    }
    const float m = static_cast<float>(pos);
    uint64_t c2[NP], s2[NP], ns2[NP];
#pragma unroll
    for (int e = 0; e < NP; ++e) {
      float cn[2], sn[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float2 ph = prm.phase[k * VEC + 2 * e + u];
        const float p = m * ph.x;
        const float err = fmaf(m, ph.x, -p);           // m*hi = p + err exactly
        const float f = (p - rintf(p)) + fmaf(m, ph.y, err);
        sincospif(2.0f * f, &sn[u], &cn[u]);
      }
      c2[e] = pk2(cn[0], cn[1]);
      s2[e] = pk2(sn[0], sn[1]);
      ns2[e] = pk2(-sn[0], -sn[1]);
    }

    for (int h0 = 0; h0 < H; h0 += kHeadsInFlight) {
      if (h0 > 0) {
#pragma unroll
        for (int j = 0; j < kHeadsInFlight; ++j) {
          if (h0 + j < H) {
            a[j] = x[(h0 + j) * head_vecs];
            b[j] = x[(h0 + j) * head_vecs + vh];
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kHeadsInFlight; ++j) {
        if (h0 + j >= H) break;
        uint64_t x1[NP], x2[NP], o1[NP], o2[NP];
        Vec<T>::unpack(a[j], x1);
        Vec<T>::unpack(b[j], x2);
#pragma unroll
        for (int e = 0; e < NP; ++e) {
          o1[e] = fma2(x1[e], c2[e], mul2(x2[e], ns2[e]));   // real:      x1 cos - x2 sin
          o2[e] = fma2(x2[e], c2[e], mul2(x1[e], s2[e]));    // imaginary: x2 cos + x1 sin
        }
        y[(h0 + j) * head_vecs] = Vec<T>::pack(o1);
        y[(h0 + j) * head_vecs + vh] = Vec<T>::pack(o2);
      }
    }
  }
}

}  // namespace

extern "C" ra_status ra_rope_gather(const void* src, int64_t src_rows, int32_t H, int32_t d, ra_dtype dt,
                                    const int32_t* idx, int64_t rows, const int32_t* positions, double base,
                                    void* dst, ra_stream stream) {
  ra::clear_error();
  RA_REQUIRE(dt == RA_BF16 || dt == RA_F32, "dtype must be RA_BF16 or RA_F32");
  const int vec = dt == RA_BF16 ? 8 : 4;
  RA_REQUIRE(H >= 1, "H must be >= 1");
  RA_REQUIRE(d >= 2 * vec && d <= 2 * kMaxHalf && d % (2 * vec) == 0,
             "d must be a multiple of %d in [%d, %d]", 2 * vec, 2 * vec, 2 * kMaxHalf);
  RA_REQUIRE(base > 1.0 && std::isfinite(base), "base must be finite and > 1");
  RA_REQUIRE(rows >= 0 && src_rows >= 0, "negative size");
  RA_REQUIRE(idx || rows == src_rows, "without idx, rows must equal src_rows");
  if (rows == 0) return RA_OK;
  RA_REQUIRE(src && dst && positions, "NULL pointer");
  RA_REQUIRE(ra::aligned16(src) && ra::aligned16(dst), "src and dst must be 16-byte aligned");
  const int64_t row_bytes = static_cast<int64_t>(H) * d * (dt == RA_BF16 ? 2 : 4);
  if (idx) {
    const char* s0 = static_cast<const char*>(src);
    const char* d0 = static_cast<const char*>(dst);
    RA_REQUIRE(d0 + rows * row_bytes <= s0 || s0 + src_rows * row_bytes <= d0,
               "dst must not overlap src when idx is given");
  } else {
    RA_REQUIRE(src == dst || static_cast<const char*>(dst) + rows * row_bytes <= static_cast<const char*>(src) ||
                   static_cast<const char*>(src) + rows * row_bytes <= static_cast<const char*>(dst),
               "dst must be src itself (in place) or not overlap it");
  }

  RopeParams prm;
  const int half = d / 2;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < half; ++i) {
    const double phi = std::pow(base, -2.0 * i / d) / two_pi;   // theta_i in turns
    const float hi = static_cast<float>(phi);
    prm.phase[i] = make_float2(hi, static_cast<float>(phi - static_cast<double>(hi)));
  }
  for (int i = half; i < kMaxHalf; ++i) prm.phase[i] = make_float2(0.f, 0.f);

  const int vh = half / vec;
  const int64_t n_blocks = ra::ceil_div(rows * vh, kRopeThreads);
  int dev = 0, sms = 0, per_sm = 0;
  RA_CUDA_TRY(cudaGetDevice(&dev));
  RA_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (dt == RA_BF16) {
    RA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rope_gather_kernel<__nv_bfloat16>,
                                                              kRopeThreads, 0));
    const int64_t blocks = std::min<int64_t>(n_blocks, static_cast<int64_t>(sms) * std::max(per_sm, 1));
    rope_gather_kernel<__nv_bfloat16><<<blocks, kRopeThreads, 0, stream>>>(
        static_cast<const uint4*>(src), src_rows, idx, rows, positions, H, vh, prm, static_cast<uint4*>(dst));
  } else {
    RA_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rope_gather_kernel<float>, kRopeThreads, 0));
    const int64_t blocks = std::min<int64_t>(n_blocks, static_cast<int64_t>(sms) * std::max(per_sm, 1));
    rope_gather_kernel<float><<<blocks, kRopeThreads, 0, stream>>>(
        static_cast<const uint4*>(src), src_rows, idx, rows, positions, H, vh, prm, static_cast<uint4*>(dst));
  }
  RA_LAUNCH_CHECK("rope_gather_kernel");
  return RA_OK;
}
