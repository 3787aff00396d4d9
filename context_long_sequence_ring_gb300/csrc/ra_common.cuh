// Shared host and device helpers of libringattn (no attention arithmetic).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ringattn.h"

namespace ra {

// ---------------------------------------------------------------- host side

// Record the thread-local error text (printf-style) and return `s`.
ra_status fail(ra_status s, const char* fmt, ...);
// Map a CUDA error to RA_ERR_CUDA with context; RA_OK on cudaSuccess.
ra_status cuda_status(cudaError_t e, const char* what);
// Clears the thread-local error text at the start of an entry point.
void clear_error();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Per-module device error words are fetched (and cleared) through these.
int fetch_error_api(int* where);
int fetch_error_cache(int* where);
int fetch_error_decode(int* where);
int fetch_error_attn_f32(int* where);
int fetch_error_attn_bf16(int* where);
int fetch_error_attn_block(int* where);
int fetch_error_rope(int* where);
int fetch_error_ring_step(int* where);

}  // namespace ra

#define RA_REQUIRE(cond, ...)                                 \
  do {                                                        \
    if (!(cond)) return ra::fail(RA_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)

#define RA_CUDA_TRY(expr)                                     \
  do {                                                        \
    cudaError_t e_ = (expr);                                  \
    if (e_ != cudaSuccess) return ra::cuda_status(e_, #expr); \
  } while (0)

// Launch-error check after a <<<>>> launch.
#define RA_LAUNCH_CHECK(name) RA_CUDA_TRY(cudaGetLastError())

// ---------------------------------------------------------------- device side
// Each translation unit that includes this header gets its own error word
// (no relocatable device code is needed); the module's fetch function reads
// and clears it.
static __device__ int ra_err_word[2];

#define RA_DEFINE_ERROR_FETCH(fn)                                                  \
  namespace ra {                                                                   \
  int fn(int* where) {                                                             \
    int w[2] = {0, 0};                                                             \
    if (cudaMemcpyFromSymbol(w, ra_err_word, sizeof(w)) != cudaSuccess) return -1; \
    if (w[0] != 0) {                                                               \
      int z[2] = {0, 0};                                                           \
      if (cudaMemcpyToSymbol(ra_err_word, z, sizeof(z)) != cudaSuccess) return -1; \
    }                                                                              \
    if (where) *where = w[1];                                                      \
    return w[0];                                                                   \
  }                                                                                \
  }

__device__ __forceinline__ void ra_record_error(int status, int where) {
  if (atomicCAS(&ra_err_word[0], 0, status) == 0) atomicExch(&ra_err_word[1], where);
}
