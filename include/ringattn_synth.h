/*
 * ringattn_synth.h -- seeded synthetic inputs on the device, for benchmarks
 * and tests whose inputs are too large to draw on the host.
 *
 * The draw is counter-based, so any element can be reproduced on its own
 * (the Python module context_long_sequence_ring_gb300.inputs implements the
 * same definition on the host):
 *   mix64(z): SplitMix64 finaliser (Steele, Lea and Flood, OOPSLA 2014)
 *     z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *     z = (z ^ (z >> 27)) * 0x94D049BB133111EB;  return z ^ (z >> 31);
 *   element i of a tensor with 64-bit key K: u = mix64(K + (i+1)*0x9E3779B97F4A7C15)
 *   value = table[u >> 48]   (all arithmetic mod 2^64)
 * The key and the 65536-entry value table are supplied by the caller.
 */
#ifndef RINGATTN_SYNTH_H
#define RINGATTN_SYNTH_H

#include "ringattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* out[i] = table[u_i >> 48] for i in [0, n), elements of elem_bytes (2 or 4).
 * table device [65536 * elem_bytes]; out device [n * elem_bytes]. */
ra_status ra_synth_fill(uint64_t key, int64_t n, const void* table, int32_t elem_bytes,
                        void* out, ra_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* RINGATTN_SYNTH_H */
