/*
 * libswa synthetic-input generator (benchmarks and tests only; no part of the
 * attention or allocation method).
 *
 * Counter-based: element i of stream s under seed S is
 *   base = mix64((S << 32) ^ s),  z = mix64(base + (i + 1) * 0x9E3779B97F4A7C15)
 * with mix64 the SplitMix64 output function (Steele, Lea & Flood, OOPSLA
 * 2014); the sum of z's four 16-bit fields, minus 131070, times
 * float32(sqrt(3)/65536) gives an approximately N(0,1) float32 (bf16 outputs
 * round it to nearest even).  The element index of token (layer, req, pos,
 * head, dim) is layer<<47 | req<<35 | pos<<15 | head<<8 | dim.
 */
#ifndef SWA_SYNTH_H
#define SWA_SYNTH_H

#include <stdint.h>

#include "swa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* out[n][heads][dim] (f32 when out_dtype == SWA_DTYPE_F32, else bf16) for
 * tokens (req[i], pos[i]) (device int64 arrays) of `layer`. */
swa_status swa_synth_tokens(uint64_t seed, int32_t stream_id, int32_t layer,
                            const int64_t *req, const int64_t *pos, int64_t n,
                            int32_t heads, int32_t dim, int32_t out_dtype,
                            void *out, swa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif
