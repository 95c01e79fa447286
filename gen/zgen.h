/*
 * zgen.h -- seeded synthetic inputs for the optimizer-step tests and benchmark.
 *
 * This module produces inputs only (gradients, master weights, foreign
 * parameter shards).  It holds none of the optimizer step's arithmetic and is
 * shared by the CPU oracle side and the GPU side of the tests as their common
 * source of inputs.  The host version (zgen.c) and the CUDA twin
 * (zgen_cuda.cu) must produce identical bits; a GPU test checks that.
 *
 * Definition of element (seed, stream, step, rank, index):
 *   G      = 0x9E3779B97F4A7C15 (the SplitMix64 increment)
 *   mix(z) = the SplitMix64 output function (Steele, Lea & Flood, 2014):
 *            z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *            z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *            z ^ (z >> 31)
 *   key    = mix(mix(mix(seed ^ (stream * G)) + step * G) + rank * G)
 *   z      = mix(key + (index + 1) * G)        (the index-th SplitMix64 output)
 *   k      = lane0 + lane1 + lane2 + lane3 - 131070, the four 16-bit lanes of z
 *            (an Irwin-Hall(4) draw, mean 0, variance 4 (65536^2 - 1) / 12)
 *   value  = ((float)k * kappa) * scale        (two binary32 multiplies)
 *   16-bit inputs: value rounded to fp16 / bf16, nearest-even.
 * kappa = sigma / sqrt(4 (65536^2 - 1) / 12) rounded to binary32 by the caller,
 * so the value has standard deviation sigma (bounded at +-3.46 sigma).
 */
#ifndef ZGEN_H
#define ZGEN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ZGEN_STREAM_GRAD = 1, ZGEN_STREAM_MASTER = 2, ZGEN_STREAM_SHARD = 3 };

uint64_t zgen_key(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank);

/* out[i] = value(index0 + i), binary32 */
void zgen_f32(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank,
              int64_t index0, int64_t n, float kappa, float scale, float* out);

/* out[i] = 16-bit value(index0 + i); dtype 0 = fp16, 1 = bf16 */
void zgen_16(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank,
             int64_t index0, int64_t n, float kappa, float scale, int dtype, uint16_t* out);

/* out[r * rank_stride + i] = 16-bit value of (rank r, index index0 + i) for
 * r < nd, i < n; out[r * rank_stride + i] = 0 for n <= i < rank_stride.      */
void zgen_ranks_16(uint64_t seed, uint32_t stream, uint32_t step, int nd,
                   int64_t index0, int64_t n, int64_t rank_stride,
                   float kappa, float scale, int dtype, uint16_t* out);

/* values at an index list (for sampled checks): out[j] = value(idx[j]) */
void zgen_16_at(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank,
                const int64_t* idx, int64_t n, float kappa, float scale, int dtype,
                uint16_t* out);
void zgen_f32_at(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank,
                 const int64_t* idx, int64_t n, float kappa, float scale, float* out);

#ifdef __cplusplus
}
#endif
#endif
