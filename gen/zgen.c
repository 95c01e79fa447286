/*
 * zgen.c -- host implementation of the seeded input generator (see zgen.h).
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared -o libzgen.so zgen.c
 */
#include "zgen.h"

#include <string.h>

#define G 0x9E3779B97F4A7C15ull

static uint64_t mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t zgen_key(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank)
{
    uint64_t k = mix(seed ^ ((uint64_t)stream * G));
    k = mix(k + (uint64_t)step * G);
    return mix(k + (uint64_t)rank * G);
}

static float sample(uint64_t key, int64_t index, float kappa, float scale)
{
    uint64_t z = mix(key + ((uint64_t)index + 1u) * G);
    int32_t k = (int32_t)(z & 0xFFFF) + (int32_t)((z >> 16) & 0xFFFF)
              + (int32_t)((z >> 32) & 0xFFFF) + (int32_t)(z >> 48) - 131070;
    float v = (float)k * kappa;
    return v * scale;
}

/* Round a binary32 to fp16 / bf16, nearest-even, by integer operations on the
 * bit pattern (input preparation; the CUDA twin uses the CUDA intrinsics). */
static uint16_t round_half(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);          /* NaN */
    if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);         /* >= 65520: inf */
    if (ax < 0x38800000u) {                                           /* < 2^-14: subnormal */
        if (ax < 0x33000000u) return (uint16_t)sign;                  /* <= 2^-25: zero */
        uint32_t e = ax >> 23;                                        /* 102..112 */
        uint32_t mant = (ax & 0x7FFFFFu) | 0x800000u;
        uint32_t shift = 126u - e;                                    /* to units of 2^-24 */
        uint32_t q = mant >> shift;
        uint32_t rem = mant & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1u);
        if (rem > half || (rem == half && (q & 1u))) q++;
        return (uint16_t)(sign | q);
    }
    uint32_t r = ax - 0x38000000u;                 /* rebias exponent 127 -> 15 */
    uint32_t q = r >> 13;
    uint32_t rem = r & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q++;
    return (uint16_t)(sign | q);
}

static uint16_t round_bf16(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    if ((x & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((x >> 16) | 0x40u);
    uint32_t lsb = (x >> 16) & 1u;
    return (uint16_t)((x + 0x7FFFu + lsb) >> 16);
}

static uint16_t round16(int dtype, float f)
{
    return dtype == 0 ? round_half(f) : round_bf16(f);
}

void zgen_f32(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank,
              int64_t index0, int64_t n, float kappa, float scale, float* out)
{
    uint64_t key = zgen_key(seed, stream, step, rank);
    for (int64_t i = 0; i < n; i++) out[i] = sample(key, index0 + i, kappa, scale);
}

void zgen_16(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank,
             int64_t index0, int64_t n, float kappa, float scale, int dtype, uint16_t* out)
{
    uint64_t key = zgen_key(seed, stream, step, rank);
    for (int64_t i = 0; i < n; i++) out[i] = round16(dtype, sample(key, index0 + i, kappa, scale));
}

void zgen_ranks_16(uint64_t seed, uint32_t stream, uint32_t step, int nd,
                   int64_t index0, int64_t n, int64_t rank_stride,
                   float kappa, float scale, int dtype, uint16_t* out)
{
    for (int r = 0; r < nd; r++) {
        uint16_t* row = out + (int64_t)r * rank_stride;
        zgen_16(seed, stream, step, (uint32_t)r, index0, n, kappa, scale, dtype, row);
        if (rank_stride > n) memset(row + n, 0, (size_t)(rank_stride - n) * sizeof(uint16_t));
    }
}

void zgen_16_at(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank,
                const int64_t* idx, int64_t n, float kappa, float scale, int dtype,
                uint16_t* out)
{
    uint64_t key = zgen_key(seed, stream, step, rank);
    for (int64_t j = 0; j < n; j++) out[j] = round16(dtype, sample(key, idx[j], kappa, scale));
}

void zgen_f32_at(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank,
                 const int64_t* idx, int64_t n, float kappa, float scale, float* out)
{
    uint64_t key = zgen_key(seed, stream, step, rank);
    for (int64_t j = 0; j < n; j++) out[j] = sample(key, idx[j], kappa, scale);
}
