// zero_qwz.cuh -- the ZeRO++ qwZ block quantizer's per-element arithmetic,
// shared by the standalone quantize kernel (zero_qwz.cu) and the quantizing
// epilogue of the ZeRO-3 update pass (zero_step_kernels.cuh), so both write the
// same codes and scales bit for bit.
//
// Quantization block: ZERO_QBLOCK consecutive elements of a shard, counted from
// the shard's start; scale = max|x| / qmax (qmax = 127 or 7, binary32
// division; NaN elements do not take part in the max), code =
// round-half-even(x / scale) clamped to [-qmax, qmax] (0 when the scale is 0 and
// for NaN).  4-bit codes are packed two per byte, the even element in the low
// nibble.
#pragma once

#include "zero_common.cuh"

namespace zero {

#define ZERO_QBLOCK 256

template <int BITS> struct QMax;
template <> struct QMax<8> { static constexpr float v = 127.0f; };
template <> struct QMax<4> { static constexpr float v = 7.0f; };

static __device__ __forceinline__ int32_t quant1(float x, float scale, float qmax)
{
    if (scale == 0.0f) return 0;
    int32_t c = __float2int_rn(__fdiv_rn(x, scale));
    const int32_t m = (int32_t)qmax;
    return c > m ? m : (c < -m ? -m : c);
}

// Adding 1.5 * 2^23 to a float t with |t| <= 2^22 rounds it to an integer (nearest,
// ties to even) and leaves that integer, two's complement, in the low mantissa
// bits of the sum; the low 8 (or 4) bits of the sum are then the code's byte
// (nibble).
#define ZERO_RND 12582912.0f

// Two fp32 values as one packed pair, and the sm_100+ packed arithmetic on pairs
// (each lane rounded to nearest-even exactly as the scalar operation).
typedef unsigned long long f32x2_t;
static __device__ __forceinline__ f32x2_t pack2(float a, float b)
{
    f32x2_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
static __device__ __forceinline__ void unpack2(f32x2_t r, float& a, float& b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
static __device__ __forceinline__ f32x2_t mul2(f32x2_t a, f32x2_t b)
{
    f32x2_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
static __device__ __forceinline__ f32x2_t add2(f32x2_t a, f32x2_t b)
{
    f32x2_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
static __device__ __forceinline__ f32x2_t sub2(f32x2_t a, f32x2_t b)
{
    f32x2_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// max that returns NaN when either input is NaN
static __device__ __forceinline__ float max_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// The codes of N elements (N even) of one block: each is the integer nearest to
// fl(v / scale) (ties to even), clamped to [-qmax, qmax]; returned as words whose
// low bits hold the two's-complement code.
//
// Fast path, for a scale in the normal range, without a division per element:
// r = 1 / scale to within 2^-23 relative (the hardware approximation refined by
// one Newton-Raphson step), t = fl(v * r).  Since |v| <= max|x| and
// scale = fl(max|x| / qmax), |v / scale| <= qmax (1 + 2^-23), so t is within 2^-16
// of v / scale and within 2^-15 of fl(v / scale).  Rounding t (by adding
// 1.5 * 2^23) therefore gives the code unless t lies within 2^-14 of a
// half-integer, and it never passes qmax (|t| < qmax + 2^-15), so no clamp is
// needed.  Those elements, and NaN, take the exact quotient instead.  With 16-bit
// weights they are not rare (about one in 300 for bf16, one in 2500 for fp16):
// v / scale is then close to qmax m_v / m_max 2^k for the short mantissas of v and
// max|x|, which often falls next to a half-integer.
template <int BITS, int N>
static __device__ __forceinline__ void codes_n(const float* v, float scale, uint32_t* c)
{
    const float qmax = QMax<BITS>::v;
    if (!(scale >= 0x1p-126f && scale <= 0x1p126f)) {
#pragma unroll
        for (int i = 0; i < N; i++) c[i] = (uint32_t)quant1(v[i], scale, qmax);
        return;
    }
    float r0;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(scale));
    const float r = __fmaf_rn(__fmaf_rn(-scale, r0, 1.0f), r0, r0);
    const f32x2_t r2 = pack2(r, r), rnd2 = pack2(ZERO_RND, ZERO_RND);
    float dmax = 0.0f;
    float d[N];                                       // t minus its rounded integer
#pragma unroll
    for (int i = 0; i < N; i += 2) {                  // two lanes at a time
        const f32x2_t t = mul2(pack2(v[i], v[i + 1]), r2);
        const f32x2_t u = add2(t, rnd2);
        float u0, u1;
        unpack2(sub2(t, sub2(u, rnd2)), d[i], d[i + 1]);
        dmax = max_nan(dmax, fabsf(d[i]));
        dmax = max_nan(dmax, fabsf(d[i + 1]));
        unpack2(u, u0, u1);
        c[i] = __float_as_uint(u0);
        c[i + 1] = __float_as_uint(u1);
    }
    // the elements within 2^-14 of a half-integer (or NaN) take the exact quotient;
    // their residuals are kept from above rather than recomputed (measured: the
    // standalone quantizer 82 -> 74 us on a 120 M-element bf16 shard)
    if (!(dmax <= 0.5f - 0x1p-14f)) {
#pragma unroll
        for (int i = 0; i < N; i++)
            if (!(fabsf(d[i]) <= 0.5f - 0x1p-14f)) c[i] = (uint32_t)quant1(v[i], scale, qmax);
    }
}

// Store the codes of elements e .. e+8 (those below n).  4-bit codes: two per
// byte, the even element in the low nibble; an odd tail leaves the high nibble 0.
template <int BITS>
static __device__ __forceinline__ void store8(uint8_t* __restrict__ codes, int64_t n, int64_t e,
                                              const uint32_t* c)
{
    if (BITS == 8) {
        const uint32_t lo = __byte_perm(__byte_perm(c[0], c[1], 0x0040),
                                        __byte_perm(c[2], c[3], 0x0040), 0x5410);
        const uint32_t hi = __byte_perm(__byte_perm(c[4], c[5], 0x0040),
                                        __byte_perm(c[6], c[7], 0x0040), 0x5410);
        if (e + 8 <= n) {
            *reinterpret_cast<uint2*>(codes + e) = make_uint2(lo, hi);
        } else {
            for (int i = 0; i < 8 && e + i < n; i++) codes[e + i] = (uint8_t)c[i];
        }
    } else {
        uint32_t w = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) w |= (c[i] & 0xFu) << (4 * i);
        if (e + 8 <= n) {
            *reinterpret_cast<uint32_t*>(codes + e / 2) = w;
        } else {
            for (int b = 0; 2 * b < 8 && e + 2 * b < n; b++)
                codes[e / 2 + b] = (uint8_t)((w >> (8 * b)) & (e + 2 * b + 1 < n ? 0xFF : 0x0F));
        }
    }
}

}  // namespace zero
