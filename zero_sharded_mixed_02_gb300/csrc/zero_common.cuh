// zero_common.cuh -- device-side definitions shared by the step kernels.
//
// Every floating-point operation of the step is written with an explicitly
// rounded intrinsic (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn, ...), so the
// compiler cannot contract a multiply and an add into one FMA and each
// operation rounds once, in the order the step defines.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define ZERO_MAX_BLOCKS 8192
#define ZERO_MAX_ND 1024
#define ZERO_THREADS 256

namespace zero {

// Optimizer scalars that persist across steps (device copy, owned by the plan).
struct DevScalars {
    float   loss_scale;
    int32_t good_steps;
    int64_t t;
    double  beta1_pow;   // beta1^t by repeated multiplication
    double  beta2_pow;
    // the next step's bias corrections, 1 - beta^(t+1) rounded to binary32 from
    // double: kept here by the one thread that advances t, so the fused pass's
    // threads read them instead of each computing them in binary64
    float   bc1_next;
    float   bc2_next;
    // ping-pong steps: which of the caller's two state sets holds the current
    // master, m, v (0 after plan creation and after a checkpoint load)
    int32_t cur;
    int32_t pad;
};

// What one step reports; written by the last block of the reduce pass.
struct DevStatus {
    int32_t skipped;
    int32_t overflow;
    double  grad_norm;
    float   clip_coef;
    float   bc1, bc2;      // bias corrections 1 - beta^t of this step
    float   used_scale;    // loss scale this step divided by
    int32_t err;
    int32_t pad;
};

struct DevState {
    DevScalars sc;
    DevStatus  st;
    unsigned int counter;               // last-block ticket, back to 0 after each pass
    unsigned int pad;
    double  partial[ZERO_MAX_BLOCKS];   // per-block sum of squares
    int32_t flag[ZERO_MAX_BLOCKS];      // per-block overflow flag
};

// Adam constants, rounded to binary32 on the host from double
// (1 - beta1, 1 - beta2 and 1 - lr*wd are each computed in double once).
struct AdamK {
    float lr, b1, b2, eps, wd, omb1, omb2, decay;
    int   decoupled, use_wd;
};

struct StepArgs {
    const uint16_t* grads;   // [nd][rank_stride]
    float*    master;
    float*    m;
    float*    v;
    uint16_t* params;
    float*    g32;           // two-pass workspace (fp32 averaged, unscaled gradient)
    int64_t   n;             // elements updated
    int64_t   rank_stride;   // elements between consecutive ranks' gradients
    int       nd;
    AdamK     k;
    float     clip;          // 0 = off
    int       dynamic;       // dynamic loss scaling: overflow skips + backoff
    int       skip_static;   // static scale: an overflow skips the step too
    float     backoff;
    int       growth_interval;
    DevState* state;
    // ping-pong step: the second set of master, m, v; the step reads set `cur`
    // (DevScalars) and writes the other, and a step that is not skipped flips cur
    float*    master2 = nullptr;
    float*    m2 = nullptr;
    float*    v2 = nullptr;
    int       pingpong = 0;
    // ZeRO-3 step with the qwZ quantizer in its epilogue: the updated 16-bit
    // parameters' block codes and scales (as zero_quantize_shard writes them)
    uint8_t*  qcodes = nullptr;
    float*    qscales = nullptr;
    // bucketed step: the reduce pass covers one bucket and records its partial
    int       bucket = -1;                // -1: a whole step
    // a bucket's reduce: this bucket's per-block squared-norm partials and flags;
    // the apply step: every bucket's, [nbuckets][bucket_grid]
    double*   bucket_partial = nullptr;
    int32_t*  bucket_flag = nullptr;
};

// ---- 16-bit formats --------------------------------------------------------
template <int DT> __device__ __forceinline__ void widen2(uint32_t w, float& lo, float& hi);
template <> __device__ __forceinline__ void widen2<0>(uint32_t w, float& lo, float& hi)
{
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
    lo = f.x;
    hi = f.y;
}
template <> __device__ __forceinline__ void widen2<1>(uint32_t w, float& lo, float& hi)
{
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
}

template <int DT> __device__ __forceinline__ float widen1(uint16_t b)
{
    if (DT == 0) return __half2float(__ushort_as_half(b));
    return __uint_as_float((uint32_t)b << 16);
}

template <int DT> __device__ __forceinline__ uint32_t narrow2(float lo, float hi)
{
    if (DT == 0) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}

template <int DT> __device__ __forceinline__ uint16_t narrow1(float x)
{
    if (DT == 0) return __half_as_ushort(__float2half_rn(x));
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// ---- stage 1: fold of the nd ranks' contributions in rank order -----------
template <int DT> __device__ __forceinline__ void add8(float (&s)[8], const uint4 q)
{
    float lo, hi;
    widen2<DT>(q.x, lo, hi); s[0] = __fadd_rn(s[0], lo); s[1] = __fadd_rn(s[1], hi);
    widen2<DT>(q.y, lo, hi); s[2] = __fadd_rn(s[2], lo); s[3] = __fadd_rn(s[3], hi);
    widen2<DT>(q.z, lo, hi); s[4] = __fadd_rn(s[4], lo); s[5] = __fadd_rn(s[5], hi);
    widen2<DT>(q.w, lo, hi); s[6] = __fadd_rn(s[6], lo); s[7] = __fadd_rn(s[7], hi);
}

// s[e] = (((0 + g_0[8vi+e]) + g_1[8vi+e]) + ...) + g_{nd-1}[8vi+e]; the loads of
// a chunk of ranks are issued before its adds so they are in flight together.
// The gradient rows are read-only for the whole step, so they take the
// read-only load path (measured faster than streaming loads for this pass).
template <int DT, int ND>
static __device__ __forceinline__ void fold8(const uint16_t* __restrict__ grads, int64_t rank_stride,
                                      int64_t vi, int nd, float (&s)[8])
{
#pragma unroll
    for (int e = 0; e < 8; e++) s[e] = 0.0f;
    const uint4* base = reinterpret_cast<const uint4*>(grads) + vi;
    const int64_t rsv = rank_stride >> 3;
    if constexpr (ND > 0) {
        constexpr int CH = ND < 16 ? ND : 16;
#pragma unroll
        for (int r0 = 0; r0 < ND; r0 += CH) {
            uint4 q[CH];
#pragma unroll
            for (int c = 0; c < CH; c++) q[c] = __ldg(base + (int64_t)(r0 + c) * rsv);
#pragma unroll
            for (int c = 0; c < CH; c++) add8<DT>(s, q[c]);
        }
    } else {
        for (int r0 = 0; r0 < nd; r0 += 8) {
            uint4 q[8];
#pragma unroll
            for (int c = 0; c < 8; c++)
                if (r0 + c < nd) q[c] = __ldg(base + (int64_t)(r0 + c) * rsv);
#pragma unroll
            for (int c = 0; c < 8; c++)
                if (r0 + c < nd) add8<DT>(s, q[c]);
        }
    }
}

// The same fold over 4 consecutive elements (8-byte loads per rank).
template <int DT>
static __device__ __forceinline__ void add4(float (&s)[4], const uint2 q)
{
    float lo, hi;
    widen2<DT>(q.x, lo, hi); s[0] = __fadd_rn(s[0], lo); s[1] = __fadd_rn(s[1], hi);
    widen2<DT>(q.y, lo, hi); s[2] = __fadd_rn(s[2], lo); s[3] = __fadd_rn(s[3], hi);
}

template <int DT, int ND>
static __device__ __forceinline__ void fold4(const uint16_t* __restrict__ grads, int64_t rank_stride,
                                             int64_t vi, int nd, float (&s)[4])
{
#pragma unroll
    for (int e = 0; e < 4; e++) s[e] = 0.0f;
    const uint2* base = reinterpret_cast<const uint2*>(grads) + vi;
    const int64_t rsv = rank_stride >> 2;
    if constexpr (ND > 0) {
        constexpr int CH = ND < 16 ? ND : 16;
#pragma unroll
        for (int r0 = 0; r0 < ND; r0 += CH) {
            uint2 q[CH];
#pragma unroll
            for (int c = 0; c < CH; c++) q[c] = __ldg(base + (int64_t)(r0 + c) * rsv);
#pragma unroll
            for (int c = 0; c < CH; c++) add4<DT>(s, q[c]);
        }
    } else {
        for (int r0 = 0; r0 < nd; r0 += 8) {
            uint2 q[8];
#pragma unroll
            for (int c = 0; c < 8; c++)
                if (r0 + c < nd) q[c] = __ldg(base + (int64_t)(r0 + c) * rsv);
#pragma unroll
            for (int c = 0; c < 8; c++)
                if (r0 + c < nd) add4<DT>(s, q[c]);
        }
    }
}

template <int DT>
static __device__ __forceinline__ float fold1(const uint16_t* __restrict__ grads, int64_t rank_stride,
                                       int64_t i, int nd)
{
    float s = 0.0f;
    for (int r = 0; r < nd; r++) s = __fadd_rn(s, widen1<DT>(grads[(int64_t)r * rank_stride + i]));
    return s;
}

// ---- stage 2: average and unscale ------------------------------------------
// Division by a power of two and multiplication by its (exact) reciprocal
// round the same real number, so they give identical results; other divisors
// use the correctly rounded division.
struct Unscale {
    float inv_nd, nd_f, inv_s, s;
    bool  nd_pow2, s_pow2;
    __device__ __forceinline__ void init(int nd, float scale)
    {
        nd_f = (float)nd;
        nd_pow2 = (nd & (nd - 1)) == 0;
        inv_nd = nd_pow2 ? __frcp_rn(nd_f) : 0.0f;
        s = scale;
        const uint32_t b = __float_as_uint(scale);
        const uint32_t e = (b >> 23) & 0xFF;
        s_pow2 = (b & 0x807FFFFFu) == 0 && e >= 2 && e <= 252;   // +2^k, 2^-125..2^125
        inv_s = s_pow2 ? __frcp_rn(scale) : 0.0f;
    }
    __device__ __forceinline__ float operator()(float sum) const
    {
        const float avg = nd_pow2 ? __fmul_rn(sum, inv_nd) : __fdiv_rn(sum, nd_f);
        return s_pow2 ? __fmul_rn(avg, inv_s) : __fdiv_rn(avg, s);
    }
};

static __device__ __forceinline__ int not_finite(float x)
{
    return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;
}

// ---- stage 4: Adam / AdamW on one element ------------------------------------
static __device__ __forceinline__ void adam1(float g, float c, float& p, float& m, float& v,
                                      float bc1, float bc2, const AdamK& k)
{
    g = __fmul_rn(g, c);
    if (k.use_wd) {
        if (k.decoupled) p = __fmul_rn(p, k.decay);
        else             g = __fadd_rn(g, __fmul_rn(k.wd, p));
    }
    m = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.omb1, g));
    v = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.omb2, __fmul_rn(g, g)));
    const float mhat = __fdiv_rn(m, bc1);
    const float vhat = __fdiv_rn(v, bc2);
    const float den  = __fadd_rn(__fsqrt_rn(vhat), k.eps);
    p = __fsub_rn(p, __fmul_rn(k.lr, __fdiv_rn(mhat, den)));
}

// ---- deterministic block reductions (fixed shuffle tree) -----------------
static __device__ __forceinline__ double warp_sum(double x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(0xFFFFFFFFu, x, o);
    return x;
}

// Sum over the block; the result is valid in thread 0.
static __device__ __forceinline__ double block_sum(double x, double* sh)
{
    x = warp_sum(x);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) sh[w] = x;
    __syncthreads();
    double r = 0.0;
    if (w == 0) {
        r = (l < (int)(blockDim.x >> 5)) ? sh[l] : 0.0;
        r = warp_sum(r);
    }
    __syncthreads();
    return r;
}

// ---- the norm's sum of squares ---------------------------------------------
// A thread's running sum of squares: an unevaluated pair of binary32 values
// hi + lo, kept normalised by Knuth's two-sum (about 48 significant bits, where
// the norm's tolerance needs 24), plus a binary64 part for the groups whose
// binary32 sum of squares would lose range.  GB300 runs binary64 at a small
// fraction of its binary32 rate, so one binary64 add per 8 elements, and a
// binary64 shuffle tree per block, were a measurable share of a small step.
struct NormAcc {
    float  hi = 0.0f, lo = 0.0f;
    double wide = 0.0;
};

// hi + lo += x, for x >= 0 and hi >= lo >= 0 (every term is a square): the
// two-sum of hi and x, its error folded into lo, renormalised.
static __device__ __forceinline__ void pair_add(float& hi, float& lo, float xh, float xl)
{
    const float s  = __fadd_rn(hi, xh);
    const float bb = __fsub_rn(s, hi);
    float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bb)), __fsub_rn(xh, bb));
    e = __fadd_rn(e, __fadd_rn(lo, xl));
    hi = __fadd_rn(s, e);
    lo = __fsub_rn(e, __fsub_rn(hi, s));
}

// One group of 8: the binary32 FMA chain of its squares, added to the pair, or,
// for groups whose binary32 sum would lose range (very large or very small
// gradients), the exact binary64 chain added to the binary64 part.  An inf or
// NaN takes the binary64 part (inf) or spreads through the pair (NaN), as it
// would through a binary64 sum.
static __device__ __forceinline__ void add_group(NormAcc& acc, const float (&g)[8])
{
    float q = 0.0f;
    int nz = 0;
#pragma unroll
    for (int e = 0; e < 8; e++) {
        q = __fmaf_rn(g[e], g[e], q);
        nz |= (g[e] != 0.0f);
    }
    if ((q > 1.2676506e30f || q < 8.6736174e-19f) && nz) {   // 2^100, 2^-60
        double d = 0.0;
#pragma unroll
        for (int e = 0; e < 8; e++) d = __fma_rn((double)g[e], (double)g[e], d);
        acc.wide = __dadd_rn(acc.wide, d);
    } else {
        pair_add(acc.hi, acc.lo, q, 0.0f);
    }
}

// One element (ragged tails), in the binary64 part.
static __device__ __forceinline__ void add_one(NormAcc& acc, float g)
{
    acc.wide = __fma_rn((double)g, (double)g, acc.wide);
}

struct NormShared {
    float  hi[32], lo[32];
    double wide[32];
    int    last;
};

static __device__ __forceinline__ bool nonzero64(double x)
{
    return (__double_as_longlong(x) << 1) != 0;    // integer test: no binary64 compare
}

static __device__ __forceinline__ void warp_norm(NormAcc& a)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h = __shfl_down_sync(0xFFFFFFFFu, a.hi, o);
        const float l = __shfl_down_sync(0xFFFFFFFFu, a.lo, o);
        pair_add(a.hi, a.lo, h, l);
    }
    if (__any_sync(0xFFFFFFFFu, nonzero64(a.wide))) a.wide = warp_sum(a.wide);
}

// The block's sum of its threads' accumulators (a fixed shuffle tree: the
// pairs always, the binary64 parts when any is non-zero), as one binary64 value
// valid in thread 0.  Any block size up to 1024 threads.
static __device__ __forceinline__ double block_norm(NormAcc a, NormShared& sh)
{
    warp_norm(a);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) {
        sh.hi[w] = a.hi;
        sh.lo[w] = a.lo;
        sh.wide[w] = a.wide;
    }
    __syncthreads();
    double r = 0.0;
    if (w == 0) {
        NormAcc b;
        if (l < (int)(blockDim.x >> 5)) {
            b.hi = sh.hi[l];
            b.lo = sh.lo[l];
            b.wide = sh.wide[l];
        }
        warp_norm(b);
        r = __dadd_rn(__dadd_rn((double)b.hi, (double)b.lo), b.wide);
    }
    __syncthreads();
    return r;
}

static __device__ __forceinline__ int block_or(int f, int* sh)
{
    f = __any_sync(0xFFFFFFFFu, f);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) sh[w] = f;
    __syncthreads();
    int r = 0;
    if (threadIdx.x == 0)
        for (int i = 0; i < (int)(blockDim.x >> 5); i++) r |= sh[i];
    __syncthreads();
    return r;
}

}  // namespace zero
