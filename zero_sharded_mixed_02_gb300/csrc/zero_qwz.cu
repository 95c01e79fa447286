// zero_qwz.cu -- ZeRO++ quantized weight gather (qwZ): block-wise symmetric
// quantization of a rank's 16-bit parameter shard to 8 or 4 bits, and the
// ZeRO-3 unit gather that reads the nd ranks' codes and scales and writes the
// dequantized 16-bit unit.
//
// Quantization block: ZERO_QBLOCK consecutive elements of a shard, counted from
// the shard's start; scale = max|x| / qmax (qmax = 127 or 7), code =
// round-half-even(x / scale) clamped to [-qmax, qmax] (0 when the scale is 0),
// dequantized value = 16-bit rounding of code * scale.  4-bit codes are packed
// two per byte, the even element in the low nibble.
#include <new>

#include "zero_b200.h"
#include "zero_launch.h"
#include "zero_plan_access.h"

namespace zero {

#define ZERO_QBLOCK 256

struct GatherQArgs {
    const uint8_t* codes[ZERO_MAX_ND];    // rank k's whole-shard codes
    const float* scales[ZERO_MAX_ND];     // rank k's whole-shard scales
    uint16_t* out;
    int64_t len, slice, offset;
    int nd;
};

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

// One warp per quantization block; lane l takes elements 8l .. 8l+7 of it.
template <int DT, int BITS>
__global__ void __launch_bounds__(ZERO_THREADS) k_quantize(const uint16_t* __restrict__ x,
                                                           int64_t n, uint8_t* __restrict__ codes,
                                                           float* __restrict__ scales)
{
    const int lane = threadIdx.x & 31;
    const int64_t blk = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t e0 = blk * ZERO_QBLOCK + lane * 8;
    if (blk * ZERO_QBLOCK >= n) return;                      // whole warp out of range
    float v[8];
    if (e0 + 8 <= n) {
        const uint4 q = __ldcs(reinterpret_cast<const uint4*>(x + e0));
        widen2<DT>(q.x, v[0], v[1]);
        widen2<DT>(q.y, v[2], v[3]);
        widen2<DT>(q.z, v[4], v[5]);
        widen2<DT>(q.w, v[6], v[7]);
    } else {
#pragma unroll
        for (int e = 0; e < 8; e++) v[e] = e0 + e < n ? widen1<DT>(x[e0 + e]) : 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; e++) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float qmax = QMax<BITS>::v;
    const float scale = __fdiv_rn(amax, qmax);
    if (lane == 0) scales[blk] = scale;
    int32_t c[8];
#pragma unroll
    for (int e = 0; e < 8; e++) c[e] = quant1(v[e], scale, qmax);
    if (BITS == 8) {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            lo |= (uint32_t)(uint8_t)(int8_t)c[e] << (8 * e);
            hi |= (uint32_t)(uint8_t)(int8_t)c[4 + e] << (8 * e);
        }
        if (e0 + 8 <= n) {
            *reinterpret_cast<uint2*>(codes + e0) = make_uint2(lo, hi);
        } else {
            for (int e = 0; e < 8 && e0 + e < n; e++) codes[e0 + e] = (uint8_t)(int8_t)c[e];
        }
    } else {
        uint32_t w = 0;
#pragma unroll
        for (int e = 0; e < 8; e++) w |= (uint32_t)(c[e] & 0xF) << (4 * e);
        if (e0 + 8 <= n) {
            *reinterpret_cast<uint32_t*>(codes + e0 / 2) = w;
        } else {
            for (int b = 0; 2 * b < 8 && e0 + 2 * b < n; b++)       // odd tail: high nibble 0
                codes[e0 / 2 + b] = (uint8_t)((w >> (8 * b)) & (e0 + 2 * b + 1 < n ? 0xFF : 0x0F));
        }
    }
}

// grid.y = rank k; one thread per 16 bytes of codes: EPT = 16 (bits 8) or 32
// (bits 4) output elements of rank k's slice, all inside one 256-element scale
// block (unit offsets are multiples of 64).  The thread whose slot runs past the
// valid part takes the tail element by element.
template <int BITS> struct Ept { static constexpr int v = BITS == 8 ? 16 : 32; };

static __device__ __forceinline__ int32_t code_at(const uint8_t* codes, int64_t e, int bits)
{
    if (bits == 8) return (int8_t)codes[e];
    const uint8_t b = codes[e / 2];
    const int32_t c = (e & 1) ? (b >> 4) : (b & 0xF);
    return c >= 8 ? c - 16 : c;
}

template <int DT, int BITS>
__global__ void __launch_bounds__(ZERO_THREADS) k_gather_q(const __grid_constant__ GatherQArgs a)
{
    constexpr int EPT = Ept<BITS>::v;
    const int k = blockIdx.y;
    const int64_t base = (int64_t)k * a.slice;
    int64_t valid = a.len - base;
    if (valid > a.slice) valid = a.slice;
    if (valid <= 0) return;
    const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nvec = valid / EPT;
    const uint8_t* codes = a.codes[k];
    const float* scales = a.scales[k];
    if (w < nvec) {
        const int64_t e = a.offset + w * EPT;                   // element of rank k's shard
        const float s = __ldg(scales + e / ZERO_QBLOCK);
        const uint4 q = __ldcs(reinterpret_cast<const uint4*>(codes + e * BITS / 8));
        const uint32_t word[4] = {q.x, q.y, q.z, q.w};
        uint4* dst = reinterpret_cast<uint4*>(a.out + base + w * EPT);
#pragma unroll
        for (int v = 0; v < EPT / 8; v++) {                       // 8 outputs per 16-byte store
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int idx = v * 8 + j;                        // element within the thread
                int32_t c;
                if (BITS == 8) {
                    c = (int8_t)(word[idx / 4] >> (8 * (idx % 4)));
                } else {
                    c = (int32_t)((word[idx / 8] >> (4 * (idx % 8))) & 0xF);
                    c = c >= 8 ? c - 16 : c;
                }
                f[j] = __fmul_rn((float)c, s);
            }
            __stcs(dst + v, make_uint4(narrow2<DT>(f[0], f[1]), narrow2<DT>(f[2], f[3]),
                                       narrow2<DT>(f[4], f[5]), narrow2<DT>(f[6], f[7])));
        }
    } else if (w == nvec) {
        for (int64_t j = nvec * EPT; j < valid; j++) {
            const int64_t e = a.offset + j;
            a.out[base + j] = narrow1<DT>(__fmul_rn((float)code_at(codes, e, BITS),
                                                    scales[e / ZERO_QBLOCK]));
        }
    }
}

template <int DT>
static const void* quantize_kernel(int bits)
{
    return bits == 8 ? (const void*)k_quantize<DT, 8> : (const void*)k_quantize<DT, 4>;
}

template <int DT>
static const void* gather_q_kernel(int bits)
{
    return bits == 8 ? (const void*)k_gather_q<DT, 8> : (const void*)k_gather_q<DT, 4>;
}

}  // namespace zero

using namespace zero;

namespace {
bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
}  // namespace

extern "C" zero_status_t zero_quantize_shard(zero_dtype_t dtype, const void* shard, uint64_t n,
                                             int bits, void* codes, float* scales, void* stream)
{
    if ((dtype != ZERO_FP16 && dtype != ZERO_BF16) || (bits != 8 && bits != 4)) return ZERO_EINVAL;
    if (n == 0) return ZERO_OK;
    if (!shard || !codes || !scales || !aligned_to(shard, 16) || !aligned_to(codes, 16) ||
        !aligned_to(scales, 4))
        return ZERO_EINVAL;
    const uint64_t nblk = (n + ZERO_QBLOCK - 1) / ZERO_QBLOCK;
    const uint64_t warps_per_cta = ZERO_THREADS / 32;
    const uint64_t grid = (nblk + warps_per_cta - 1) / warps_per_cta;
    if (grid > 0x7FFFFFFFull) return ZERO_EINVAL;
    const void* fn = dtype == ZERO_FP16 ? quantize_kernel<0>(bits) : quantize_kernel<1>(bits);
    const uint16_t* x = static_cast<const uint16_t*>(shard);
    int64_t n64 = (int64_t)n;
    uint8_t* c = static_cast<uint8_t*>(codes);
    void* args[] = {&x, &n64, &c, &scales};
    if (cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(ZERO_THREADS), args, 0,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ZERO_ECUDA;
    return ZERO_OK;
}

extern "C" zero_status_t zero_gather_layer_q(zero_plan_t plan, int unit, int bits,
                                             const void* const* code_ptrs,
                                             const float* const* scale_ptrs, void* out,
                                             void* stream)
{
    if (!plan || plan_stage(plan) != 3 || (bits != 8 && bits != 4)) return ZERO_EINVAL;
    if (plan_poisoned(plan)) return ZERO_ESTATE;
    uint64_t len = 0, slice = 0, off = 0;
    if (zero_plan_unit(plan, unit, &len, &slice, &off) != ZERO_OK) return ZERO_EINVAL;
    if (!code_ptrs || !scale_ptrs || !out || !aligned_to(out, 16)) return ZERO_EINVAL;
    const int nd = plan_nd(plan);
    GatherQArgs* a = new (std::nothrow) GatherQArgs();
    if (!a) return ZERO_ENOMEM;
    for (int k = 0; k < nd; k++) {
        if (!code_ptrs[k] || !scale_ptrs[k] || !aligned_to(code_ptrs[k], 16) ||
            !aligned_to(scale_ptrs[k], 4)) {
            delete a;
            return ZERO_EINVAL;
        }
        a->codes[k] = static_cast<const uint8_t*>(code_ptrs[k]);
        a->scales[k] = scale_ptrs[k];
    }
    a->out = static_cast<uint16_t*>(out);
    a->len = (int64_t)len;
    a->slice = (int64_t)slice;
    a->offset = (int64_t)off;
    a->nd = nd;
    cudaError_t e = cudaSuccess;
    if (len > 0) {
        const int64_t slots = (int64_t)slice / (bits == 8 ? 16 : 32) + 1;
        const int64_t bx = (slots + ZERO_THREADS - 1) / ZERO_THREADS;
        const void* fn = plan_dtype(plan) == ZERO_FP16 ? gather_q_kernel<0>(bits)
                                                       : gather_q_kernel<1>(bits);
        void* args[] = {a};
        e = cudaLaunchKernel(fn, dim3((unsigned)bx, (unsigned)nd), dim3(ZERO_THREADS), args, 0,
                             static_cast<cudaStream_t>(stream));
    }
    delete a;
    return e == cudaSuccess ? ZERO_OK : ZERO_ECUDA;
}
