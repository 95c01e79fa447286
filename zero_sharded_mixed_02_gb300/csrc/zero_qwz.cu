// zero_qwz.cu -- ZeRO++ quantized weight gather (qwZ): block-wise symmetric
// quantization of a rank's 16-bit parameter shard to 8 or 4 bits, and the
// ZeRO-3 unit gather that reads the nd ranks' codes and scales and writes the
// dequantized 16-bit unit.
//
// The block quantizer's arithmetic is in zero_qwz.cuh; the dequantized value is
// the 16-bit rounding of code * scale.
#include <new>

#include "zero_b200.h"
#include "zero_launch.h"
#include "zero_plan_access.h"
#include "zero_qwz.cuh"
#include "zero_trace.h"

namespace zero {

struct GatherQArgs {
    const uint8_t* codes[ZERO_MAX_ND];    // rank k's whole-shard codes
    const float* scales[ZERO_MAX_ND];     // rank k's whole-shard scales
    uint16_t* out;
    int64_t len, slice, offset;
    int nd;
};

// The 16 bytes x[e .. e+8) when all eight lie below n (else zeros: the widening
// step then reads the tail element by element).
static __device__ __forceinline__ uint4 load8_raw(const uint16_t* __restrict__ x, int64_t n, int64_t e)
{
    return e + 8 <= n ? __ldcs(reinterpret_cast<const uint4*>(x + e)) : make_uint4(0, 0, 0, 0);
}

// Eight elements x[e .. e+8) widened to fp32 from their raw 16 bytes q; elements
// at or past n read as 0.
template <int DT>
static __device__ __forceinline__ void widen8(uint4 q, const uint16_t* __restrict__ x, int64_t n,
                                              int64_t e, float* v)
{
    if (e + 8 <= n) {
        widen2<DT>(q.x, v[0], v[1]);
        widen2<DT>(q.y, v[2], v[3]);
        widen2<DT>(q.z, v[4], v[5]);
        widen2<DT>(q.w, v[6], v[7]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; i++) v[i] = e + i < n ? widen1<DT>(x[e + i]) : 0.0f;
    }
}

// One lane's part of a pair: its 16 elements (chunks at e0 and e0 + 128 of block
// blk, raw bytes q0 and q1) quantized and stored, and the block's scale from the
// half-warp's first lane.  FULL: the whole pair lies below n (no bounds checks).
template <int DT, int BITS, bool FULL>
static __device__ __forceinline__ void quantize_pair(uint4 q0, uint4 q1, const uint16_t* __restrict__ x,
                                                     int64_t n, int64_t e0, int64_t blk, int lane,
                                                     uint8_t* __restrict__ codes,
                                                     float* __restrict__ scales)
{
    constexpr int64_t HALF = ZERO_QBLOCK / 2;
    float v[16];
    widen8<DT>(q0, x, FULL ? INT64_MAX : n, e0, v);
    widen8<DT>(q1, x, FULL ? INT64_MAX : n, e0 + HALF, v + 8);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    const float scale = __fdiv_rn(amax, QMax<BITS>::v);
    if ((lane & 15) == 0 && (FULL || blk * ZERO_QBLOCK < n)) scales[blk] = scale;
    uint32_t c[16];
    codes_n<BITS, 16>(v, scale, c);
    if (FULL) {
        store8<BITS>(codes, INT64_MAX, e0, c);
        store8<BITS>(codes, INT64_MAX, e0 + HALF, c + 8);
    } else {
        if (e0 < n) store8<BITS>(codes, n, e0, c);
        if (e0 + HALF < n) store8<BITS>(codes, n, e0 + HALF, c + 8);
    }
}

// Each warp takes two quantization blocks (a pair) at a time, over a persistent
// grid: half-warp h takes block 2p + h of pair p, and its lane j (0..15) the
// 8-element chunks j and j + 16 of that block, so every load and store
// instruction covers two contiguous runs.  The next pair's 32 bytes per lane are
// loaded before the current pair is quantized, so loads overlap arithmetic.
template <int DT, int BITS>
__global__ void __launch_bounds__(ZERO_THREADS, 3) k_quantize(const uint16_t* __restrict__ x,
                                                           int64_t n, uint8_t* __restrict__ codes,
                                                           float* __restrict__ scales)
{
    constexpr int64_t PAIR = 2 * ZERO_QBLOCK;
    const int lane = threadIdx.x & 31;
    const int64_t npairs = (n + PAIR - 1) / PAIR;
    const int64_t stride = (int64_t)gridDim.x * (ZERO_THREADS / 32);
    const int64_t sub = (lane >> 4) * ZERO_QBLOCK + (lane & 15) * 8;   // lane's first element
    int64_t p = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    uint4 nx0 = make_uint4(0, 0, 0, 0), nx1 = nx0;
    if (p < npairs) {
        nx0 = load8_raw(x, n, p * PAIR + sub);
        nx1 = load8_raw(x, n, p * PAIR + sub + ZERO_QBLOCK / 2);
    }
    for (; p < npairs; p += stride) {
        const uint4 q0 = nx0, q1 = nx1;
        const int64_t e0 = p * PAIR + sub;
        if (p + stride < npairs) {                               // prefetch the next pair
            nx0 = load8_raw(x, n, e0 + stride * PAIR);
            nx1 = load8_raw(x, n, e0 + stride * PAIR + ZERO_QBLOCK / 2);
        }
        if ((p + 1) * PAIR <= n)                                  // warp-uniform
            quantize_pair<DT, BITS, true>(q0, q1, x, n, e0, 2 * p + (lane >> 4), lane, codes, scales);
        else
            quantize_pair<DT, BITS, false>(q0, q1, x, n, e0, 2 * p + (lane >> 4), lane, codes, scales);
    }
}

// grid.y = rank k.  A CTA covers QG groups of 8 * ZERO_THREADS consecutive
// outputs of rank k's slice; in group g thread j takes the 8 outputs starting at
// 8 j, so one warp store writes 512 contiguous bytes.  8 outputs never straddle a
// 256-element scale block (unit offsets are multiples of 64).  The thread whose
// 8 outputs run past the valid part takes them element by element.  QG = 2 at 8
// bits and 4 at 4 bits: at 4 bits a group loads only 4 bytes of codes, and two
// groups per thread left too few loads in flight.  The 4-bit decode makes each
// code a float by exponent-field arithmetic rather than an integer conversion
// (measured: 3.46 -> 3.08 ms for LLaMA-3-8B's 34 unit gathers at Nd = 64).
template <int BITS> struct Qg { static constexpr int v = BITS == 8 ? 2 : 4; };

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
    const int k = blockIdx.y;
    const int64_t base = (int64_t)k * a.slice;
    int64_t valid = a.len - base;
    if (valid > a.slice) valid = a.slice;
    if (valid <= 0) return;
    const uint8_t* codes = a.codes[k];
    const float* scales = a.scales[k];
    constexpr int QG = Qg<BITS>::v;
    const int64_t j0 = (int64_t)blockIdx.x * (QG * 8 * ZERO_THREADS) + 8 * threadIdx.x;
    uint32_t word[QG][2];
    float s[QG];
#pragma unroll
    for (int g = 0; g < QG; g++) {                                 // all loads first
        const int64_t j = j0 + g * 8 * ZERO_THREADS;
        if (j + 8 <= valid) {
            const int64_t e = a.offset + j;                        // element of rank k's shard
            s[g] = __ldg(scales + e / ZERO_QBLOCK);
            if (BITS == 8) {
                const uint2 q = __ldcs(reinterpret_cast<const uint2*>(codes + e));
                word[g][0] = q.x;
                word[g][1] = q.y;
            } else {
                word[g][0] = __ldcs(reinterpret_cast<const unsigned int*>(codes + e / 2));
                word[g][1] = 0;
            }
        }
    }
    // keep every load above ahead of the decode below: left to itself the
    // compiler sinks them into the decode loop, and fewer are in flight
    asm volatile("" ::: "memory");
#pragma unroll
    for (int g = 0; g < QG; g++) {
        const int64_t j = j0 + g * 8 * ZERO_THREADS;
        if (j + 8 <= valid) {
            float f[8];
            if (BITS == 8) {
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const int32_t c = (int8_t)(word[g][i / 4] >> (8 * (i % 4)));
                    f[i] = __fmul_rn((float)c, s[g]);
                }
            } else {
                // 4-bit code c (two's complement nibble q): q ^ 8 = c + 8, and the
                // binary32 with exponent field 150 and that value in its mantissa
                // is 2^23 + c + 8 exactly, so one subtraction of 2^23 + 8 gives c
                // as a float without an integer conversion; then the product c *
                // scale, rounded once as before (on packed pairs).
                const f32x2_t bias = pack2(8388616.0f, 8388616.0f), s2 = pack2(s[g], s[g]);
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const uint32_t w = word[g][0] >> (4 * i);
                    const float a0 = __uint_as_float(((w & 0xFu) ^ 8u) | 0x4B000000u);
                    const float a1 = __uint_as_float((((w >> 4) & 0xFu) ^ 8u) | 0x4B000000u);
                    unpack2(mul2(sub2(pack2(a0, a1), bias), s2), f[i], f[i + 1]);
                }
            }
            __stcs(reinterpret_cast<uint4*>(a.out + base + j),
                   make_uint4(narrow2<DT>(f[0], f[1]), narrow2<DT>(f[2], f[3]),
                              narrow2<DT>(f[4], f[5]), narrow2<DT>(f[6], f[7])));
        } else if (j < valid) {
            for (int64_t i = j; i < valid; i++) {
                const int64_t e = a.offset + i;
                a.out[base + i] = narrow1<DT>(__fmul_rn((float)code_at(codes, e, BITS),
                                                        scales[e / ZERO_QBLOCK]));
            }
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
    zero::TraceRange trace_("zero_quantize_shard");
    if ((dtype != ZERO_FP16 && dtype != ZERO_BF16) || (bits != 8 && bits != 4)) return ZERO_EINVAL;
    if (n == 0) return ZERO_OK;
    if (!shard || !codes || !scales || !aligned_to(shard, 16) || !aligned_to(codes, 16) ||
        !aligned_to(scales, 4))
        return ZERO_EINVAL;
    const void* fn = dtype == ZERO_FP16 ? quantize_kernel<0>(bits) : quantize_kernel<1>(bits);
    // persistent grid: every resident CTA, or fewer when there are fewer pairs
    int dev = 0, sms = 1, occ = 1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, ZERO_THREADS, 0) != cudaSuccess)
        return ZERO_ECUDA;
    const uint64_t pairs = (n + 2 * ZERO_QBLOCK - 1) / (2 * ZERO_QBLOCK);
    const uint64_t warps_per_cta = ZERO_THREADS / 32;
    uint64_t grid = (pairs + warps_per_cta - 1) / warps_per_cta;
    const uint64_t resident = (uint64_t)sms * (uint64_t)(occ > 0 ? occ : 1);
    if (grid > resident) grid = resident;
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
    zero::TraceRange trace_("zero_gather_layer_q");
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
        const int64_t per_cta = (int64_t)(bits == 8 ? Qg<8>::v : Qg<4>::v) * 8 * ZERO_THREADS;
        const int64_t bx = ((int64_t)slice + per_cta - 1) / per_cta;
        const void* fn = plan_dtype(plan) == ZERO_FP16 ? gather_q_kernel<0>(bits)
                                                       : gather_q_kernel<1>(bits);
        void* args[] = {a};
        e = cudaLaunchKernel(fn, dim3((unsigned)bx, (unsigned)nd), dim3(ZERO_THREADS), args, 0,
                             static_cast<cudaStream_t>(stream));
    }
    delete a;
    return e == cudaSuccess ? ZERO_OK : ZERO_ECUDA;
}
