// zero_tma.cuh -- the reduce pass with TMA bulk staging of the rank-strided
// gradient rows.
//
// One producer warp issues cp.async.bulk copies of the nd ranks' rows of a
// 1024-element tile into a ring of shared-memory stages, completing an mbarrier
// by transaction count; eight consumer warps fold the staged rows in rank order,
// release the stage through a second mbarrier, and write the fp32 gradient.
// Every wait is bounded: after WAIT_LIMIT polls the block raises a shared abort
// flag and the sticky error bit of the step status; once every warp has stopped,
// the producer lets the block's copies still in flight land (again bounded), and
// the block finishes without further work (the host sees ZERO_ETIMEOUT).
#pragma once

#include "zero_step_kernels.cuh"

namespace zero {

#define ZERO_TMA_TILE 1024            // elements per tile (4 per consumer thread)
#define ZERO_TMA_MAX_STAGES 8
#define ZERO_TMA_THREADS 288          // 8 consumer warps + 1 producer warp
#ifndef ZERO_TMA_WAIT_LIMIT                  // polls before a wait gives up
#define ZERO_TMA_WAIT_LIMIT (1u << 20)
#endif

static __device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}
static __device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
static __device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
static __device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
static __device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}
// 1-D bulk copy global -> shared, completing `bar` by its byte count.  Source and
// destination 16-byte aligned, size a multiple of 16.
static __device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                                uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
static __device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Bounded wait; 0 when the phase completed, 1 when the block gave up.
static __device__ __forceinline__ int wait_bounded(uint32_t bar, uint32_t parity,
                                                   volatile int* abort_flag, int32_t* err)
{
    for (uint32_t it = 0; it < ZERO_TMA_WAIT_LIMIT; it++) {
        if (mbar_try_wait(bar, parity)) return 0;
        if (*abort_flag) return 1;
    }
    *abort_flag = 1;
    atomicOr(err, 1);
    return 1;
}

struct TmaShared {
    uint64_t full[ZERO_TMA_MAX_STAGES];
    uint64_t empty[ZERO_TMA_MAX_STAGES];
    NormShared norm;
    int abort_flag;
};

// Stage count for nd rank rows of 2 KB: about 128 KB of staged rows, 2..8 stages.
__host__ __device__ constexpr int tma_stages_for(int nd)
{
    return nd <= 0 ? 2 : (131072 / (nd * 2048) < 2 ? 2 : (131072 / (nd * 2048) > 8 ? 8 : 131072 / (nd * 2048)));
}

// Pass 1 with TMA staging (writes the fp32 gradient).  ND > 0: compile-time rank
// count; ND = 0: runtime nd (a.nd) with `stages` stages.  Dynamic shared memory:
// stages * nd * 2 * ZERO_TMA_TILE bytes.  Grid: persistent, static tile order;
// the stage index and its phase advance incrementally (no division per tile).
template <int DT, int ND>
__global__ void __launch_bounds__(ZERO_TMA_THREADS, 1) k_reduce_tma(const StepArgs a, int stages_rt)
{
    extern __shared__ __align__(128) unsigned char stage_mem[];
    __shared__ TmaShared sh;
    const int nd = ND > 0 ? ND : a.nd;
    const int stages = ND > 0 ? tma_stages_for(ND) : stages_rt;
    const uint32_t ROW = ZERO_TMA_TILE * 2, STAGE = (uint32_t)nd * ROW;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Unscale un;
    un.init(nd, a.state->sc.loss_scale);
    const int64_t ntiles = a.n / ZERO_TMA_TILE;
    const int64_t my = ntiles > blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int64_t tile_step = (int64_t)gridDim.x * ZERO_TMA_TILE;
    int32_t* err = &a.state->st.err;
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; s++) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), 8);
        }
        sh.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    NormAcc acc;
    int bad = 0;
    int64_t issued = 0;                                     // tiles the producer issued
    if (warp == 8) {                                        // producer
        if (lane == 0) {
            int64_t j = 0, base = (int64_t)blockIdx.x * ZERO_TMA_TILE;
            int s = 0;
            uint32_t ph = 0;                                // phase of this round of stages
            for (; j < my; j++, base += tile_step) {
                if (j >= stages &&
                    wait_bounded(smem_u32(&sh.empty[s]), ph ^ 1u, &sh.abort_flag, err))
                    break;
                const uint32_t sb = smem_u32(stage_mem + (size_t)s * STAGE);
                const uint32_t bar = smem_u32(&sh.full[s]);
                mbar_expect_tx(bar, STAGE);
#pragma unroll
                for (int r = 0; r < (ND > 0 ? ND : 1); r++) {
                    if (ND > 0) bulk_g2s(sb + r * ROW, a.grads + (int64_t)r * a.rank_stride + base, ROW, bar);
                }
                if (ND == 0)
                    for (int r = 0; r < nd; r++)
                        bulk_g2s(sb + r * ROW, a.grads + (int64_t)r * a.rank_stride + base, ROW, bar);
                if (++s == stages) { s = 0; ph ^= 1u; }
            }
            issued = j;
        }
    } else {                                                // consumers: elements 4t..4t+3
        const int t = threadIdx.x;
        int s = 0;
        uint32_t ph = 0;
        int64_t base = (int64_t)blockIdx.x * ZERO_TMA_TILE;
        for (int64_t j = 0; j < my; j++, base += tile_step) {
            if (wait_bounded(smem_u32(&sh.full[s]), ph, &sh.abort_flag, err)) break;
            const unsigned char* sb = stage_mem + (size_t)s * STAGE;
            float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if constexpr (ND > 0) {
                constexpr int CH = ND < 16 ? ND : 16;
#pragma unroll
                for (int r0 = 0; r0 < ND; r0 += CH) {
                    uint2 q[CH];
#pragma unroll
                    for (int c = 0; c < CH; c++)
                        q[c] = reinterpret_cast<const uint2*>(sb + (r0 + c) * ROW)[t];
#pragma unroll
                    for (int c = 0; c < CH; c++) add4<DT>(s4, q[c]);
                }
            } else {
                for (int r0 = 0; r0 < nd; r0 += 8) {
                    uint2 q[8];
#pragma unroll
                    for (int c = 0; c < 8; c++)
                        if (r0 + c < nd) q[c] = reinterpret_cast<const uint2*>(sb + (r0 + c) * ROW)[t];
#pragma unroll
                    for (int c = 0; c < 8; c++)
                        if (r0 + c < nd) add4<DT>(s4, q[c]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.empty[s]));
            if (++s == stages) { s = 0; ph ^= 1u; }
            float g[8];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                g[e] = un(s4[e]);
                bad |= not_finite(g[e]);
                g[4 + e] = 0.0f;
            }
            add_group(acc, g);
            __stcs(reinterpret_cast<float4*>(a.g32 + base) + t, make_float4(g[0], g[1], g[2], g[3]));
        }
        if (blockIdx.x == gridDim.x - 1 && !*(volatile int*)&sh.abort_flag) {   // ragged remainder
            for (int64_t i = ntiles * ZERO_TMA_TILE + t; i < a.n; i += 256) {
                const float g = un(fold1<DT>(a.grads, a.rank_stride, i, nd));
                bad |= not_finite(g);
                add_one(acc, g);
                a.g32[i] = g;
            }
        }
    }
    // Every consumer has left its loop, so the abort flag is final.  After an
    // abort, whichever side gave up and however the producer's loop ended, only
    // the last `stages` issued tiles can still have copies in flight (an earlier
    // tile's stage was reissued only after its consumers released it, which
    // needs its copies complete): wait, bounded, for those to land before the
    // block reuses or releases its shared memory.
    __syncthreads();
    if (warp == 8 && lane == 0 && *(volatile int*)&sh.abort_flag)
        for (int64_t k = (issued > stages ? issued - stages : 0); k < issued; k++)
            for (uint32_t it = 0; it < ZERO_TMA_WAIT_LIMIT &&
                                  !mbar_try_wait(smem_u32(&sh.full[k % stages]),
                                                 (uint32_t)((k / stages) & 1));
                 it++) {
            }
    reduce_and_finalize(a, acc, bad, sh.norm);
}

}  // namespace zero
