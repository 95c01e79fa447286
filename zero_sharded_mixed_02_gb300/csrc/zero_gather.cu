// zero_gather.cu -- ZeRO-3 unit gather: nd slices of a unit, one per rank's
// shard, copied into one contiguous buffer in rank order and trimmed to the
// unit length.  Pure data movement: 2 bytes read and 2 written per element.
#include "zero_launch.h"

namespace zero {

#define GATHER_UNROLL 4

// grid.y = rank k; grid.x blocks stride over rank k's slice in tiles of
// GATHER_UNROLL * blockDim vectors of 8 elements, each load coalesced.
__global__ void __launch_bounds__(ZERO_THREADS) k_gather(const __grid_constant__ GatherArgs a)
{
    const int k = blockIdx.y;
    const int64_t base = (int64_t)k * a.slice;
    int64_t valid = a.len - base;
    if (valid > a.slice) valid = a.slice;
    if (valid <= 0) return;
    const uint4* __restrict__ src = reinterpret_cast<const uint4*>(a.src[k]);
    uint4* __restrict__ dst = reinterpret_cast<uint4*>(a.out + base);
    const int64_t nvec = valid >> 3;
    const int64_t tile = (int64_t)GATHER_UNROLL * blockDim.x;
    for (int64_t t0 = (int64_t)blockIdx.x * tile; t0 < nvec; t0 += (int64_t)gridDim.x * tile) {
        uint4 q[GATHER_UNROLL];
#pragma unroll
        for (int u = 0; u < GATHER_UNROLL; u++) {
            const int64_t w = t0 + (int64_t)u * blockDim.x + threadIdx.x;
            if (w < nvec) q[u] = __ldcs(src + w);
        }
#pragma unroll
        for (int u = 0; u < GATHER_UNROLL; u++) {
            const int64_t w = t0 + (int64_t)u * blockDim.x + threadIdx.x;
            if (w < nvec) __stcs(dst + w, q[u]);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < (valid & 7)) {
        const int64_t j = (nvec << 3) + threadIdx.x;
        a.out[base + j] = a.src[k][j];
    }
}

cudaError_t launch_gather(const GatherArgs& a, int sms, cudaStream_t stream)
{
    const int64_t per_rank_vec = (a.slice + 7) / 8;
    const int64_t tile = (int64_t)GATHER_UNROLL * ZERO_THREADS;
    int64_t bx = (per_rank_vec + tile - 1) / tile;
    const int64_t cap = ((int64_t)sms * 8 + a.nd - 1) / a.nd;
    if (bx > cap) bx = cap;
    if (bx < 1) bx = 1;
    dim3 grid((unsigned)bx, (unsigned)a.nd);
    k_gather<<<grid, ZERO_THREADS, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace zero
