// zero_gather.cu -- ZeRO-3 unit gather: nd slices of a unit, one per rank's
// shard, copied into one contiguous buffer in rank order and trimmed to the
// unit length.  Pure data movement: 2 bytes read and 2 written per element.
#include "zero_launch.h"

namespace zero {

// grid.y = rank k; one thread per 8-element (16-byte) vector of rank k's slice,
// no persistent grid (measured faster for this copy, as for the update pass).
// The thread whose vector crosses the end of the valid part copies the tail.
__global__ void __launch_bounds__(ZERO_THREADS) k_gather(const __grid_constant__ GatherArgs a)
{
    const int k = blockIdx.y;
    const int64_t base = (int64_t)k * a.slice;
    int64_t valid = a.len - base;
    if (valid > a.slice) valid = a.slice;
    if (valid <= 0) return;
    const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nvec = valid >> 3;
    if (w < nvec) {
        const uint4 q = __ldcs(reinterpret_cast<const uint4*>(a.src[k]) + w);
        __stcs(reinterpret_cast<uint4*>(a.out + base) + w, q);
    } else if (w == nvec) {
        for (int64_t j = nvec << 3; j < valid; j++) a.out[base + j] = a.src[k][j];
    }
}

cudaError_t launch_gather(const GatherArgs& a, int sms, cudaStream_t stream)
{
    (void)sms;
    const int64_t slots = a.slice / 8 + 1;                // vectors of one slice, plus a tail slot
    const int64_t bx = (slots + ZERO_THREADS - 1) / ZERO_THREADS;
    if (bx > 0x7FFFFFFF || a.nd > 65535) return cudaErrorInvalidValue;
    dim3 grid((unsigned)bx, (unsigned)a.nd);
    k_gather<<<grid, ZERO_THREADS, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace zero
