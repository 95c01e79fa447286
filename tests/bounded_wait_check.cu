// bounded_wait_check.cu -- test helper (built by tests/test_gpu_bounded_wait.py):
// one thread waits, through the TMA reduce pass's bounded wait, on an mbarrier
// phase that nothing completes, so the wait must give up on its own, raise the
// abort flag and set the error word, and the kernel must end.
#include <cstdint>

#include "zero_tma.cuh"

namespace {

__global__ void k_wait_on_nothing(int* ret, int32_t* err, long long* cycles, int* abort_seen)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        zero::mbar_init(zero::smem_u32(&bar), 1);     // one arrival expected; none comes
        abort_flag = 0;
        zero::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const long long t0 = clock64();
        *ret = zero::wait_bounded(zero::smem_u32(&bar), 0u, &abort_flag, err);
        *cycles = clock64() - t0;
        *abort_seen = abort_flag;
    }
}

}  // namespace

// Runs the kernel once; returns the CUDA error code of the launch and the sync.
extern "C" int bounded_wait_on_nothing(int* h_ret, int* h_err, long long* h_cycles, int* h_abort)
{
    int* d = nullptr;
    cudaError_t e = cudaMalloc(&d, 4 * sizeof(long long));
    if (e != cudaSuccess) return (int)e;
    e = cudaMemset(d, 0, 4 * sizeof(long long));
    int* ret = d;
    int32_t* err = d + 2;
    long long* cycles = reinterpret_cast<long long*>(d + 4);
    int* abort_seen = d + 6;
    if (e == cudaSuccess) {
        k_wait_on_nothing<<<1, 32>>>(ret, err, cycles, abort_seen);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(h_ret, ret, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(h_err, err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(h_cycles, cycles, sizeof(long long), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(h_abort, abort_seen, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return (int)e;
}
