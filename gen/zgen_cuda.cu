/*
 * zgen_cuda.cu -- CUDA twin of the seeded input generator (definition in
 * zgen.h).  Fills device buffers with the same bits the host version writes;
 * the 16-bit rounding here is CUDA's own nearest-even conversion.
 * Input preparation only: nothing here is part of the optimizer step.
 */
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define G 0x9E3779B97F4A7C15ull

static __host__ __device__ __forceinline__ uint64_t mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t host_key(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank)
{
    uint64_t k = mix(seed ^ ((uint64_t)stream * G));
    k = mix(k + (uint64_t)step * G);
    return mix(k + (uint64_t)rank * G);
}

static __device__ __forceinline__ float sample(uint64_t key, int64_t index, float kappa,
                                               float scale)
{
    uint64_t z = mix(key + ((uint64_t)index + 1u) * G);
    int32_t k = (int32_t)(z & 0xFFFF) + (int32_t)((z >> 16) & 0xFFFF)
              + (int32_t)((z >> 32) & 0xFFFF) + (int32_t)(z >> 48) - 131070;
    return __fmul_rn(__fmul_rn(__int2float_rn(k), kappa), scale);
}

static __device__ __forceinline__ uint16_t round16(int dtype, float v)
{
    return dtype == 0 ? __half_as_ushort(__float2half_rn(v))
                      : __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

struct KeyTable { uint64_t k[128]; };

/* out[r * rank_stride + i]: value of (rank r, index0 + i) for i < n, else 0 */
__global__ void ranks16_kernel(KeyTable keys, int nd, int64_t index0, int64_t n,
                               int64_t rank_stride, float kappa, float scale, int dtype,
                               uint16_t* __restrict__ out)
{
    const int64_t total = (int64_t)nd * rank_stride;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += step) {
        const int64_t r = e / rank_stride;
        const int64_t i = e - r * rank_stride;
        uint16_t b = 0;
        if (i < n) b = round16(dtype, sample(keys.k[r], index0 + i, kappa, scale));
        out[e] = b;
    }
}

__global__ void f32_kernel(uint64_t key, int64_t index0, int64_t n, float kappa, float scale,
                           float* __restrict__ out)
{
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += step)
        out[i] = sample(key, index0 + i, kappa, scale);
}

__global__ void s16_kernel(uint64_t key, int64_t index0, int64_t n, float kappa, float scale,
                           int dtype, uint16_t* __restrict__ out)
{
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += step)
        out[i] = round16(dtype, sample(key, index0 + i, kappa, scale));
}

static int grid_for(int64_t work)
{
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t want = (work + 255) / 256;
    int64_t cap = (int64_t)sms * 8;
    if (want < 1) want = 1;
    return (int)(want < cap ? want : cap);
}

extern "C" {

int zgen_cuda_ranks_16(uint64_t seed, uint32_t stream, uint32_t step, int nd, int64_t index0,
                       int64_t n, int64_t rank_stride, float kappa, float scale, int dtype,
                       void* out, void* cuda_stream)
{
    if (nd < 1 || nd > 128 || n < 0 || rank_stride < n) return (int)cudaErrorInvalidValue;
    KeyTable keys;
    for (int r = 0; r < nd; r++) keys.k[r] = host_key(seed, stream, step, (uint32_t)r);
    ranks16_kernel<<<grid_for((int64_t)nd * rank_stride), 256, 0, (cudaStream_t)cuda_stream>>>(
        keys, nd, index0, n, rank_stride, kappa, scale, dtype, (uint16_t*)out);
    return (int)cudaGetLastError();
}

int zgen_cuda_f32(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank, int64_t index0,
                  int64_t n, float kappa, float scale, void* out, void* cuda_stream)
{
    if (n <= 0) return 0;
    f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
        host_key(seed, stream, step, rank), index0, n, kappa, scale, (float*)out);
    return (int)cudaGetLastError();
}

int zgen_cuda_16(uint64_t seed, uint32_t stream, uint32_t step, uint32_t rank, int64_t index0,
                 int64_t n, float kappa, float scale, int dtype, void* out, void* cuda_stream)
{
    if (n <= 0) return 0;
    s16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
        host_key(seed, stream, step, rank), index0, n, kappa, scale, dtype, (uint16_t*)out);
    return (int)cudaGetLastError();
}

}  /* extern "C" */
