// zero_noalloc.cu -- zero_grad_norm_noalloc: the global gradient norm and the
// overflow flag of the averaged, unscaled gradient, computed without allocating
// any memory.
//
// Who needs it: code that may not call cudaMalloc -- for example a caller that
// runs inside another framework's memory pool or allocator hooks, where an
// allocation the pool does not know about is forbidden, or a caller that only
// holds pre-allocated device buffers and cannot create a plan (plans allocate
// their device block).  Such a caller passes its gradients and two small output
// buffers it already owns; the scratch this computation needs (one partial sum
// and one flag per tile, and a ticket counter) lives in the file-scope array
// below, which every GPU that loads the library keeps until the process exits.
//
// The computation is the reduce pass of zero_step without the fp32 gradient
// write: fold the nd ranks' 16-bit gradients in rank order, divide by nd and by
// the loss scale, flag any inf/NaN, sum the squares.  Partials are per tile of
// NOALLOC_TILE elements (so the result does not depend on the grid) and are
// combined in tile order by the last block to finish.
#include <mutex>

#include "zero_b200.h"
#include "zero_step_kernels.cuh"

namespace {

constexpr int64_t NOALLOC_TILE = int64_t(1) << 17;         // elements per partial
constexpr int64_t NOALLOC_MAX_TILES = 16384;               // => n <= 2^31 per rank
constexpr size_t OFF_FLAG = NOALLOC_MAX_TILES * sizeof(double);
constexpr size_t OFF_COUNTER = OFF_FLAG + NOALLOC_MAX_TILES * sizeof(int32_t);
constexpr size_t SCRATCH_BYTES = OFF_COUNTER + 256;          // 196,864 bytes

// The scratch.  Host code must not use this name as an address: it is a
// host-side stand-in.  The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SCRATCH_BYTES];

template <int DT>
__global__ void __launch_bounds__(ZERO_THREADS)
k_norm_noalloc(const uint16_t* __restrict__ grads, int nd, int64_t n, int64_t rank_stride,
               float scale, unsigned char* scratch, double* norm_out, int* overflow_out)
{
    using namespace zero;
    __shared__ RedShared sh;
    double* partial = reinterpret_cast<double*>(scratch);
    int32_t* flag = reinterpret_cast<int32_t*>(scratch + OFF_FLAG);
    unsigned int* counter = reinterpret_cast<unsigned int*>(scratch + OFF_COUNTER);
    Unscale un;
    un.init(nd, scale);
    const int64_t ntiles = (n + NOALLOC_TILE - 1) / NOALLOC_TILE;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t lo = tile * NOALLOC_TILE;
        const int64_t hi = lo + NOALLOC_TILE < n ? lo + NOALLOC_TILE : n;
        double acc = 0.0;
        int bad = 0;
        for (int64_t vi = (lo >> 3) + threadIdx.x; vi < (hi >> 3); vi += blockDim.x) {
            float s[8], g[8];
            fold8<DT, 0>(grads, rank_stride, vi, nd, s);
#pragma unroll
            for (int e = 0; e < 8; e++) {
                g[e] = un(s[e]);
                bad |= not_finite(g[e]);
            }
            acc += group_sumsq(g);
        }
        if (hi == n && threadIdx.x < (n & 7)) {                // ragged tail of the last tile
            const float g = un(fold1<DT>(grads, rank_stride, (n & ~int64_t(7)) + threadIdx.x, nd));
            bad |= not_finite(g);
            acc = __fma_rn((double)g, (double)g, acc);
        }
        const double tsum = block_sum(acc, sh.d);
        const int tbad = block_or(bad, sh.i);
        if (threadIdx.x == 0) {
            partial[tile] = tsum;
            flag[tile] = tbad;
        }
    }
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned ticket = atomicAdd(counter, 1u);
        sh.last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (!sh.last) return;
    __threadfence();
    double x = 0.0;
    int f = 0;
    for (int64_t t = threadIdx.x; t < ntiles; t += blockDim.x) {
        x += __ldcg(&partial[t]);
        f |= __ldcg(&flag[t]);
    }
    const double total = block_sum(x, sh.d);
    const int any = block_or(f, sh.i);
    if (threadIdx.x == 0) {
        *norm_out = __dsqrt_rn(total);
        *overflow_out = any;
        *counter = 0;
    }
}

// Device address of the scratch array, looked up once per device context.
// The address belongs to the module loaded in that context: after the device's
// primary context is destroyed and created again (cudaDeviceReset), the module
// is loaded anew and the array may sit elsewhere, so each entry remembers the
// driver's unique id of the context it was looked up in and is refreshed when
// the current context's id differs.
constexpr int MAX_CACHED_DEVICES = 64;
struct ScratchEntry {
    unsigned long long ctx_id = 0;     // 0: unknown (no driver query available)
    void* addr = nullptr;
};
std::mutex g_setup_mutex;
ScratchEntry g_scratch[MAX_CACHED_DEVICES];

using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
bool g_ctx_fns_looked_up = false;

// Unique id of the calling thread's current context, 0 when there is none or
// the driver offers no query (caller holds g_setup_mutex).
unsigned long long current_ctx_id()
{
    if (!g_ctx_fns_looked_up) {
        g_ctx_fns_looked_up = true;
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault,
                                             &q1) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
                cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess) {
            g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f1);
            g_ctx_id = reinterpret_cast<CtxGetIdFn>(f2);
        }
    }
    if (!g_ctx_current || !g_ctx_id) return 0;
    void* ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&ctx) != 0 || ctx == nullptr) return 0;
    if (g_ctx_id(ctx, &id) != 0) return 0;
    return id;
}

cudaError_t scratch_address(int device, unsigned char** out)
{
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    const bool cached = device >= 0 && device < MAX_CACHED_DEVICES;
    const unsigned long long id = current_ctx_id();
    if (cached && g_scratch[device].addr && g_scratch[device].ctx_id == id) {
        *out = static_cast<unsigned char*>(g_scratch[device].addr);
        return cudaSuccess;
    }
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    if (cached) {
        g_scratch[device].ctx_id = current_ctx_id();   // the lookup made the context current
        g_scratch[device].addr = p;
    }
    *out = static_cast<unsigned char*>(p);
    return cudaSuccess;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" zero_status_t zero_grad_norm_noalloc(const void* grads, int nd, uint64_t n,
                                                uint64_t rank_stride, zero_dtype_t dtype,
                                                float loss_scale, double* norm_out,
                                                int* overflow_out, void* stream)
{
    if (nd < 1 || nd > ZERO_MAX_ND || (dtype != ZERO_FP16 && dtype != ZERO_BF16))
        return ZERO_EINVAL;
    if (n > (uint64_t)(NOALLOC_TILE * NOALLOC_MAX_TILES)) return ZERO_EINVAL;  // scratch limit
    if (rank_stride < n || (rank_stride & 7) != 0 || rank_stride > (uint64_t)INT64_MAX / 1024)
        return ZERO_EINVAL;
    if (!(loss_scale > 0.0f) || loss_scale == INFINITY) return ZERO_EINVAL;
    if (!norm_out || !overflow_out || !aligned(norm_out, 8) || !aligned(overflow_out, 4))
        return ZERO_EINVAL;
    if (n > 0 && (!grads || !aligned(grads, 16))) return ZERO_EINVAL;

    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZERO_ECUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ZERO_ECUDA;
    unsigned char* scratch = nullptr;
    if (scratch_address(dev, &scratch) != cudaSuccess) return ZERO_ECUDA;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the ticket counter must start at zero (a failed earlier call may have left it)
    if (cudaMemsetAsync(scratch + OFF_COUNTER, 0, sizeof(unsigned int), s) != cudaSuccess)
        return ZERO_ECUDA;
    const void* fn = dtype == ZERO_FP16 ? (const void*)k_norm_noalloc<0>
                                        : (const void*)k_norm_noalloc<1>;
    int occ = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, ZERO_THREADS, 0) != cudaSuccess ||
        occ < 1)
        occ = 1;
    const int64_t ntiles = ((int64_t)n + NOALLOC_TILE - 1) / NOALLOC_TILE;
    int64_t grid = (int64_t)sms * occ;
    if (grid > ntiles) grid = ntiles;
    if (grid < 1) grid = 1;
    const uint16_t* g16 = static_cast<const uint16_t*>(grads);
    int64_t n64 = (int64_t)n, rs64 = (int64_t)rank_stride;
    void* args[] = {&g16, &nd, &n64, &rs64, &loss_scale, &scratch, &norm_out, &overflow_out};
    if (cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(ZERO_THREADS), args, 0, s) != cudaSuccess)
        return ZERO_ECUDA;
    return ZERO_OK;
}
