// zero_offload.cu -- ZeRO-Offload: the reduce on the device, the Adam update on
// the host ([L18] sec. 4.4: the device keeps the 16-bit parameters and
// gradients, the host the fp32 master, m and v and the Adam update; each step
// copies the 16-bit gradients to the host, 2 Psi, and the 16-bit parameters
// back, 2 Psi; [ZL8] sec. 6.2, 7: the host runs the parameter update and
// returns the updated parameters).
//
// Device pass (k_reduce16): the rank-order fp32 fold divided by nd is rounded
// to the 16-bit type (the value the copy carries); the overflow flag and the
// norm are taken from that value divided by the loss scale, and the last block
// settles the step's scalars (skip, clip coefficient, bias corrections), as
// the plain reduce pass does.
//
// Host pipeline: the 16-bit gradient streams to pinned staging in chunks; a
// pool of host threads runs the Adam update on each chunk (zero_cpu_adam.cpp)
// and the chunk's 16-bit parameters stream back, so both copies overlap the
// host arithmetic of the neighbouring chunks.
#include <algorithm>
#include <new>

#include "zero_b200.h"
#include "zero_cpu_adam.h"
#include "zero_launch.h"
#include "zero_plan_access.h"
#include "zero_step_kernels.cuh"
#include "zero_trace.h"

namespace zero {

template <int DT, int ND>
__global__ void __launch_bounds__(ZERO_THREADS, 4) k_reduce16(const StepArgs a,
                                                              uint16_t* __restrict g16)
{
    __shared__ NormShared sh;
    const int nd = ND > 0 ? ND : a.nd;
    Unscale mean, unscale;
    mean.init(nd, 1.0f);                            // fold / nd
    unscale.init(1, a.state->sc.loss_scale);        // copied value / S
    NormAcc acc;
    int bad = 0;
    const int64_t nvec = a.n >> 3;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t vi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; vi < nvec; vi += stride) {
        float s[8], g[8];
        fold8<DT, ND>(a.grads, a.rank_stride, vi, nd, s);
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            w[e] = narrow2<DT>(mean(s[2 * e]), mean(s[2 * e + 1]));
            float lo, hi;
            widen2<DT>(w[e], lo, hi);
            g[2 * e] = unscale(lo);
            g[2 * e + 1] = unscale(hi);
        }
#pragma unroll
        for (int e = 0; e < 8; e++) bad |= not_finite(g[e]);
        add_group(acc, g);
        __stcs(reinterpret_cast<uint4*>(g16) + vi, make_uint4(w[0], w[1], w[2], w[3]));
    }
    if (blockIdx.x == 0 && threadIdx.x < 8) {            // the ragged tail (< 8 elements)
        const int64_t i = (nvec << 3) + threadIdx.x;
        if (i < a.n) {
            const uint16_t q = narrow1<DT>(mean(fold1<DT>(a.grads, a.rank_stride, i, nd)));
            const float g = unscale(widen1<DT>(q));
            bad |= not_finite(g);
            add_one(acc, g);
            g16[i] = q;
        }
    }
    reduce_and_finalize(a, acc, bad, sh);
}

template <int DT>
static const void* reduce16_dt(int nd)
{
    switch (nd) {
    case 1:  return (const void*)k_reduce16<DT, 1>;
    case 2:  return (const void*)k_reduce16<DT, 2>;
    case 4:  return (const void*)k_reduce16<DT, 4>;
    case 8:  return (const void*)k_reduce16<DT, 8>;
    case 16: return (const void*)k_reduce16<DT, 16>;
    case 32: return (const void*)k_reduce16<DT, 32>;
    case 64: return (const void*)k_reduce16<DT, 64>;
    default: return (const void*)k_reduce16<DT, 0>;
    }
}

}  // namespace zero

namespace {

constexpr uint64_t OFFLOAD_CHUNK = 1ull << 24;    // elements per pipelined chunk

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Copies {
    cudaStream_t d2h = nullptr, h2d = nullptr;
    cudaEvent_t ev_d[2] = {nullptr, nullptr}, ev_h[2] = {nullptr, nullptr};
    ~Copies()
    {
        // an early return may leave copies in flight into the plan's staging: let
        // them finish before the next call can reuse it
        if (d2h) cudaStreamSynchronize(d2h);
        if (h2d) cudaStreamSynchronize(h2d);
        for (cudaEvent_t e : ev_d)
            if (e) cudaEventDestroy(e);
        for (cudaEvent_t e : ev_h)
            if (e) cudaEventDestroy(e);
        if (d2h) cudaStreamDestroy(d2h);
        if (h2d) cudaStreamDestroy(h2d);
    }
    bool init()
    {
        if (cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking) != cudaSuccess)
            return false;
        for (int b = 0; b < 2; b++)
            if (cudaEventCreateWithFlags(&ev_d[b], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&ev_h[b], cudaEventDisableTiming) != cudaSuccess)
                return false;
        return true;
    }
};

zero_status_t host_pipeline(zero_plan_t plan, const zero::HostAdamArgs& a, uint64_t n,
                            const uint16_t* g16_dev, float* master, float* m, float* v,
                            uint16_t* params_dev, int nthreads)
{
    void* const* staging = zero::plan_staging(plan, 4, OFFLOAD_CHUNK * 2);
    if (!staging) return ZERO_ENOMEM;
    uint16_t* G[2] = {static_cast<uint16_t*>(staging[0]), static_cast<uint16_t*>(staging[1])};
    uint16_t* P[2] = {static_cast<uint16_t*>(staging[2]), static_cast<uint16_t*>(staging[3])};
    Copies cp;
    if (!cp.init()) return ZERO_ECUDA;
    const uint64_t K = (n + OFFLOAD_CHUNK - 1) / OFFLOAD_CHUNK;
    auto count = [&](uint64_t k) { return std::min(OFFLOAD_CHUNK, n - k * OFFLOAD_CHUNK); };
    auto fetch = [&](uint64_t k) {
        const int b = (int)(k & 1);
        return cudaMemcpyAsync(G[b], g16_dev + k * OFFLOAD_CHUNK, count(k) * 2,
                               cudaMemcpyDeviceToHost, cp.d2h) == cudaSuccess &&
               cudaEventRecord(cp.ev_d[b], cp.d2h) == cudaSuccess;
    };
    if (K > 0 && !fetch(0)) return ZERO_ECUDA;
    if (K > 1 && !fetch(1)) return ZERO_ECUDA;
    zero::HostPool pool(nthreads > 0 ? nthreads : zero::host_threads_default());
    for (uint64_t k = 0; k < K; k++) {
        const int b = (int)(k & 1);
        if (cudaEventSynchronize(cp.ev_d[b]) != cudaSuccess) return ZERO_ECUDA;
        if (k >= 2 && cudaEventSynchronize(cp.ev_h[b]) != cudaSuccess) return ZERO_ECUDA;
        const uint64_t base = k * OFFLOAD_CHUNK, cnt = count(k);
        const int64_t groups = (int64_t)((cnt + 63) / 64);
        pool.run([&](int i, int size) {
            const int64_t lo = std::min<int64_t>((int64_t)cnt, groups * i / size * 64);
            const int64_t hi = std::min<int64_t>((int64_t)cnt, groups * (i + 1) / size * 64);
            if (hi > lo)
                zero::host_adam_range(a, G[b] + lo, master + base + lo, m + base + lo,
                                      v + base + lo, P[b] + lo, hi - lo);
        });
        if (cudaMemcpyAsync(params_dev + base, P[b], cnt * 2, cudaMemcpyHostToDevice, cp.h2d) !=
                cudaSuccess ||
            cudaEventRecord(cp.ev_h[b], cp.h2d) != cudaSuccess)
            return ZERO_ECUDA;
        if (k + 2 < K && !fetch(k + 2)) return ZERO_ECUDA;
    }
    return cudaStreamSynchronize(cp.h2d) == cudaSuccess ? ZERO_OK : ZERO_ECUDA;
}

}  // namespace

extern "C" zero_status_t zero_offload_step(zero_plan_t plan, const void* grads, float* master,
                                           float* m, float* v, void* params, void* workspace,
                                           int nthreads, void* stream)
{
    zero::TraceRange trace_("zero_offload_step");
    if (!plan || zero::plan_stage(plan) > 2) return ZERO_EINVAL;
    if (zero::plan_poisoned(plan)) return ZERO_ESTATE;
    zero::PlanLayout L;
    zero::plan_layout(plan, &L);
    if (L.psi > 0) {
        const void* dev[] = {grads, params, workspace};
        for (const void* p : dev)
            if (!p || !aligned_to(p, 16)) return ZERO_EINVAL;
        const void* host[] = {master, m, v};
        for (const void* p : host)
            if (!p || !aligned_to(p, 4)) return ZERO_EINVAL;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZERO_ECUDA;
    if (dev != L.device) return ZERO_EINVAL;
    const void* fn = L.dtype == ZERO_FP16 ? zero::reduce16_dt<0>(L.nd) : zero::reduce16_dt<1>(L.nd);
    zero_status_t st = zero::plan_launch_reduce16(plan, fn, grads, workspace, stream);
    if (st != ZERO_OK) return st;
    zero::PlanStepStatus ps;
    st = zero::plan_step_status(plan, &ps);                       // waits for the pass
    if (st != ZERO_OK || ps.skipped || L.psi == 0) return st;
    zero_hparams_t hp;
    zero::plan_hparams(plan, &hp);
    zero::HostAdamArgs a;
    a.dtype = L.dtype;
    a.loss_scale = ps.used_scale;
    a.clip_coef = ps.clip_coef;
    a.bc1 = ps.bc1;
    a.bc2 = ps.bc2;
    a.lr = hp.lr;
    a.beta1 = hp.beta1;
    a.beta2 = hp.beta2;
    a.eps = hp.eps;
    a.weight_decay = hp.weight_decay;
    a.decoupled_wd = hp.decoupled_wd;
    try {
        return host_pipeline(plan, a, L.psi, static_cast<const uint16_t*>(workspace), master, m, v,
                             static_cast<uint16_t*>(params), nthreads);
    } catch (...) {                             // host allocation or threads: nothing escapes
        return ZERO_ENOMEM;
    }
}
