// zero_abi.cu -- plans, validation, kernel dispatch and the extern "C" entry
// points of libzero_b200 (declared and documented in include/zero_b200.h).
#include <algorithm>
#include <array>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "zero_b200.h"
#include "zero_launch.h"
#include "zero_plan_access.h"
#include "zero_trace.h"

using namespace zero;

namespace {

constexpr int PATH_FUSED = 0, PATH_G32 = 1, PATH_RECOMPUTE = 2;
constexpr int PROFILE_RING = 256;
constexpr uint64_t LAYOUT_ALIGN = 64;   // elements; keeps 16-byte vectors inside a shard
constexpr uint64_t REDUCE_WAVES = 12;   // reduce grid: at most this many waves (measured)
constexpr uint64_t FUSED_WAVES = 8;     // fused single-pass grid: at most this many waves
constexpr uint64_t TMA_STAGE_BUDGET = 131072;  // bytes of staged rows per CTA (4 stages at nd 16)
constexpr uint64_t TMA_SMEM_MAX = 196608;      // largest ring of stages a CTA may hold

struct ProfileSlot {
    cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
    bool used = false;
    bool one_kernel = false;        // fused path: the step is the first interval
};

}  // namespace

struct zero_plan {
    uint64_t psi = 0;
    int nd = 1, stage = 0;
    zero_dtype_t dtype = ZERO_FP16;
    zero_hparams_t hp{};
    AdamK k{};
    // stages 0-2
    uint64_t shard = 0, padded = 0;
    // stage 3
    std::vector<uint64_t> unit_len, unit_slice, unit_off;
    uint64_t shard_total = 0;
    // what zero_step runs
    uint64_t n = 0, rank_stride = 0;
    int path = PATH_FUSED;
    const void* fn_a = nullptr;
    const void* fn_b = nullptr;
    int grid_a = 1;
    int block_a = ZERO_THREADS;
    size_t smem_a = 0;              // dynamic shared memory of the reduce pass
    int reduce_kernel = 0;          // 0: 128-bit loads; 1: TMA bulk staging
    int tma_stages = 0;
    uint64_t grid_b = 1;
    uint64_t workspace = 0;
    // ZeRO-3 steps with the qwZ epilogue ([0]: 8 bits, [1]: 4 bits), resolved
    // on first use: the single pass, or the update pass of the two-pass paths
    const void* fn_q[2] = {nullptr, nullptr};
    int grid_q[2] = {1, 1};
    // ping-pong steps, resolved on first use: the single pass and its repair pass
    const void* fn_pp = nullptr;
    const void* fn_pp_repair = nullptr;
    int grid_pp = 1;
    // device
    int device = 0, sms = 1;
    DevState* d_state = nullptr;
    DevScalars* h_mirror = nullptr;     // pinned: DevScalars followed by DevStatus
    cudaEvent_t ev_done = nullptr;
    cudaStream_t copy_stream = nullptr;
    bool stepped = false;
    // diagnostics
    bool profile = false;
    std::vector<ProfileSlot> ring;
    int ring_pos = 0;
    double ms_a = 0.0, ms_b = 0.0;
    int64_t prof_steps = 0;
    int64_t launches = 0;
    // bucketed steps (constant-size gradient buckets)
    uint64_t bucket_elems = 0, nbuckets = 0, bucket_ws = 0;
    int bucket_grid = 0, bucket_last_grid = 0;   // reduce blocks of a full / the last bucket
    std::vector<uint8_t> bucket_seen;
    const void* fn_bucket_reduce = nullptr;
    const void* fn_bucket_final = nullptr;
    const void* fn_bucket_update = nullptr;
    // checkpoints
    uint64_t model_hash = 0;          // FNV-1a 64 of the tensor shape list
    bool poisoned = false;            // a failed load left the state half-written
    std::vector<void*> staging;       // pinned host staging for checkpoint IO
    uint64_t staging_bytes = 0;
};

namespace {

uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }
uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite_f(float x) { return std::isfinite(x); }

zero_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? ZERO_OK : ZERO_ECUDA; }

// 1 - beta^(t+1) from beta^t, as the device's step bookkeeping computes it: one
// binary64 product, one binary64 difference, one rounding to binary32 (the
// volatile keeps the host compiler from fusing the two into one rounding).
float next_bias_correction(double beta_pow, float beta)
{
    volatile double prod = beta_pow * (double)beta;
    return (float)(1.0 - prod);
}

zero_status_t check_hparams(const zero_hparams_t& h, zero_dtype_t dtype)
{
    if (!finite_f(h.lr) || !finite_f(h.eps) || h.eps < 0.0f) return ZERO_EINVAL;
    if (!(h.beta1 >= 0.0f && h.beta1 < 1.0f) || !(h.beta2 >= 0.0f && h.beta2 < 1.0f))
        return ZERO_EINVAL;
    if (!finite_f(h.weight_decay) || !finite_f(h.clip_norm) || h.clip_norm < 0.0f)
        return ZERO_EINVAL;
    if (!finite_f(h.loss_scale) || !(h.loss_scale > 0.0f)) return ZERO_EINVAL;
    if (h.dynamic_scale) {
        if (dtype != ZERO_FP16) return ZERO_EINVAL;
        if (!(h.backoff > 0.0f && h.backoff <= 1.0f)) return ZERO_EINVAL;
    }
    return ZERO_OK;
}

void destroy_plan(zero_plan* p)
{
    if (!p) return;
    for (auto& s : p->ring)
        for (auto& e : s.ev)
            if (e) cudaEventDestroy(e);
    if (p->d_state) cudaFree(p->d_state);
    if (p->h_mirror) cudaFreeHost(p->h_mirror);
    if (p->ev_done) cudaEventDestroy(p->ev_done);
    if (p->copy_stream) cudaStreamDestroy(p->copy_stream);
    for (void* b : p->staging) cudaFreeHost(b);
    delete p;
}

// Reduce and fused passes: a whole number of waves of (SMs x resident blocks per
// SM), at most max_waves, and no more waves than leave every thread at least
// MIN_VECTORS_PER_THREAD of its 8-element vectors; capped by the work (one
// thread per vector) and by the per-block partials array.  Measured on the
// fused pass: more waves are faster while a thread keeps about six vectors or
// more (2^26-2^31 elements: 8 waves, 0.94-1.07 of the copy rate, against
// 0.89-1.05 for 1-3), and slower below that (2^24 elements: 2 waves, 0.85-1.02,
// against 0.74-0.97 for 8, where a thread has two or three vectors and the
// last round runs a third full).
constexpr uint64_t MIN_VECTORS_PER_THREAD = 6;
int grid_reduce(const void* fn, int sms, uint64_t n, uint64_t max_waves)
{
    int occ = 1;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, ZERO_THREADS, 0) != cudaSuccess ||
        occ < 1)
        occ = 1;
    const uint64_t nvec = n / 8;
    const uint64_t per_wave = (uint64_t)sms * (uint64_t)occ;
    const uint64_t waves = std::min<uint64_t>(
        max_waves, std::max<uint64_t>(1, nvec / (per_wave * ZERO_THREADS * MIN_VECTORS_PER_THREAD)));
    const uint64_t want = std::max<uint64_t>(1, ceil_div(nvec, ZERO_THREADS));
    uint64_t g = std::min<uint64_t>(per_wave * waves, want);
    g = std::min<uint64_t>(g, ZERO_MAX_BLOCKS);
    return (int)std::max<uint64_t>(g, 1);
}

// Update pass: one thread per 4 elements (the last slot may be partial).
uint64_t grid_update(uint64_t n)
{
    return std::max<uint64_t>(1, ceil_div(ceil_div(n, 4), ZERO_THREADS));
}

// FNV-1a 64 over the little-endian bytes of the int64 sequence ntensors,
// then for each tensor its ndims and its dims: the identity of a model's
// parameter list, stored in checkpoints.
uint64_t shape_hash(const int64_t* dims, const int* ndims, int ntensors)
{
    uint64_t h = 0xCBF29CE484222325ull;
    auto put = [&h](int64_t x) {
        for (int b = 0; b < 8; b++) {
            h ^= (uint64_t)((uint64_t)x >> (8 * b)) & 0xFFu;
            h *= 0x100000001B3ull;
        }
    };
    put(ntensors);
    size_t di = 0;
    for (int t = 0; t < ntensors; t++) {
        put(ndims[t]);
        for (int d = 0; d < ndims[t]; d++) put(dims[di++]);
    }
    return h;
}

zero_status_t create_impl(uint64_t psi, int nd, int stage, zero_dtype_t dtype,
                          const int64_t* dims, const int* ndims, int ntensors,
                          const int* unit_of_tensor, const zero_hparams_t* hp, zero_plan_t* out)
{
    if (!out || !hp) return ZERO_EINVAL;
    *out = nullptr;
    if (nd < 1 || nd > ZERO_MAX_ND || stage < 0 || stage > 3) return ZERO_EINVAL;
    if (dtype != ZERO_FP16 && dtype != ZERO_BF16) return ZERO_EINVAL;
    if (ntensors < 0 || (ntensors > 0 && (!dims || !ndims))) return ZERO_EINVAL;
    zero_status_t s = check_hparams(*hp, dtype);
    if (s != ZERO_OK) return s;

    // tensor sizes; their sum must be psi
    std::vector<uint64_t> tlen((size_t)ntensors);
    uint64_t total = 0;
    size_t di = 0;
    for (int t = 0; t < ntensors; t++) {
        if (ndims[t] < 0 || ndims[t] > 16) return ZERO_EINVAL;
        uint64_t len = 1;
        for (int d = 0; d < ndims[t]; d++) {
            const int64_t x = dims[di++];
            if (x < 0) return ZERO_EINVAL;
            if (x != 0 && len > UINT64_MAX / (uint64_t)x) return ZERO_EINVAL;
            len *= (uint64_t)x;
        }
        tlen[(size_t)t] = len;
        if (total > UINT64_MAX - len) return ZERO_EINVAL;
        total += len;
    }
    if (total != psi || psi > ZERO_MAX_PSI) return ZERO_EINVAL;

    zero_plan* p = new (std::nothrow) zero_plan();
    if (!p) return ZERO_ENOMEM;
    p->model_hash = shape_hash(dims, ndims, ntensors);
    p->psi = psi;
    p->nd = nd;
    p->stage = stage;
    p->dtype = dtype;
    p->hp = *hp;

    if (stage <= 2) {
        p->shard = round_up(ceil_div(psi, (uint64_t)nd), LAYOUT_ALIGN);
        p->padded = p->shard * (uint64_t)nd;
        p->n = psi;
        p->rank_stride = p->padded;
    } else {
        // units: given, or one per tensor; each unit's tensors contiguous
        int nunits = 0;
        std::vector<uint64_t> ulen;
        for (int t = 0; t < ntensors; t++) {
            const int u = unit_of_tensor ? unit_of_tensor[t] : t;
            if (u == nunits) {
                ulen.push_back(0);
                nunits++;
            } else if (u != nunits - 1) {
                destroy_plan(p);
                return ZERO_EINVAL;
            }
            ulen.back() += tlen[(size_t)t];
        }
        uint64_t off = 0;
        for (int u = 0; u < nunits; u++) {
            const uint64_t sl = round_up(ceil_div(ulen[(size_t)u], (uint64_t)nd), LAYOUT_ALIGN);
            p->unit_len.push_back(ulen[(size_t)u]);
            p->unit_slice.push_back(sl);
            p->unit_off.push_back(off);
            off += sl;
        }
        p->shard_total = off;
        p->shard = off;
        p->padded = off;
        p->n = off;
        p->rank_stride = off;
    }

    // Adam constants: 1 - beta1, 1 - beta2 and 1 - lr*wd in double, rounded once
    p->k.lr = hp->lr;
    p->k.b1 = hp->beta1;
    p->k.b2 = hp->beta2;
    p->k.eps = hp->eps;
    p->k.wd = hp->weight_decay;
    p->k.omb1 = (float)(1.0 - (double)hp->beta1);
    p->k.omb2 = (float)(1.0 - (double)hp->beta2);
    p->k.decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
    p->k.decoupled = hp->decoupled_wd ? 1 : 0;
    p->k.use_wd = hp->weight_decay != 0.0f;

    // kernel path
    // anything that must be known before the first update forces two passes
    const bool needs_global = hp->clip_norm > 0.0f || hp->dynamic_scale || hp->skip_on_overflow;
    int kind_a, kind_b = -1;
    if (!needs_global) {
        p->path = PATH_FUSED;
        kind_a = K_FUSED;
    } else if (nd >= 4) {
        p->path = PATH_G32;
        kind_a = K_REDUCE_G32;
        kind_b = K_UPDATE_G32;
        p->workspace = round_up(p->n * sizeof(float), 256);
    } else {
        p->path = PATH_RECOMPUTE;
        kind_a = K_REDUCE_ONLY;
        kind_b = K_UPDATE_RECOMPUTE;
    }
    p->fn_a = step_kernel((int)dtype, kind_a, nd);
    p->fn_b = kind_b >= 0 ? step_kernel((int)dtype, kind_b, nd) : nullptr;
    if (!p->fn_a || (kind_b >= 0 && !p->fn_b)) {
        destroy_plan(p);
        return ZERO_EINVAL;
    }

    // device resources
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&p->sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) {
        destroy_plan(p);
        return ZERO_ECUDA;
    }
    p->grid_a = grid_reduce(p->fn_a, p->sms, p->n,
                            p->path == PATH_FUSED ? FUSED_WAVES : REDUCE_WAVES);
    p->grid_b = grid_update(p->n);
    if (p->grid_b > 0x7FFFFFFFull) {
        destroy_plan(p);
        return ZERO_EINVAL;
    }

    if (cudaMalloc(&p->d_state, sizeof(DevState)) != cudaSuccess ||
        cudaMallocHost(&p->h_mirror, sizeof(DevScalars) + sizeof(DevStatus)) != cudaSuccess) {
        destroy_plan(p);
        return ZERO_ENOMEM;
    }
    DevState* init = new (std::nothrow) DevState();
    if (!init) {
        destroy_plan(p);
        return ZERO_ENOMEM;
    }
    std::memset(init, 0, sizeof(DevState));
    init->sc.loss_scale = hp->loss_scale;
    init->sc.good_steps = 0;
    init->sc.t = 0;
    init->sc.beta1_pow = 1.0;
    init->sc.beta2_pow = 1.0;
    init->sc.bc1_next = next_bias_correction(1.0, hp->beta1);
    init->sc.bc2_next = next_bias_correction(1.0, hp->beta2);
    init->st.clip_coef = 1.0f;
    init->st.used_scale = hp->loss_scale;
    e = cudaMemcpy(p->d_state, init, sizeof(DevState), cudaMemcpyHostToDevice);
    std::memcpy(p->h_mirror, &init->sc, sizeof(DevScalars));
    std::memcpy(reinterpret_cast<char*>(p->h_mirror) + sizeof(DevScalars), &init->st,
                sizeof(DevStatus));
    delete init;
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->copy_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
        destroy_plan(p);
        return ZERO_ECUDA;
    }
    *out = p;
    return ZERO_OK;
}

void harvest(zero_plan* p, ProfileSlot& s)
{
    if (!s.used) return;
    float a = 0.0f, b = 0.0f;
    if (cudaEventSynchronize(s.ev[2]) == cudaSuccess &&
        cudaEventElapsedTime(&a, s.ev[0], s.ev[1]) == cudaSuccess &&
        (s.one_kernel || cudaEventElapsedTime(&b, s.ev[1], s.ev[2]) == cudaSuccess)) {
        p->ms_a += a;
        p->ms_b += b;
        p->prof_steps += 1;
    }
    s.used = false;
}

zero_status_t fetch_mirror(zero_plan* p)
{
    if (!p->stepped) return ZERO_OK;
    cudaError_t e = cudaEventSynchronize(p->ev_done);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(p->h_mirror, p->d_state, sizeof(DevScalars) + sizeof(DevStatus),
                            cudaMemcpyDeviceToHost, p->copy_stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->copy_stream);
    return cuda_status(e);
}

StepArgs step_args(const zero_plan* plan, const void* grads, float* master, float* m, float* v,
                   void* params, void* workspace)
{
    StepArgs a;
    a.grads = static_cast<const uint16_t*>(grads);
    a.master = master;
    a.m = m;
    a.v = v;
    a.params = static_cast<uint16_t*>(params);
    a.g32 = static_cast<float*>(workspace);
    a.n = (int64_t)plan->n;
    a.rank_stride = (int64_t)plan->rank_stride;
    a.nd = plan->nd;
    a.k = plan->k;
    a.clip = plan->hp.clip_norm;
    a.dynamic = plan->hp.dynamic_scale ? 1 : 0;
    a.skip_static = plan->hp.skip_on_overflow ? 1 : 0;
    a.backoff = plan->hp.backoff;
    a.growth_interval = plan->hp.growth_interval;
    a.state = plan->d_state;
    return a;
}

}  // namespace

namespace zero {
int plan_nd(zero_plan_t plan) { return plan->nd; }
int plan_stage(zero_plan_t plan) { return plan->stage; }
int plan_dtype(zero_plan_t plan) { return (int)plan->dtype; }

void plan_layout(zero_plan_t plan, PlanLayout* out)
{
    out->psi = plan->psi;
    out->nd = plan->nd;
    out->stage = plan->stage;
    out->dtype = (int)plan->dtype;
    out->device = plan->device;
    out->shard = plan->stage <= 2 ? plan->shard : plan->shard_total;
    out->model_hash = plan->model_hash;
    out->unit_len = plan->unit_len;
    out->unit_slice = plan->unit_slice;
    out->unit_off = plan->unit_off;
}

zero_status_t plan_scalars_get(zero_plan_t plan, PlanScalars* out)
{
    const zero_status_t s = fetch_mirror(plan);
    if (s != ZERO_OK) return s;
    const DevScalars* sc = plan->h_mirror;
    out->loss_scale = sc->loss_scale;
    out->good_steps = sc->good_steps;
    out->t = sc->t;
    out->beta1_pow = sc->beta1_pow;
    out->beta2_pow = sc->beta2_pow;
    return ZERO_OK;
}

zero_status_t plan_scalars_set(zero_plan_t plan, const PlanScalars& in)
{
    if (plan->stepped && cudaEventSynchronize(plan->ev_done) != cudaSuccess) return ZERO_ECUDA;
    DevScalars sc{};
    sc.loss_scale = in.loss_scale;
    sc.good_steps = in.good_steps;
    sc.t = in.t;
    sc.beta1_pow = in.beta1_pow;
    sc.beta2_pow = in.beta2_pow;
    sc.bc1_next = next_bias_correction(in.beta1_pow, plan->hp.beta1);
    sc.bc2_next = next_bias_correction(in.beta2_pow, plan->hp.beta2);
    sc.cur = 0;                         // a restored state is the ping-pong set 0
    DevStatus st{};
    st.clip_coef = 1.0f;
    st.used_scale = in.loss_scale;
    std::memcpy(plan->h_mirror, &sc, sizeof(DevScalars));
    std::memcpy(reinterpret_cast<char*>(plan->h_mirror) + sizeof(DevScalars), &st,
                sizeof(DevStatus));
    // DevState starts with the scalars and the status, in this order
    cudaError_t e = cudaMemcpyAsync(plan->d_state, plan->h_mirror,
                                    sizeof(DevScalars) + sizeof(DevStatus),
                                    cudaMemcpyHostToDevice, plan->copy_stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(plan->copy_stream);
    if (e != cudaSuccess) return ZERO_ECUDA;
    plan->stepped = false;
    std::fill(plan->bucket_seen.begin(), plan->bucket_seen.end(), 0);
    return ZERO_OK;
}

zero_status_t plan_step_status(zero_plan_t plan, PlanStepStatus* out)
{
    const zero_status_t s = fetch_mirror(plan);
    if (s != ZERO_OK) return s;
    const DevStatus* st = reinterpret_cast<const DevStatus*>(
        reinterpret_cast<const char*>(plan->h_mirror) + sizeof(DevScalars));
    out->skipped = st->skipped;
    out->overflow = st->overflow;
    out->grad_norm = st->grad_norm;
    out->clip_coef = st->clip_coef;
    out->bc1 = st->bc1;
    out->bc2 = st->bc2;
    out->used_scale = st->used_scale;
    return st->err ? ZERO_ETIMEOUT : ZERO_OK;
}

void plan_hparams(zero_plan_t plan, zero_hparams_t* out) { *out = plan->hp; }

zero_status_t plan_launch_reduce16(zero_plan_t plan, const void* fn, const void* grads, void* g16,
                                   void* stream)
{
    if (!fn) return ZERO_EINVAL;
    StepArgs a = step_args(plan, grads, nullptr, nullptr, nullptr, nullptr, nullptr);
    const int grid = grid_reduce(fn, plan->sms, plan->n, REDUCE_WAVES);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* args[] = {&a, &g16};
    if (cudaLaunchKernel(fn, dim3(grid), dim3(ZERO_THREADS), args, 0, s) != cudaSuccess)
        return ZERO_ECUDA;
    plan->launches++;
    if (cudaEventRecord(plan->ev_done, s) != cudaSuccess) return ZERO_ECUDA;
    plan->stepped = true;
    return ZERO_OK;
}

void plan_set_poisoned(zero_plan_t plan, bool poisoned) { plan->poisoned = poisoned; }
bool plan_poisoned(zero_plan_t plan) { return plan->poisoned; }

void* const* plan_staging(zero_plan_t plan, int count, uint64_t bytes)
{
    if ((int)plan->staging.size() >= count && plan->staging_bytes >= bytes)
        return plan->staging.data();
    for (void* b : plan->staging) cudaFreeHost(b);
    plan->staging.clear();
    plan->staging_bytes = 0;
    for (int i = 0; i < count; i++) {
        void* b = nullptr;
        if (cudaHostAlloc(&b, bytes, cudaHostAllocDefault) != cudaSuccess) {
            for (void* q : plan->staging) cudaFreeHost(q);
            plan->staging.clear();
            return nullptr;
        }
        plan->staging.push_back(b);
    }
    plan->staging_bytes = bytes;
    return plan->staging.data();
}

const void* step_kernel(int dtype, int kind, int nd)
{
    if (kind >= K_FUSED_Q8)
        return dtype == 0 ? step_kernel_q_fp16(kind, nd) : step_kernel_q_bf16(kind, nd);
    return dtype == 0 ? step_kernel_fp16(kind, nd) : step_kernel_bf16(kind, nd);
}
}  // namespace zero

extern "C" {

zero_status_t zero_plan_create(uint64_t psi, int nd, int stage, zero_dtype_t dtype,
                               const int64_t* dims, const int* ndims, int ntensors,
                               const zero_hparams_t* hp, zero_plan_t* out)
{
    try {
        return create_impl(psi, nd, stage, dtype, dims, ndims, ntensors, nullptr, hp, out);
    } catch (...) {                             // host allocation failed: nothing escapes the ABI
        return ZERO_ENOMEM;
    }
}

zero_status_t zero_plan_create_units(uint64_t psi, int nd, int stage, zero_dtype_t dtype,
                                     const int64_t* dims, const int* ndims, int ntensors,
                                     const int* unit_of_tensor, const zero_hparams_t* hp,
                                     zero_plan_t* out)
{
    if (stage == 3 && ntensors > 0 && !unit_of_tensor) return ZERO_EINVAL;
    try {
        return create_impl(psi, nd, stage, dtype, dims, ndims, ntensors, unit_of_tensor, hp, out);
    } catch (...) {
        return ZERO_ENOMEM;
    }
}

zero_status_t zero_plan_destroy(zero_plan_t plan)
{
    if (plan && plan->stepped) cudaEventSynchronize(plan->ev_done);
    destroy_plan(plan);
    return ZERO_OK;
}

zero_status_t zero_plan_layout(zero_plan_t plan, uint64_t* shard_elems, uint64_t* padded_elems,
                               int* nunits, uint64_t* workspace_bytes)
{
    if (!plan) return ZERO_EINVAL;
    if (shard_elems) *shard_elems = plan->shard;
    if (padded_elems) *padded_elems = plan->padded;
    if (nunits) *nunits = plan->stage == 3 ? (int)plan->unit_len.size() : 0;
    if (workspace_bytes) *workspace_bytes = plan->workspace;
    return ZERO_OK;
}

zero_status_t zero_plan_unit(zero_plan_t plan, int unit, uint64_t* len, uint64_t* slice_elems,
                             uint64_t* offset)
{
    if (!plan || plan->stage != 3 || unit < 0 || unit >= (int)plan->unit_len.size())
        return ZERO_EINVAL;
    if (len) *len = plan->unit_len[(size_t)unit];
    if (slice_elems) *slice_elems = plan->unit_slice[(size_t)unit];
    if (offset) *offset = plan->unit_off[(size_t)unit];
    return ZERO_OK;
}

int zero_plan_path(zero_plan_t plan) { return plan ? plan->path : -1; }

zero_status_t zero_plan_set_bucket(zero_plan_t plan, uint64_t bucket_elems,
                                   uint64_t* workspace_bytes)
{
    if (!plan) return ZERO_EINVAL;
    if (plan->stepped && cudaEventSynchronize(plan->ev_done) != cudaSuccess) return ZERO_ECUDA;
    if (bucket_elems == 0) {
        plan->bucket_elems = plan->nbuckets = plan->bucket_ws = 0;
        plan->bucket_grid = plan->bucket_last_grid = 0;
        plan->bucket_seen.clear();
        if (workspace_bytes) *workspace_bytes = 0;
        return ZERO_OK;
    }
    if (bucket_elems % LAYOUT_ALIGN != 0) return ZERO_EINVAL;
    const uint64_t nb = ceil_div(plan->n, bucket_elems);
    if (nb > (1ull << 24)) return ZERO_EINVAL;
    const void* red = step_kernel((int)plan->dtype, K_REDUCE_G32, plan->nd);
    if (!red) red = step_kernel((int)plan->dtype, K_REDUCE_G32, 0);   // generic rank count
    const void* fin = step_kernel((int)plan->dtype, K_BUCKET_FINALIZE, 0);
    const void* upd = step_kernel((int)plan->dtype, K_UPDATE_G32, plan->nd);
    if (!red || !fin || !upd) return ZERO_EINVAL;
    // each bucket's reduce grid (a full bucket's, and the last bucket's) and its
    // per-block partial slots
    const int grid = grid_reduce(red, plan->sms, bucket_elems, REDUCE_WAVES);
    const int last = grid_reduce(red, plan->sms, plan->n - (nb - 1) * bucket_elems, REDUCE_WAVES);
    plan->bucket_elems = bucket_elems;
    plan->nbuckets = nb;
    plan->bucket_grid = grid;
    plan->bucket_last_grid = last;
    plan->bucket_ws = round_up(plan->n * sizeof(float), 256) +
                      round_up(nb * (uint64_t)grid * sizeof(double), 256) +
                      round_up(nb * (uint64_t)grid * sizeof(int32_t), 256);
    try {
        plan->bucket_seen.assign((size_t)nb, 0);
    } catch (...) {
        plan->bucket_elems = plan->nbuckets = plan->bucket_ws = 0;
        return ZERO_ENOMEM;
    }
    plan->fn_bucket_reduce = red;
    plan->fn_bucket_final = fin;
    plan->fn_bucket_update = upd;
    if (workspace_bytes) *workspace_bytes = plan->bucket_ws;
    return ZERO_OK;
}

namespace {
// The bucketed step's workspace: the fp32 reduced gradient [n], then every
// bucket's per-block squared-norm partials [nb][grid] and overflow flags [nb][grid].
void bucket_pointers(const zero_plan* plan, void* workspace, float** g32, double** partial,
                     int32_t** flag)
{
    char* w = static_cast<char*>(workspace);
    *g32 = reinterpret_cast<float*>(w);
    w += round_up(plan->n * sizeof(float), 256);
    *partial = reinterpret_cast<double*>(w);
    w += round_up(plan->nbuckets * (uint64_t)plan->bucket_grid * sizeof(double), 256);
    *flag = reinterpret_cast<int32_t*>(w);
}
}  // namespace

zero_status_t zero_step_bucket(zero_plan_t plan, uint64_t bucket, const void* bucket_grads,
                               void* workspace, void* stream)
{
    zero::TraceRange trace_("zero_step_bucket");
    if (!plan || plan->bucket_elems == 0 || bucket >= plan->nbuckets) return ZERO_EINVAL;
    if (plan->poisoned) return ZERO_ESTATE;
    if (!bucket_grads || !aligned16(bucket_grads) || !workspace || !aligned16(workspace))
        return ZERO_EINVAL;
    if (plan->bucket_seen[(size_t)bucket]) return ZERO_EINVAL;        // once per step
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZERO_ECUDA;
    if (dev != plan->device) return ZERO_EINVAL;
    const uint64_t first = bucket * plan->bucket_elems;
    const uint64_t count = std::min(plan->bucket_elems, plan->n - first);
    float* g32;
    double* partial;
    int32_t* flag;
    bucket_pointers(plan, workspace, &g32, &partial, &flag);
    StepArgs a = step_args(plan, bucket_grads, nullptr, nullptr, nullptr, nullptr, g32 + first);
    a.n = (int64_t)count;
    a.rank_stride = (int64_t)plan->bucket_elems;
    a.bucket = (int)bucket;
    a.bucket_partial = partial + bucket * (uint64_t)plan->bucket_grid;
    a.bucket_flag = flag + bucket * (uint64_t)plan->bucket_grid;
    void* args[] = {&a};
    const int grid = bucket == plan->nbuckets - 1 ? plan->bucket_last_grid : plan->bucket_grid;
    // A programmatic dependent launch: the blocks may be placed while the previous
    // grid on the stream finishes; the kernel waits (griddepcontrol.wait) for that
    // grid's completion before its first read, so this is safe whatever that grid
    // was (the previous bucket, or a kernel of the caller's that wrote this
    // bucket's gradients).  Measured: bucketed GPT-2 1.5B steps at B = 2^23,
    // 16.15 -> 15.75 ms.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(ZERO_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelExC(&cfg, plan->fn_bucket_reduce, args) != cudaSuccess)
        return ZERO_ECUDA;
    plan->launches++;
    plan->bucket_seen[(size_t)bucket] = 1;
    return ZERO_OK;
}

zero_status_t zero_step_apply(zero_plan_t plan, float* master, float* m, float* v, void* params,
                              void* workspace, void* stream)
{
    zero::TraceRange trace_("zero_step_apply");
    if (!plan || plan->bucket_elems == 0) return ZERO_EINVAL;
    if (plan->poisoned) return ZERO_ESTATE;
    for (uint8_t seen : plan->bucket_seen)
        if (!seen) return ZERO_EINVAL;                                 // a bucket is missing
    if (plan->n > 0) {
        const void* ptrs[] = {master, m, v, params, workspace};
        for (const void* q : ptrs)
            if (!q || !aligned16(q)) return ZERO_EINVAL;
    }
    float* g32;
    double* partial;
    int32_t* flag;
    bucket_pointers(plan, workspace, &g32, &partial, &flag);
    StepArgs a = step_args(plan, nullptr, master, m, v, params, g32);
    a.bucket_partial = partial;
    a.bucket_flag = flag;
    int nb = (int)plan->nbuckets, grid = plan->bucket_grid, last = plan->bucket_last_grid;
    const unsigned fblocks = (unsigned)std::min<uint64_t>(
        std::min<uint64_t>(plan->nbuckets, 4ull * (uint64_t)plan->sms), ZERO_MAX_BLOCKS);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void* fargs[] = {&a, &nb, &grid, &last};
    if (cudaLaunchKernel(plan->fn_bucket_final, dim3(fblocks), dim3(ZERO_THREADS), fargs, 0, s) !=
        cudaSuccess)
        return ZERO_ECUDA;
    void* uargs[] = {&a};
    if (cudaLaunchKernel(plan->fn_bucket_update, dim3((unsigned)plan->grid_b), dim3(ZERO_THREADS),
                         uargs, 0, s) != cudaSuccess)
        return ZERO_ECUDA;
    plan->launches += 2;
    if (cudaEventRecord(plan->ev_done, s) != cudaSuccess) return ZERO_ECUDA;
    plan->stepped = true;
    std::fill(plan->bucket_seen.begin(), plan->bucket_seen.end(), 0);
    return ZERO_OK;
}

zero_status_t zero_plan_set_reduce_kernel(zero_plan_t plan, int kind)
{
    if (!plan || (kind != 0 && kind != 1)) return ZERO_EINVAL;
    if (plan->stepped && cudaEventSynchronize(plan->ev_done) != cudaSuccess) return ZERO_ECUDA;
    if (kind == 0) {
        plan->fn_a = step_kernel((int)plan->dtype, plan->path == PATH_FUSED ? K_FUSED
                                 : plan->path == PATH_G32 ? K_REDUCE_G32 : K_REDUCE_ONLY,
                                 plan->nd);
        plan->grid_a = grid_reduce(plan->fn_a, plan->sms, plan->n,
                                   plan->path == PATH_FUSED ? FUSED_WAVES : REDUCE_WAVES);
        plan->block_a = ZERO_THREADS;
        plan->smem_a = 0;
        plan->tma_stages = 0;
        plan->reduce_kernel = 0;
        return ZERO_OK;
    }
    // TMA staging: the two-pass path, with a ring of at least two stages of
    // nd rows x 2 KB that fits in one CTA's shared memory
    const uint64_t stage = (uint64_t)plan->nd * 2 * 1024;
    if (plan->path != PATH_G32 || 2 * stage > TMA_SMEM_MAX) return ZERO_EINVAL;
    // the same rule as tma_stages_for(): ~128 KB of rows, 2..8 stages
    uint64_t stages = std::max<uint64_t>(2, TMA_STAGE_BUDGET / stage);
    stages = std::min<uint64_t>(stages, 8);
    const void* fn = step_kernel((int)plan->dtype, K_REDUCE_G32_TMA, plan->nd);
    if (!fn) return ZERO_EINVAL;
    const size_t smem = (size_t)(stages * stage);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return ZERO_ECUDA;
    plan->fn_a = fn;
    plan->grid_a = std::min(plan->sms, ZERO_MAX_BLOCKS);
    plan->block_a = 288;
    plan->smem_a = smem;
    plan->tma_stages = (int)stages;
    plan->reduce_kernel = 1;
    return ZERO_OK;
}

}  // extern "C"

namespace {

// Validation shared by zero_step and zero_step_qwz.
zero_status_t check_step_args(const zero_plan* plan, const void* grads, float* master, float* m,
                              float* v, void* params, void* workspace, bool uses_workspace = true)
{
    if (plan->poisoned) return ZERO_ESTATE;
    if (plan->n > 0) {
        const void* ptrs[] = {grads, master, m, v, params};
        for (const void* q : ptrs)
            if (!q || !aligned16(q)) return ZERO_EINVAL;
    }
    if (uses_workspace && plan->path == PATH_G32 && plan->n > 0 &&
        (!workspace || !aligned16(workspace)))
        return ZERO_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZERO_ECUDA;
    if (dev != plan->device) return ZERO_EINVAL;
    return ZERO_OK;
}

// The step's launch sequence: pass 1 (fn_a; the fused pass, or the reduce pass
// in the plan's configured form), then, when fn_b is given, pass 2 (fn_b, grid_b
// blocks) as its programmatic dependent; per-kernel events when profiling; the
// step's completion event.
zero_status_t launch_step(zero_plan* plan, StepArgs& a, const void* fn_a, int grid_a,
                          const void* fn_b, uint64_t grid_b, cudaStream_t s)
{
    ProfileSlot* slot = nullptr;
    if (plan->profile) {
        slot = &plan->ring[(size_t)(plan->ring_pos % PROFILE_RING)];
        harvest(plan, *slot);
        plan->ring_pos++;
        if (cudaEventRecord(slot->ev[0], s) != cudaSuccess) return ZERO_ECUDA;
    }
    const bool tma = plan->reduce_kernel && fn_a == plan->fn_a;
    int stages = plan->tma_stages;
    void* args_tma[] = {&a, &stages};
    void* args[] = {&a};
    cudaError_t e = cudaLaunchKernel(fn_a, dim3(grid_a), dim3(tma ? plan->block_a : ZERO_THREADS),
                                     tma ? args_tma : args, tma ? plan->smem_a : 0, s);
    if (e != cudaSuccess) return ZERO_ECUDA;
    plan->launches++;
    if (slot && cudaEventRecord(slot->ev[1], s) != cudaSuccess) return ZERO_ECUDA;
    if (fn_b) {
        // a programmatic dependent of pass 1: scheduled while pass 1 finishes, it
        // waits (griddepcontrol.wait) before reading what pass 1 wrote
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid_b);
        cfg.blockDim = dim3(ZERO_THREADS);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelExC(&cfg, fn_b, args);
        if (e != cudaSuccess) return ZERO_ECUDA;
        plan->launches++;
    }
    if (slot) {
        if (cudaEventRecord(slot->ev[2], s) != cudaSuccess) return ZERO_ECUDA;
        slot->used = true;
        slot->one_kernel = !fn_b;
    }
    if (cudaEventRecord(plan->ev_done, s) != cudaSuccess) return ZERO_ECUDA;
    plan->stepped = true;
    return ZERO_OK;
}

}  // namespace

extern "C" {

zero_status_t zero_step(zero_plan_t plan, const void* grads, float* master, float* m, float* v,
                        void* params, void* workspace, void* stream)
{
    zero::TraceRange trace_("zero_step");
    if (!plan) return ZERO_EINVAL;
    const zero_status_t st = check_step_args(plan, grads, master, m, v, params, workspace);
    if (st != ZERO_OK) return st;
    StepArgs a = step_args(plan, grads, master, m, v, params, workspace);
    return launch_step(plan, a, plan->fn_a, plan->grid_a, plan->fn_b, plan->grid_b,
                       static_cast<cudaStream_t>(stream));
}

zero_status_t zero_step_qwz(zero_plan_t plan, const void* grads, float* master, float* m,
                            float* v, void* params, void* workspace, int bits, void* codes,
                            float* scales, void* stream)
{
    zero::TraceRange trace_("zero_step_qwz");
    if (!plan || plan->stage != 3 || (bits != 8 && bits != 4)) return ZERO_EINVAL;
    const zero_status_t st = check_step_args(plan, grads, master, m, v, params, workspace);
    if (st != ZERO_OK) return st;
    if (plan->n > 0 && (!codes || !scales || !aligned16(codes) ||
                        (reinterpret_cast<uintptr_t>(scales) & 3u) != 0))
        return ZERO_EINVAL;
    const int q = bits == 8 ? 0 : 1;
    if (!plan->fn_q[q]) {
        const int kind = plan->path == PATH_FUSED ? (q ? K_FUSED_Q4 : K_FUSED_Q8)
                         : plan->path == PATH_G32 ? (q ? K_UPDATE_G32_Q4 : K_UPDATE_G32_Q8)
                                                  : (q ? K_UPDATE_RECOMPUTE_Q4
                                                       : K_UPDATE_RECOMPUTE_Q8);
        const void* fn = step_kernel((int)plan->dtype, kind, plan->nd);
        if (!fn) return ZERO_EINVAL;
        plan->grid_q[q] = plan->path == PATH_FUSED
                              ? grid_reduce(fn, plan->sms, plan->n, FUSED_WAVES) : 0;
        plan->fn_q[q] = fn;
    }
    StepArgs a = step_args(plan, grads, master, m, v, params, workspace);
    a.qcodes = static_cast<uint8_t*>(codes);
    a.qscales = scales;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan->path == PATH_FUSED)
        return launch_step(plan, a, plan->fn_q[q], plan->grid_q[q], nullptr, 0, s);
    return launch_step(plan, a, plan->fn_a, plan->grid_a, plan->fn_q[q], plan->grid_b, s);
}

zero_status_t zero_step_pingpong(zero_plan_t plan, const void* grads, float* master0, float* m0,
                                 float* v0, float* master1, float* m1, float* v1, void* params,
                                 void* stream)
{
    zero::TraceRange trace_("zero_step_pingpong");
    if (!plan || plan->hp.clip_norm > 0.0f) return ZERO_EINVAL;   // a clip gates the update
    const zero_status_t st = check_step_args(plan, grads, master0, m0, v0, params, nullptr, false);
    if (st != ZERO_OK) return st;
    if (plan->n > 0) {
        const void* ptrs[] = {master1, m1, v1};
        for (const void* q : ptrs)
            if (!q || !aligned16(q)) return ZERO_EINVAL;
    }
    if (!plan->fn_pp) {
        const void* fn = step_kernel((int)plan->dtype, K_FUSED_PP, plan->nd);
        const void* rep = step_kernel((int)plan->dtype, K_PP_REPAIR, 0);
        if (!fn || !rep) return ZERO_EINVAL;
        plan->grid_pp = grid_reduce(fn, plan->sms, plan->n, FUSED_WAVES);
        plan->fn_pp = fn;
        plan->fn_pp_repair = rep;
    }
    StepArgs a = step_args(plan, grads, master0, m0, v0, params, nullptr);
    a.master2 = master1;
    a.m2 = m1;
    a.v2 = v1;
    a.pingpong = 1;
    // the repair pass: one thread per 4 elements, like the update pass
    return launch_step(plan, a, plan->fn_pp, plan->grid_pp, plan->fn_pp_repair, plan->grid_b,
                       static_cast<cudaStream_t>(stream));
}

zero_status_t zero_plan_state_set(zero_plan_t plan, int* set)
{
    if (!plan || !set) return ZERO_EINVAL;
    const zero_status_t s = fetch_mirror(plan);
    if (s != ZERO_OK) return s;
    *set = plan->h_mirror->cur;
    return ZERO_OK;
}

zero_status_t zero_step_result(zero_plan_t plan, int* skipped, double* grad_norm,
                               float* clip_coef, float* loss_scale, int64_t* t)
{
    if (!plan) return ZERO_EINVAL;
    zero_status_t s = fetch_mirror(plan);
    if (s != ZERO_OK) return s;
    const DevScalars* sc = plan->h_mirror;
    const DevStatus* st = reinterpret_cast<const DevStatus*>(
        reinterpret_cast<const char*>(plan->h_mirror) + sizeof(DevScalars));
    if (skipped) *skipped = st->skipped;
    if (grad_norm) *grad_norm = st->grad_norm;
    if (clip_coef) *clip_coef = st->clip_coef;
    if (loss_scale) *loss_scale = sc->loss_scale;
    if (t) *t = sc->t;
    return st->err ? ZERO_ETIMEOUT : ZERO_OK;
}

zero_status_t zero_step_overflow(zero_plan_t plan, int* overflow)
{
    if (!plan || !overflow) return ZERO_EINVAL;
    zero_status_t s = fetch_mirror(plan);
    if (s != ZERO_OK) return s;
    const DevStatus* st = reinterpret_cast<const DevStatus*>(
        reinterpret_cast<const char*>(plan->h_mirror) + sizeof(DevScalars));
    *overflow = st->overflow;
    return ZERO_OK;
}

zero_status_t zero_gather_layer(zero_plan_t plan, int unit, const void* const* shard_ptrs,
                                void* out, void* stream)
{
    zero::TraceRange trace_("zero_gather_layer");
    if (!plan || plan->stage != 3 || unit < 0 || unit >= (int)plan->unit_len.size())
        return ZERO_EINVAL;
    if (plan->poisoned) return ZERO_ESTATE;
    if (!shard_ptrs || !out || !aligned16(out)) return ZERO_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZERO_ECUDA;
    if (dev != plan->device) return ZERO_EINVAL;
    GatherArgs* a = new (std::nothrow) GatherArgs();
    if (!a) return ZERO_ENOMEM;
    const uint64_t off = plan->unit_off[(size_t)unit];
    for (int k = 0; k < plan->nd; k++) {
        const uint16_t* b = static_cast<const uint16_t*>(shard_ptrs[k]);
        if (!b || !aligned16(b)) {
            delete a;
            return ZERO_EINVAL;
        }
        a->src[k] = b + off;
    }
    a->out = static_cast<uint16_t*>(out);
    a->len = (int64_t)plan->unit_len[(size_t)unit];
    a->slice = (int64_t)plan->unit_slice[(size_t)unit];
    a->nd = plan->nd;
    cudaError_t e = cudaSuccess;
    if (a->len > 0) {
        e = launch_gather(*a, plan->sms, static_cast<cudaStream_t>(stream));
        if (e == cudaSuccess) plan->launches++;
    }
    delete a;
    return cuda_status(e);
}

uint64_t zero_state_bytes(uint64_t psi, uint64_t nd, int stage, int K)
{
    if (nd == 0 || K < 0) return 0;
    using u128 = unsigned __int128;
    const u128 P = psi, N = nd, k = (u128)K;
    u128 r;
    switch (stage) {
    case 0: r = (4 + k) * P; break;
    case 1: r = 4 * P + (k * P + N - 1) / N; break;
    case 2: r = 2 * P + ((2 + k) * P + N - 1) / N; break;
    case 3: r = ((4 + k) * P + N - 1) / N; break;
    default: return 0;
    }
    return r > (u128)UINT64_MAX ? UINT64_MAX : (uint64_t)r;
}

uint64_t zero_comm_volume(uint64_t psi, uint64_t nd, int stage, int exact)
{
    if (nd == 0 || stage < 0 || stage > 3) return 0;
    using u128 = unsigned __int128;
    const u128 v = (u128)(stage == 3 ? 3 : 2) * psi;
    const u128 r = exact ? (v * (nd - 1) + nd - 1) / nd : v;
    return r > (u128)UINT64_MAX ? UINT64_MAX : (uint64_t)r;
}

uint64_t zero_max_params(uint64_t mem_bytes, uint64_t nd, int stage, int K)
{
    if (nd == 0 || K < 0) return 0;
    using u128 = unsigned __int128;
    const u128 M = mem_bytes, N = nd, k = (u128)K;
    u128 r;
    switch (stage) {
    case 0: r = M / (4 + k); break;
    case 1: r = M * N / (4 * N + k); break;
    case 2: r = M * N / (2 * N + 2 + k); break;
    case 3: r = M * N / (4 + k); break;
    default: return 0;
    }
    return r > (u128)UINT64_MAX ? UINT64_MAX : (uint64_t)r;
}

const char* zero_status_string(zero_status_t status)
{
    switch (status) {
    case ZERO_OK: return "ZERO_OK";
    case ZERO_EINVAL: return "ZERO_EINVAL: invalid argument";
    case ZERO_ENOMEM: return "ZERO_ENOMEM: allocation failed";
    case ZERO_ECUDA: return "ZERO_ECUDA: CUDA call failed";
    case ZERO_ETIMEOUT: return "ZERO_ETIMEOUT: bounded device wait gave up";
    case ZERO_ENOENT: return "ZERO_ENOENT: a checkpoint file is missing";
    case ZERO_ECORRUPT: return "ZERO_ECORRUPT: a checkpoint file is damaged or does not belong";
    case ZERO_EIO: return "ZERO_EIO: reading or writing a file failed";
    case ZERO_ESTATE: return "ZERO_ESTATE: a failed checkpoint load left the state incomplete";
    default: return "unknown zero_status_t";
    }
}

zero_status_t zero_plan_profile(zero_plan_t plan, int enable)
{
    if (!plan) return ZERO_EINVAL;
    if (!enable) {
        plan->profile = false;
        return ZERO_OK;
    }
    if (plan->ring.empty()) {
        try {
            plan->ring.resize(PROFILE_RING);
        } catch (...) {
            return ZERO_ENOMEM;
        }
        for (auto& s : plan->ring)
            for (auto& e : s.ev)
                if (cudaEventCreate(&e) != cudaSuccess) {   // undo: no half-made ring is kept
                    for (auto& s2 : plan->ring)
                        for (auto& e2 : s2.ev)
                            if (e2) cudaEventDestroy(e2);
                    plan->ring.clear();
                    return ZERO_ECUDA;
                }
    }
    for (auto& s : plan->ring) {
        if (s.used) cudaEventSynchronize(s.ev[2]);
        s.used = false;
    }
    plan->ms_a = plan->ms_b = 0.0;
    plan->prof_steps = 0;
    plan->ring_pos = 0;
    plan->profile = true;
    return ZERO_OK;
}

zero_status_t zero_plan_kernel_times(zero_plan_t plan, double* reduce_ms, double* update_ms,
                                     int64_t* steps, int64_t* launches)
{
    if (!plan) return ZERO_EINVAL;
    if (!plan->ring.empty()) {
        const int start = plan->ring_pos;
        for (int i = 0; i < PROFILE_RING; i++)
            harvest(plan, plan->ring[(size_t)((start + i) % PROFILE_RING)]);
    }
    if (reduce_ms) *reduce_ms = plan->ms_a;
    if (update_ms) *update_ms = plan->ms_b;
    if (steps) *steps = plan->prof_steps;
    if (launches) *launches = plan->launches;
    return ZERO_OK;
}

}  // extern "C"
