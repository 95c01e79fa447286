// zero_step_kernels.cuh -- the optimizer-step kernels (templates).
//
// Reduce and fused passes: a grid of ZERO_THREADS-thread blocks, a few waves of
// the SM count times the kernel's occupancy, sized once per plan.  Thread t of
// block b handles the 8-element vectors b*T + t, b*T + t + G*T, ... (static
// assignment), so the per-block sums of squares and their fixed-order
// combination are the same on every run.  The last block to finish (an atomic
// ticket, no waiting) combines the per-block partials in block order and
// writes the step status.  The update pass uses one thread per 4 elements.
// The sums of squares are kept as binary32 pairs up to each block's partial
// (NormAcc, zero_common.cuh); the partials and their combination are binary64.
#pragma once

#include "zero_common.cuh"
#include "zero_qwz.cuh"

namespace zero {

// Norm partial of one group of 8 for the no-allocation norm: an FMA chain in
// binary32, moved to binary64 per group.  Groups whose binary32 sum of squares
// would lose range (very large or very small gradients) are summed exactly in
// binary64 instead.
static __device__ __forceinline__ double group_sumsq(const float (&g)[8])
{
    float q = 0.0f;
    int nz = 0;
#pragma unroll
    for (int e = 0; e < 8; e++) {
        q = __fmaf_rn(g[e], g[e], q);
        nz |= (g[e] != 0.0f);
    }
    if ((q > 1.2676506e30f || q < 8.6736174e-19f) && nz) {   // 2^100, 2^-60
        double d = 0.0;
#pragma unroll
        for (int e = 0; e < 8; e++) d = __fma_rn((double)g[e], (double)g[e], d);
        return d;
    }
    return (double)q;
}

// Scalar bookkeeping of the step (thread 0 of the last block): global norm,
// clip coefficient, skip decision, loss-scale backoff/growth, t and the bias
// corrections.  sc and err: the step's scalars and sticky error word.  Binary64
// operations are IEEE round-to-nearest.
static __device__ __noinline__ void finalize(const StepArgs& a, DevScalars sc, int32_t err,
                                             double sumsq, int overflow)
{
    DevState* S = a.state;
    DevStatus st;
    st.overflow   = overflow;
    st.used_scale = sc.loss_scale;
    st.grad_norm  = __dsqrt_rn(sumsq);
    st.clip_coef  = (a.clip > 0.0f && st.grad_norm > (double)a.clip)
                        ? __double2float_rn(__ddiv_rn((double)a.clip, st.grad_norm)) : 1.0f;
    st.err = err;              // sticky: a bounded wait that gave up, in any step
    st.pad = 0;
    if (overflow && (a.dynamic || a.skip_static)) {
        st.skipped = 1;
        if (a.dynamic) {                       // only a dynamic scale backs off
            sc.loss_scale = __fmul_rn(sc.loss_scale, a.backoff);
            sc.good_steps = 0;
        }
        st.bc1 = st.bc2 = 0.0f;
    } else {
        st.skipped = 0;
        sc.t += 1;
        sc.beta1_pow = __dmul_rn(sc.beta1_pow, (double)a.k.b1);
        sc.beta2_pow = __dmul_rn(sc.beta2_pow, (double)a.k.b2);
        st.bc1 = __double2float_rn(__dsub_rn(1.0, sc.beta1_pow));
        st.bc2 = __double2float_rn(__dsub_rn(1.0, sc.beta2_pow));
        sc.bc1_next = __double2float_rn(__dsub_rn(1.0, __dmul_rn(sc.beta1_pow, (double)a.k.b1)));
        sc.bc2_next = __double2float_rn(__dsub_rn(1.0, __dmul_rn(sc.beta2_pow, (double)a.k.b2)));
        if (a.pingpong) sc.cur ^= 1;           // the step's writes become the state
        if (a.dynamic && a.growth_interval > 0) {
            sc.good_steps += 1;
            if (sc.good_steps >= a.growth_interval) {
                sc.loss_scale = __fmul_rn(sc.loss_scale, 2.0f);
                sc.good_steps = 0;
            }
        }
    }
    S->sc = sc;
    S->st = st;
}

struct RedShared {
    double d[ZERO_THREADS / 32];
    int    i[ZERO_THREADS / 32];
    int    last;
};

// The ticket: an atomic add with release and acquire semantics at GPU scope.
// Its release orders this thread's partial and flag stores (and, through the
// block's barriers, its block's stores) before the increment; the last block's
// acquire, with the barrier after it, orders every block's partial before its
// reads.  No separate fences.
static __device__ __forceinline__ unsigned ticket_acq_rel(unsigned* counter)
{
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    return old;
}

// Publish this block's partial; the last block to arrive finalizes the step.  A
// bucket's reduce only stores its blocks' partials: the apply step combines every
// bucket's, so a bucket's grid ends with its last block's store.
static __device__ __forceinline__ void reduce_and_finalize(const StepArgs& a, const NormAcc& acc,
                                                           int bad, NormShared& sh)
{
    const double bsum = block_norm(acc, sh);
    const int    bbad = __syncthreads_or(bad);
    if (a.bucket >= 0) {
        if (threadIdx.x == 0) {
            a.bucket_partial[blockIdx.x] = bsum;
            a.bucket_flag[blockIdx.x] = bbad;
        }
        return;
    }
    if (threadIdx.x == 0) {
        a.state->partial[blockIdx.x] = bsum;
        a.state->flag[blockIdx.x]    = bbad;
        sh.last = (ticket_acq_rel(&a.state->counter) == gridDim.x - 1);
    }
    __syncthreads();
    if (!sh.last) return;
    // thread 0's acquire (the ticket) and the barrier order every block's
    // partial before these reads
    double x = 0.0;
    int f = 0;
    for (int b = threadIdx.x; b < (int)gridDim.x; b += blockDim.x) {
        x = __dadd_rn(x, __ldcg(&a.state->partial[b]));
        f |= __ldcg(&a.state->flag[b]);
    }
    NormAcc xa;
    xa.wide = x;
    const double total = block_norm(xa, sh);
    const int    any   = __syncthreads_or(f);
    if (threadIdx.x == 0) {
        finalize(a, a.state->sc, a.state->st.err, total, any);
        a.state->counter = 0;
    }
}

// Bucketed step, after every bucket is reduced: the global norm and overflow flag
// from every bucket's per-block partials ([nbuckets][grid], the last bucket using
// its first last_grid slots), then the step's scalar bookkeeping.  Block f of
// the grid takes the buckets [nb f / F, nb (f+1) / F) in bucket order, each
// thread the slots t, t + 256, ... of each; the block sums are combined in block
// order by the last block to arrive.  The order is fixed by the plan's layout.
template <int DT>
__global__ void __launch_bounds__(ZERO_THREADS) k_bucket_finalize(const StepArgs a, int nbuckets,
                                                                  int grid, int last_grid)
{
    __shared__ NormShared sh;
    const int F = gridDim.x;
    const int b0 = (int)((int64_t)nbuckets * blockIdx.x / F);
    const int b1 = (int)((int64_t)nbuckets * (blockIdx.x + 1) / F);
    NormAcc x;
    int f = 0;
    for (int b = b0; b < b1; b++) {
        const int slots = b == nbuckets - 1 ? last_grid : grid;
        const double* p = a.bucket_partial + (int64_t)b * grid;
        const int32_t* q = a.bucket_flag + (int64_t)b * grid;
        for (int s = threadIdx.x; s < slots; s += blockDim.x) {
            x.wide = __dadd_rn(x.wide, p[s]);
            f |= q[s];
        }
    }
    reduce_and_finalize(a, x, f, sh);
}

static __device__ __forceinline__ void unpack8(const float4 a, const float4 b, float (&x)[8])
{
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// ---- pass 1: stages 1-3a (fold, average, unscale, flag, squares) ----------
// At most 4 resident blocks per SM leaves each thread the registers to keep
// all 16 rank loads of a chunk in flight (measured fastest).
template <int DT, int ND, bool WRITE_G>
__global__ void __launch_bounds__(ZERO_THREADS, 4) k_reduce(const StepArgs a)
{
    __shared__ NormShared sh;
    // the update pass may be scheduled now: it loads its state, then waits for
    // this grid to finish before it reads anything this grid writes
    asm volatile("griddepcontrol.launch_dependents;");
    // a bucket's reduce is launched as a programmatic dependent of whatever the
    // stream ran before it (so its blocks are placed during the previous grid's
    // tail): it reads nothing until that grid has completed and its writes are
    // visible, whoever wrote the bucket's gradients
    if (a.bucket >= 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int nd = ND > 0 ? ND : a.nd;
    Unscale un;
    un.init(nd, a.state->sc.loss_scale);
    NormAcc acc;
    int bad = 0;
    const int64_t nvec = a.n >> 3;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t vi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; vi < nvec; vi += stride) {
        float s[8], g[8];
        fold8<DT, ND>(a.grads, a.rank_stride, vi, nd, s);
#pragma unroll
        for (int e = 0; e < 8; e++) {
            g[e] = un(s[e]);
            bad |= not_finite(g[e]);
        }
        add_group(acc, g);
        if (WRITE_G) {
            float4* o = reinterpret_cast<float4*>(a.g32) + 2 * vi;
            __stcs(o, make_float4(g[0], g[1], g[2], g[3]));
            __stcs(o + 1, make_float4(g[4], g[5], g[6], g[7]));
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < 8) {            // the ragged tail (< 8 elements)
        const int64_t i = (nvec << 3) + threadIdx.x;
        if (i < a.n) {
            const float g = un(fold1<DT>(a.grads, a.rank_stride, i, nd));
            bad |= not_finite(g);
            add_one(acc, g);
            if (WRITE_G) a.g32[i] = g;
        }
    }
    reduce_and_finalize(a, acc, bad, sh);
}

// ---- qwZ epilogue: the updated 16-bit parameters quantized block by block ----
// x: a lane's 16-bit parameters widened back to binary32 (0 for elements past
// the shard's end).  The ZERO_QBLOCK-element block's absmax is a warp shuffle
// reduction, then (when a block spans W warps) a shared-memory combine; the
// codes and the scale are those codes_n / zero_quantize_shard give.
template <int QB, int N, int W>
static __device__ __forceinline__ void quant_epilogue(const float (&x)[N], int64_t e0, bool live,
                                                      const StepArgs& a, float* sh_amax)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < N; i++) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if constexpr (W > 1) {
        const int w = threadIdx.x >> 5;
        if ((threadIdx.x & 31) == 0) sh_amax[w] = amax;
        __syncthreads();
        const int w0 = w - w % W;
#pragma unroll
        for (int k = 0; k < W; k++) amax = fmaxf(amax, sh_amax[w0 + k]);
    }
    const float scale = __fdiv_rn(amax, QMax<QB>::v);
    if (live && (e0 % ZERO_QBLOCK) == 0) a.qscales[e0 / ZERO_QBLOCK] = scale;
    uint32_t c[N];
    codes_n<QB, N>(x, scale, c);
    if (!live) return;
    if constexpr (N == 8) {
        store8<QB>(a.qcodes, INT64_MAX, e0, c);
    } else {                                           // N == 4
        if (QB == 8) {
            *reinterpret_cast<uint32_t*>(a.qcodes + e0) =
                __byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040),
                            0x5410);
        } else {
            *reinterpret_cast<uint16_t*>(a.qcodes + e0 / 2) =
                (uint16_t)((c[0] & 0xFu) | ((c[1] & 0xFu) << 4) | ((c[2] & 0xFu) << 8) |
                           ((c[3] & 0xFu) << 12));
        }
    }
}

// ---- pass 2: stages 4-6a (clip, Adam, cast, write-back) -------------------
// One thread per 4 consecutive elements, one launch-wide block per 1024
// elements (not a persistent grid: measured faster for this read-write mix).
// The thread whose 4-element slot runs past n takes the ragged tail alone.
// Launched as a programmatic dependent of pass 1: master, m, v (and, when
// recomputing, the 16-bit gradients' rank-order sums) are loaded first, since
// pass 1 does not write them; griddepcontrol.wait then waits for pass 1 to
// complete before the step status and the fp32 gradient are read.
// QB = 8 or 4: the qwZ epilogue (ZeRO-3 shards only, whose length is a multiple
// of 64, so there is no ragged tail); a 256-element block is two warps.  On a
// skipped step the unchanged parameters are quantized, so the codes are valid
// whatever the buffers held.
template <int DT, int ND, bool RECOMPUTE, int QB = 0>
__global__ void __launch_bounds__(ZERO_THREADS) k_update(const StepArgs a)
{
    const int nd = ND > 0 ? ND : a.nd;
    const int64_t vi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nvec = a.n >> 2;
    float4* pm = reinterpret_cast<float4*>(a.master) + vi;
    float4* mm = reinterpret_cast<float4*>(a.m) + vi;
    float4* vv = reinterpret_cast<float4*>(a.v) + vi;
    float4 p{}, m{}, v{};
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (vi < nvec) {
        p = __ldcs(pm);
        m = __ldcs(mm);
        v = __ldcs(vv);
        if (RECOMPUTE) fold4<DT, ND>(a.grads, a.rank_stride, vi, nd, s);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const DevStatus st = a.state->st;
    if constexpr (QB != 0) {
        __shared__ float sh_amax[ZERO_THREADS / 32];
        if (st.err) return;
        float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const bool live = vi < nvec;
        if (st.skipped) {                              // quantize the unchanged parameters
            if (live) {
                const uint2 w = __ldcs(reinterpret_cast<const uint2*>(a.params) + vi);
                widen2<DT>(w.x, x[0], x[1]);
                widen2<DT>(w.y, x[2], x[3]);
            }
        } else if (live) {
            const float c = st.clip_coef, bc1 = st.bc1, bc2 = st.bc2;
            float g[4];
            if (RECOMPUTE) {
                Unscale un;
                un.init(nd, st.used_scale);
#pragma unroll
                for (int e = 0; e < 4; e++) g[e] = un(s[e]);
            } else {
                const float4 g4 = __ldcs(reinterpret_cast<const float4*>(a.g32) + vi);
                g[0] = g4.x; g[1] = g4.y; g[2] = g4.z; g[3] = g4.w;
            }
            adam1(g[0], c, p.x, m.x, v.x, bc1, bc2, a.k);
            adam1(g[1], c, p.y, m.y, v.y, bc1, bc2, a.k);
            adam1(g[2], c, p.z, m.z, v.z, bc1, bc2, a.k);
            adam1(g[3], c, p.w, m.w, v.w, bc1, bc2, a.k);
            __stcs(pm, p);
            __stcs(mm, m);
            __stcs(vv, v);
            const uint2 w = make_uint2(narrow2<DT>(p.x, p.y), narrow2<DT>(p.z, p.w));
            __stcs(reinterpret_cast<uint2*>(a.params) + vi, w);
            widen2<DT>(w.x, x[0], x[1]);
            widen2<DT>(w.y, x[2], x[3]);
        }
        quant_epilogue<QB, 4, ZERO_QBLOCK / 128>(x, vi << 2, live, a, sh_amax);
        return;
    }
    if (st.skipped || st.err) return;
    const float c = st.clip_coef, bc1 = st.bc1, bc2 = st.bc2;
    Unscale un;
    if (RECOMPUTE) un.init(nd, st.used_scale);
    if (vi < nvec) {
        float g[4];
        if (RECOMPUTE) {
#pragma unroll
            for (int e = 0; e < 4; e++) g[e] = un(s[e]);
        } else {
            const float4 g4 = __ldcs(reinterpret_cast<const float4*>(a.g32) + vi);
            g[0] = g4.x; g[1] = g4.y; g[2] = g4.z; g[3] = g4.w;
        }
        adam1(g[0], c, p.x, m.x, v.x, bc1, bc2, a.k);
        adam1(g[1], c, p.y, m.y, v.y, bc1, bc2, a.k);
        adam1(g[2], c, p.z, m.z, v.z, bc1, bc2, a.k);
        adam1(g[3], c, p.w, m.w, v.w, bc1, bc2, a.k);
        __stcs(pm, p);
        __stcs(mm, m);
        __stcs(vv, v);
        __stcs(reinterpret_cast<uint2*>(a.params) + vi,
               make_uint2(narrow2<DT>(p.x, p.y), narrow2<DT>(p.z, p.w)));
    } else if (vi == nvec) {
        for (int64_t i = nvec << 2; i < a.n; i++) {
            const float g = RECOMPUTE ? un(fold1<DT>(a.grads, a.rank_stride, i, nd)) : a.g32[i];
            float pi = a.master[i], mi = a.m[i], vi1 = a.v[i];
            adam1(g, c, pi, mi, vi1, bc1, bc2, a.k);
            a.master[i] = pi;
            a.m[i] = mi;
            a.v[i] = vi1;
            a.params[i] = narrow1<DT>(pi);
        }
    }
}

// ---- fused single pass (no clip, no dynamic scale, no skip on overflow):
// stages 1-6a ----------------------------------------------------------------
// One 8-element vector of the step: fold, unscale, flag, squares, Adam, cast,
// write-back; returns the 8 new 16-bit parameters packed in w.  PP: a ping-pong
// step, reading state set `cur` and writing the other one.
template <int DT, int ND, bool PP = false>
static __device__ __forceinline__ void fused8(const StepArgs& a, int64_t vi, int nd,
                                              const Unscale& un, float bc1, float bc2,
                                              NormAcc& acc, int& bad, uint4& w, int cur = 0)
{
    float4* pm = reinterpret_cast<float4*>(a.master);
    float4* mm = reinterpret_cast<float4*>(a.m);
    float4* vv = reinterpret_cast<float4*>(a.v);
    float4* po = pm;
    float4* mo = mm;
    float4* vo = vv;
    if constexpr (PP) {
        float4* p2 = reinterpret_cast<float4*>(a.master2);
        float4* m2 = reinterpret_cast<float4*>(a.m2);
        float4* v2 = reinterpret_cast<float4*>(a.v2);
        if (cur) {
            po = pm; mo = mm; vo = vv;
            pm = p2; mm = m2; vv = v2;
        } else {
            po = p2; mo = m2; vo = v2;
        }
    }
    float s[8], g[8], p[8], m[8], v[8];
    const float4 p0 = __ldcs(pm + 2 * vi), p1 = __ldcs(pm + 2 * vi + 1);
    const float4 m0 = __ldcs(mm + 2 * vi), m1 = __ldcs(mm + 2 * vi + 1);
    const float4 v0 = __ldcs(vv + 2 * vi), v1 = __ldcs(vv + 2 * vi + 1);
    fold8<DT, ND>(a.grads, a.rank_stride, vi, nd, s);
#pragma unroll
    for (int e = 0; e < 8; e++) {
        g[e] = un(s[e]);
        bad |= not_finite(g[e]);
    }
    add_group(acc, g);
    unpack8(p0, p1, p);
    unpack8(m0, m1, m);
    unpack8(v0, v1, v);
#pragma unroll
    for (int e = 0; e < 8; e++) adam1(g[e], 1.0f, p[e], m[e], v[e], bc1, bc2, a.k);
    __stcs(po + 2 * vi, make_float4(p[0], p[1], p[2], p[3]));
    __stcs(po + 2 * vi + 1, make_float4(p[4], p[5], p[6], p[7]));
    __stcs(mo + 2 * vi, make_float4(m[0], m[1], m[2], m[3]));
    __stcs(mo + 2 * vi + 1, make_float4(m[4], m[5], m[6], m[7]));
    __stcs(vo + 2 * vi, make_float4(v[0], v[1], v[2], v[3]));
    __stcs(vo + 2 * vi + 1, make_float4(v[4], v[5], v[6], v[7]));
    w = make_uint4(narrow2<DT>(p[0], p[1]), narrow2<DT>(p[2], p[3]), narrow2<DT>(p[4], p[5]),
                   narrow2<DT>(p[6], p[7]));
    __stcs(reinterpret_cast<uint4*>(a.params) + vi, w);
}

// The fused pass.  QB = 8 or 4 adds the qwZ epilogue (ZeRO-3 shards only, whose
// length is a multiple of 64): a warp's 32 vectors are 256 consecutive elements
// starting on a multiple of 256, one quantization block, so the block's absmax
// is one warp shuffle reduction.  The loop then runs while the warp's first
// vector is in range, with the lanes past the end idle, so every lane takes the
// shuffles.  PP: the ping-pong step (state set sc.cur in, the other out), whose
// repair pass is a programmatic dependent of this grid.
template <int DT, int ND, int QB, bool PP = false>
static __device__ __forceinline__ void fused_pass(const StepArgs& a)
{
    __shared__ NormShared sh;
    if constexpr (PP) asm volatile("griddepcontrol.launch_dependents;");
    const DevScalars sc = a.state->sc;
    const int nd = ND > 0 ? ND : a.nd;
    Unscale un;
    un.init(nd, sc.loss_scale);
    // bias corrections of step t+1 (this path never skips), kept by the last step
    const float bc1 = sc.bc1_next, bc2 = sc.bc2_next;
    NormAcc acc;
    int bad = 0;
    const int64_t nvec = a.n >> 3;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if constexpr (QB == 0) {
        for (int64_t vi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; vi < nvec; vi += stride) {
            uint4 w;
            fused8<DT, ND, PP>(a, vi, nd, un, bc1, bc2, acc, bad, w, PP ? sc.cur : 0);
        }
    } else {
        const int lane = threadIdx.x & 31;
        for (int64_t vi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; vi - lane < nvec;
             vi += stride) {
            float x[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
            const bool live = vi < nvec;
            if (live) {
                uint4 w;
                fused8<DT, ND>(a, vi, nd, un, bc1, bc2, acc, bad, w);
                widen2<DT>(w.x, x[0], x[1]);
                widen2<DT>(w.y, x[2], x[3]);
                widen2<DT>(w.z, x[4], x[5]);
                widen2<DT>(w.w, x[6], x[7]);
            }
            quant_epilogue<QB, 8, 1>(x, vi << 3, live, a, nullptr);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < 8) {
        const int64_t i = (nvec << 3) + threadIdx.x;
        if (i < a.n) {
            const float g = un(fold1<DT>(a.grads, a.rank_stride, i, nd));
            bad |= not_finite(g);
            add_one(acc, g);
            float* pi = a.master;
            float* mi = a.m;
            float* vi1 = a.v;
            float* po = pi;
            float* mo = mi;
            float* vo = vi1;
            if constexpr (PP) {
                if (sc.cur) {
                    pi = a.master2; mi = a.m2; vi1 = a.v2;
                } else {
                    po = a.master2; mo = a.m2; vo = a.v2;
                }
            }
            float p = pi[i], m = mi[i], v = vi1[i];
            adam1(g, 1.0f, p, m, v, bc1, bc2, a.k);
            po[i] = p;
            mo[i] = m;
            vo[i] = v;
            a.params[i] = narrow1<DT>(p);
        }
    }
    reduce_and_finalize(a, acc, bad, sh);
}

// Held to 4 blocks per SM (2 for the generic rank count), which every
// compiled-in rank count reaches without spilling.
template <int DT, int ND>
__global__ void __launch_bounds__(ZERO_THREADS, ND == 0 ? 2 : 4) k_fused(const StepArgs a)
{
    fused_pass<DT, ND, 0>(a);
}

// The ping-pong step's single pass (zero_step_pingpong), held to 3 blocks per SM
// (2 for the generic rank count): unbounded, the two pointer sets took it to 172
// registers at nd 64.
template <int DT, int ND>
__global__ void __launch_bounds__(ZERO_THREADS, ND == 0 ? 2 : 3) k_fused_pp(const StepArgs a)
{
    fused_pass<DT, ND, 0, true>(a);
}

// After a ping-pong step: when the step was skipped, its pass has already
// written the 16-bit parameters from the discarded new state, so they are
// rewritten from the current set's master (cur, unchanged by a skipped step);
// otherwise nothing.  A programmatic dependent of the pass: it waits for the
// pass's completion before reading the step status.  One thread per 4 elements.
template <int DT>
__global__ void __launch_bounds__(ZERO_THREADS) k_pp_repair(const StepArgs a)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!a.state->st.skipped) return;
    const float* master = a.state->sc.cur ? a.master2 : a.master;
    const int64_t vi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nvec = a.n >> 2;
    if (vi < nvec) {
        const float4 p = __ldcs(reinterpret_cast<const float4*>(master) + vi);
        __stcs(reinterpret_cast<uint2*>(a.params) + vi,
               make_uint2(narrow2<DT>(p.x, p.y), narrow2<DT>(p.z, p.w)));
    } else if (vi == nvec) {
        for (int64_t i = nvec << 2; i < a.n; i++) a.params[i] = narrow1<DT>(master[i]);
    }
}

// The qwZ instances are held to 4 blocks per SM (64 registers; 2 for the
// generic rank count), the occupancy the plain instances reach; unbounded, the
// compiler keeps every rank's load of a vector in flight at once (254 registers,
// one block per SM at nd 64).
template <int DT, int ND, int QB>
__global__ void __launch_bounds__(ZERO_THREADS, ND == 0 ? 2 : 4) k_fused_q(const StepArgs a)
{
    fused_pass<DT, ND, QB>(a);
}

}  // namespace zero
