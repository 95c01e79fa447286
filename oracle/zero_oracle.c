/*
 * zero_oracle.c -- plain CPU oracle for the ZeRO-DP sharded mixed-precision
 * optimizer step.  TEST INFRASTRUCTURE ONLY (see zero_oracle.h).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared
 *        -pthread -o liboracle.so zero_oracle.c -lm
 * C11 with FLT_EVAL_METHOD == 0 (x86-64 SSE, AArch64): every float
 * expression below is evaluated in binary32, one rounding per operation.
 */
#include "zero_oracle.h"

#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#if FLT_EVAL_METHOD != 0
#error "the oracle needs binary32 evaluation of float expressions"
#endif

/* ======================================================================
 * 16-bit formats.  Written from the format definitions with exact double
 * arithmetic (scalings by powers of two and integer-valued doubles), so
 * that the rounding rule is visible: find the binade, divide by its
 * quantum, round the quotient to the nearest integer with ties to even.
 * ====================================================================== */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float zo_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e    = (h >> 10) & 31;
    int f    = h & 1023;
    double mag;
    if (e == 31) {
        if (f != 0) return NAN;
        return sign ? -INFINITY : INFINITY;
    }
    if (e == 0) mag = ldexp((double)f, -24);          /* subnormal f * 2^-24      */
    else        mag = ldexp(1024.0 + f, e - 25);      /* (1 + f/1024) * 2^(e-15)  */
    return (float)(sign ? -mag : mag);                /* exact in binary32        */
}

/* round a >= 0 to the grid of multiples of q, ties to the even multiple */
static double round_to_quantum(double a, double q)
{
    double k = a / q;              /* exact: q is a power of two        */
    double r = floor(k);
    double frac = k - r;           /* exact                             */
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    return r * q;                  /* exact                             */
}

/* exponent E of the binade [2^E, 2^(E+1)) that holds a > 0 */
static int binade(double a)
{
    int e;
    (void)frexp(a, &e);            /* a = mant * 2^e, mant in [0.5, 1)  */
    return e - 1;
}

uint16_t zo_float_to_half(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00);
    if (isinf(x)) return (uint16_t)(sign | 0x7C00);
    double a = fabs((double)x);
    if (a == 0.0) return sign;
    int E = binade(a);
    if (E < -14) E = -14;                             /* subnormal binades share 2^-24 */
    double val = round_to_quantum(a, ldexp(1.0, E - 10));
    if (val >= 65536.0) return (uint16_t)(sign | 0x7C00);   /* past 65504 */
    if (val < ldexp(1.0, -14))                              /* subnormal or zero */
        return (uint16_t)(sign | (uint16_t)(val / ldexp(1.0, -24)));
    E = binade(val);                                  /* rounding may carry */
    uint16_t frac = (uint16_t)(val / ldexp(1.0, E - 10) - 1024.0);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | frac);
}

/* bfloat16: the upper 16 bits of a binary32 (8 exponent bits, 7 fraction). */
float zo_bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t zo_float_to_bf16(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0);
    if (isinf(x)) return (uint16_t)(sign | 0x7F80);
    double a = fabs((double)x);
    if (a == 0.0) return sign;
    int E = binade(a);
    if (E < -126) E = -126;                           /* subnormal binades share 2^-133 */
    double val = round_to_quantum(a, ldexp(1.0, E - 7));
    if (val >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float fv = (float)val;                            /* exact: <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &fv, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));    /* low 16 bits are zero */
}

static float to_float(int dtype, uint16_t b)
{
    return dtype == 0 ? zo_half_to_float(b) : zo_bf16_to_float(b);
}

static uint16_t from_float(int dtype, float x)
{
    return dtype == 0 ? zo_float_to_half(x) : zo_float_to_bf16(x);
}

void zo_to_float_n(int dtype, const uint16_t* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = to_float(dtype, in[i]);
}

void zo_from_float_n(int dtype, const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = from_float(dtype, in[i]);
}

/* ======================================================================
 * Memory ledger and communication volume.
 * [L18] sec. 1.2: per parameter 2 (fp16 weight) + 2 (fp16 gradient) + K
 * bytes of optimizer state (K = 12 for Adam: fp32 master, m, v; the slides'
 * variant counts an fp32 gradient too, K = 16).  [L18] sec. 2.1 and
 * [L32] sec. 2.3 give the per-rank formula of each stage.
 * ====================================================================== */
double zo_state_bytes(double psi, double nd, int stage, double K)
{
    switch (stage) {
    case 0: return (2.0 + 2.0 + K) * psi;
    case 1: return 4.0 * psi + K * psi / nd;
    case 2: return 2.0 * psi + (2.0 + K) * psi / nd;
    case 3: return (4.0 + K) * psi / nd;
    default: return NAN;
    }
}

/* [L18] sec. 3.1, [L32] sec. 2.3 table, [PZ] 0x07: all-reduce = reduce-
 * scatter (Psi) + all-gather (Psi); ZeRO-1/2 keep 2 Psi; ZeRO-3 gathers the
 * parameters again in the backward pass: 3 Psi.  Each collective moves the
 * (Nd - 1)/Nd share of its message that is not already local.           */
double zo_comm_volume(double psi, double nd, int stage, int exact)
{
    double v;
    if (stage >= 0 && stage <= 2) v = 2.0 * psi;
    else if (stage == 3)          v = 3.0 * psi;
    else return NAN;
    if (exact) v = v * (nd - 1.0) / nd;
    return v;
}

double zo_max_params(double mem_bytes, double nd, int stage, double K)
{
    return mem_bytes / zo_state_bytes(1.0, nd, stage, K);
}

/* ======================================================================
 * Flat partition.  All parameters concatenated in list order and split
 * into nd equal contiguous pieces; the piece length is rounded up to a
 * multiple of 64 elements and the tail is zero padding.
 * ====================================================================== */
int64_t zo_shard_elems(int64_t psi, int nd)
{
    int64_t per = (psi + nd - 1) / nd;
    return (per + 63) / 64 * 64;
}

/* ======================================================================
 * The step, stage by stage.
 * ====================================================================== */

/* Stages 1-2.  [L18] sec. 2.2: the reduce-scatter leaves each rank the
 * average of its slice over all ranks; sec. 2.5: the sum is taken in a
 * fixed rank order.  Loss-scale unscale: [L32] 4.3 ("loss NaN: check the
 * fp16 loss_scale").  The average is divided by nd, then by the scale. */
int zo_reduce(int nd, int64_t n, int dtype, const uint16_t* grads,
              int64_t rank_stride, float loss_scale, float* g)
{
    int overflow = 0;
    for (int64_t i = 0; i < n; i++) {
        float s = 0.0f;
        for (int r = 0; r < nd; r++)
            s = s + to_float(dtype, grads[(int64_t)r * rank_stride + i]);
        float avg = s / (float)nd;
        float gi  = avg / loss_scale;
        if (!isfinite(gi)) overflow = 1;
        g[i] = gi;
    }
    return overflow;
}

/* Stage 3a: the squared L2 norm of the whole gradient.  Each square of a
 * binary32 value is exact in binary64; the sum is taken in index order. */
double zo_sumsq(int64_t n, const float* g)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; i++) acc = acc + (double)g[i] * (double)g[i];
    return acc;
}

/* Stage 3b: gradient clipping by global norm ([L32] 4.2 "gradient_clipping",
 * 0 = off).  c = clip / norm when the norm exceeds clip, computed in double
 * and rounded once to binary32. */
float zo_clip_coef(double norm, float clip)
{
    if (clip > 0.0f && norm > (double)clip) return (float)((double)clip / norm);
    return 1.0f;
}

void zo_advance(const zo_hparams* hp, zo_scalars* st, int overflow, zo_result* res)
{
    res->overflow = overflow;
    if (overflow && (hp->dynamic_scale || hp->skip_on_overflow)) {
        /* skipped step: nothing moves except, under dynamic scaling, the
         * loss scale, which backs off */
        res->skipped  = 1;
        if (hp->dynamic_scale) {
            st->loss_scale = st->loss_scale * hp->backoff;
            st->good_steps = 0;
        }
        res->bc1 = res->bc2 = 0.0f;
        return;
    }
    res->skipped = 0;
    st->t = st->t + 1;
    st->beta1_pow = st->beta1_pow * (double)hp->beta1;
    st->beta2_pow = st->beta2_pow * (double)hp->beta2;
    res->bc1 = (float)(1.0 - st->beta1_pow);
    res->bc2 = (float)(1.0 - st->beta2_pow);
    if (hp->dynamic_scale && hp->growth_interval > 0) {
        st->good_steps = st->good_steps + 1;
        if (st->good_steps >= hp->growth_interval) {
            st->loss_scale = st->loss_scale * 2.0f;
            st->good_steps = 0;
        }
    }
}

/* Stages 4-5.  [L18] sec. 2.1: Adam is elementwise, so a rank needs only the
 * m, v, master weight and averaged gradient of its own slice; sec. 2.2: it
 * updates its fp32 variance, momentum and master, then copies to fp16.
 * The update is Adam with bias correction (AdamW when decoupled_wd). */
void zo_adam(int64_t n, const float* g, float c, float* master, float* m, float* v,
             uint16_t* params, int dtype, const zo_hparams* hp, float bc1, float bc2)
{
    const float omb1  = (float)(1.0 - (double)hp->beta1);
    const float omb2  = (float)(1.0 - (double)hp->beta2);
    const float decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
    for (int64_t i = 0; i < n; i++) {
        float gi = g[i] * c;
        float p  = master[i];
        if (hp->weight_decay != 0.0f) {
            if (hp->decoupled_wd) p  = p * decay;
            else                  gi = gi + hp->weight_decay * p;
        }
        float mi   = hp->beta1 * m[i] + omb1 * gi;
        float vi   = hp->beta2 * v[i] + omb2 * (gi * gi);
        float mhat = mi / bc1;
        float vhat = vi / bc2;
        float upd  = mhat / (sqrtf(vhat) + hp->eps);
        p = p - hp->lr * upd;
        master[i] = p;
        m[i] = mi;
        v[i] = vi;
        params[i] = from_float(dtype, p);
    }
}

int zo_step(int nd, int64_t n, int dtype, const uint16_t* grads,
            float* master, float* m, float* v, uint16_t* params,
            const zo_hparams* hp, zo_scalars* st, zo_result* res)
{
    float* g = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    if (!g) return -1;
    int overflow   = zo_reduce(nd, n, dtype, grads, n, st->loss_scale, g);
    res->grad_norm = sqrt(zo_sumsq(n, g));
    res->clip_coef = zo_clip_coef(res->grad_norm, hp->clip_norm);
    zo_advance(hp, st, overflow, res);
    if (!res->skipped)
        zo_adam(n, g, res->clip_coef, master, m, v, params, dtype, hp, res->bc1, res->bc2);
    free(g);
    return 0;
}

/* ---- sharded execution: each emulated rank on its own slice --------- */
typedef struct {
    int nd, dtype, first_rank, rank_step;
    int64_t n, shard;
    const uint16_t* grads;
    float *g, *master, *m, *v;
    uint16_t* params;
    const zo_hparams* hp;
    float loss_scale, c, bc1, bc2;
    int phase;                      /* 0: reduce + partial, 1: update      */
    double* partial;                /* [nd] squared-norm partial per rank   */
    int* overflow;                  /* [nd]                                 */
} shard_job;

static void* shard_worker(void* arg)
{
    shard_job* j = (shard_job*)arg;
    for (int r = j->first_rank; r < j->nd; r += j->rank_step) {
        int64_t lo = (int64_t)r * j->shard;
        int64_t hi = lo + j->shard < j->n ? lo + j->shard : j->n;
        if (lo > hi) lo = hi;
        if (j->phase == 0) {
            j->overflow[r] = zo_reduce(j->nd, hi - lo, j->dtype, j->grads + lo, j->n,
                                       j->loss_scale, j->g + lo);
            j->partial[r]  = zo_sumsq(hi - lo, j->g + lo);
        } else {
            zo_adam(hi - lo, j->g + lo, j->c, j->master + lo, j->m + lo, j->v + lo,
                    j->params + lo, j->dtype, j->hp, j->bc1, j->bc2);
        }
    }
    return NULL;
}

/* Thread k runs ranks k, k + nthreads, ...  Each rank's work depends only on
 * its own slice, so the result does not depend on nthreads. */
static void run_ranks(const shard_job* base, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > base->nd) nthreads = base->nd;
    shard_job* jobs    = (shard_job*)malloc(sizeof(shard_job) * (size_t)nthreads);
    pthread_t* threads = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int*       started = (int*)calloc((size_t)nthreads, sizeof(int));
    if (!jobs || !threads || !started) {          /* run every rank on this thread */
        shard_job one = *base;
        one.first_rank = 0;
        one.rank_step  = 1;
        shard_worker(&one);
        free(jobs); free(threads); free(started);
        return;
    }
    for (int k = 0; k < nthreads; k++) {
        jobs[k] = *base;
        jobs[k].first_rank = k;
        jobs[k].rank_step  = nthreads;
    }
    for (int k = 1; k < nthreads; k++)
        started[k] = pthread_create(&threads[k], NULL, shard_worker, &jobs[k]) == 0;
    shard_worker(&jobs[0]);
    for (int k = 1; k < nthreads; k++) {
        if (started[k]) pthread_join(threads[k], NULL);
        else            shard_worker(&jobs[k]);
    }
    free(jobs); free(threads); free(started);
}

int zo_step_sharded(int nd, int64_t n, int64_t shard, int dtype, const uint16_t* grads,
                    float* master, float* m, float* v, uint16_t* params,
                    const zo_hparams* hp, zo_scalars* st, zo_result* res, int nthreads)
{
    float*  g       = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    double* partial = (double*)calloc((size_t)nd, sizeof(double));
    int*    ovf     = (int*)calloc((size_t)nd, sizeof(int));
    if (!g || !partial || !ovf) { free(g); free(partial); free(ovf); return -1; }

    shard_job job;
    memset(&job, 0, sizeof job);
    job.nd = nd; job.dtype = dtype; job.n = n; job.shard = shard;
    job.grads = grads; job.g = g; job.master = master; job.m = m; job.v = v;
    job.params = params; job.hp = hp; job.loss_scale = st->loss_scale;
    job.partial = partial; job.overflow = ovf;

    job.phase = 0;
    run_ranks(&job, nthreads);

    /* the scalar all-reduces: OR of the flags, sum of the partials in rank order */
    int overflow = 0;
    double sumsq = 0.0;
    for (int r = 0; r < nd; r++) { overflow |= ovf[r]; sumsq = sumsq + partial[r]; }
    res->grad_norm = sqrt(sumsq);
    res->clip_coef = zo_clip_coef(res->grad_norm, hp->clip_norm);
    zo_advance(hp, st, overflow, res);

    if (!res->skipped) {
        job.phase = 1;
        job.c = res->clip_coef; job.bc1 = res->bc1; job.bc2 = res->bc2;
        run_ranks(&job, nthreads);
    }
    free(g); free(partial); free(ovf);
    return 0;
}

/* ======================================================================
 * ZeRO-3 unit gather / shard.  [L18] sec. 2.4: before a unit is used its
 * owners send their pieces to every rank; [ZL8] sec. 8.4: the pieces of a
 * module are gathered into one contiguous buffer.
 * ====================================================================== */
void zo_gather_unit(int nd, int64_t len, int64_t slice,
                    const uint16_t* const* slices, uint16_t* out)
{
    for (int64_t j = 0; j < len; j++) {
        int64_t k = j / slice;
        if (k >= nd) break;
        out[j] = slices[k][j % slice];
    }
}

void zo_shard_unit(int nd, int64_t len, int64_t slice,
                   const uint16_t* unit, uint16_t* const* slices)
{
    for (int k = 0; k < nd; k++)
        for (int64_t j = 0; j < slice; j++) {
            int64_t src = (int64_t)k * slice + j;
            slices[k][j] = src < len ? unit[src] : (uint16_t)0;
        }
}

/* ======================================================================
 * ZeRO++ qwZ: block-wise symmetric quantization of the weights that are
 * gathered ([L18] 4.5).
 * ====================================================================== */
static int32_t round_half_even_to_int(float v)
{
    double r = floor((double)v);
    double frac = (double)v - r;                       /* exact */
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    return (int32_t)r;
}

static void put_code(uint8_t* q, int64_t i, int bits, int32_t code)
{
    if (bits == 8) {
        q[i] = (uint8_t)(int8_t)code;
    } else {
        uint8_t nib = (uint8_t)(code & 0xF);
        if (i % 2 == 0) q[i / 2] = (uint8_t)((q[i / 2] & 0xF0) | nib);
        else            q[i / 2] = (uint8_t)((q[i / 2] & 0x0F) | (nib << 4));
    }
}

static int32_t get_code(const uint8_t* q, int64_t i, int bits)
{
    if (bits == 8) return (int32_t)(int8_t)q[i];
    uint8_t nib = (i % 2 == 0) ? (q[i / 2] & 0xF) : (q[i / 2] >> 4);
    return nib >= 8 ? (int32_t)nib - 16 : (int32_t)nib;      /* two's complement nibble */
}

void zo_quantize_f32(const float* x, int64_t n, int bits, int64_t block,
                     uint8_t* q, float* scales)
{
    const float qmax = (float)((1 << (bits - 1)) - 1);
    for (int64_t b0 = 0, blk = 0; b0 < n; b0 += block, blk++) {
        int64_t b1 = b0 + block < n ? b0 + block : n;
        float amax = 0.0f;
        for (int64_t i = b0; i < b1; i++) {
            float a = fabsf(x[i]);
            if (a > amax) amax = a;
        }
        float scale = amax / qmax;
        scales[blk] = scale;
        for (int64_t i = b0; i < b1; i++) {
            int32_t code = 0;
            if (scale != 0.0f) {
                code = round_half_even_to_int(x[i] / scale);
                if (code > (int32_t)qmax) code = (int32_t)qmax;
                if (code < -(int32_t)qmax) code = -(int32_t)qmax;
            }
            put_code(q, i, bits, code);
        }
    }
}

void zo_dequantize_f32(const uint8_t* q, const float* scales, int64_t n, int bits,
                       int64_t block, float* out)
{
    for (int64_t i = 0; i < n; i++) out[i] = (float)get_code(q, i, bits) * scales[i / block];
}

void zo_quantize_16(int dtype, const uint16_t* x, int64_t n, int bits, int64_t block,
                    uint8_t* q, float* scales)
{
    float* f = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    if (!f) return;
    for (int64_t i = 0; i < n; i++) f[i] = to_float(dtype, x[i]);
    zo_quantize_f32(f, n, bits, block, q, scales);
    free(f);
}

void zo_dequantize_16(int dtype, const uint8_t* q, const float* scales, int64_t n, int bits,
                      int64_t block, uint16_t* out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = from_float(dtype, (float)get_code(q, i, bits) * scales[i / block]);
}

void zo_gather_unit_q(int dtype, int nd, int64_t len, int64_t slice, int64_t offset, int bits,
                      int64_t block, const uint8_t* const* q, const float* const* scales,
                      uint16_t* out)
{
    for (int64_t j = 0; j < len; j++) {
        int64_t k = j / slice;
        if (k >= nd) break;
        int64_t e = offset + j % slice;             /* element of rank k's shard */
        out[j] = from_float(dtype, (float)get_code(q[k], e, bits) * scales[k][e / block]);
    }
}

/* ======================================================================
 * Sharded checkpoint: regroup the shards of one layout into another
 * ([Z026] sec. 5; [L32] sec. 4.3).  Written as the definition: every shard
 * position names one flat index (or padding); the flat vector is rebuilt from
 * the old layout and read back through the new one.
 * ====================================================================== */
int64_t zo_layout_shard_len(const zo_layout* L)
{
    int64_t total = 0;
    for (int u = 0; u < L->nunits; u++) total += zo_shard_elems(L->len[u], L->nd);
    return total;
}

int64_t zo_layout_global(const zo_layout* L, int r, int64_t j)
{
    int64_t unit_start = 0;                   /* flat index of the unit's first element */
    int64_t slice_start = 0;                  /* shard position of the unit's slice     */
    for (int u = 0; u < L->nunits; u++) {
        int64_t s = zo_shard_elems(L->len[u], L->nd);
        if (j < slice_start + s) {
            int64_t local = (int64_t)r * s + (j - slice_start);   /* element of the unit */
            return local < L->len[u] ? unit_start + local : -1;
        }
        unit_start += L->len[u];
        slice_start += s;
    }
    return -1;
}

void zo_reshard(const zo_layout* A, const void* const* old_shards, const zo_layout* B,
                void* const* new_shards, int elem_bytes)
{
    int64_t psi = 0;
    for (int u = 0; u < A->nunits; u++) psi += A->len[u];
    unsigned char* flat = (unsigned char*)calloc((size_t)(psi > 0 ? psi : 1), (size_t)elem_bytes);
    if (!flat) return;
    int64_t la = zo_layout_shard_len(A);
    for (int r = 0; r < A->nd; r++)
        for (int64_t j = 0; j < la; j++) {
            int64_t g = zo_layout_global(A, r, j);
            if (g >= 0)
                memcpy(flat + g * elem_bytes,
                       (const unsigned char*)old_shards[r] + j * elem_bytes, (size_t)elem_bytes);
        }
    int64_t lb = zo_layout_shard_len(B);
    for (int r = 0; r < B->nd; r++)
        for (int64_t j = 0; j < lb; j++) {
            int64_t g = zo_layout_global(B, r, j);
            unsigned char* dst = (unsigned char*)new_shards[r] + j * elem_bytes;
            if (g >= 0) memcpy(dst, flat + g * elem_bytes, (size_t)elem_bytes);
            else memset(dst, 0, (size_t)elem_bytes);
        }
    free(flat);
}

/* ======================================================================
 * ZeRO-Offload: the reduced gradient is copied to the host in the 16-bit
 * type and the host runs the update ([L18] sec. 4.4; [ZL8] sec. 6.2, 7).
 * ====================================================================== */
int zo_reduce16(int nd, int64_t n, int dtype, const uint16_t* grads, int64_t rank_stride,
                float loss_scale, uint16_t* g16, float* g)
{
    int bad = 0;
    for (int64_t i = 0; i < n; i++) {
        float sum = 0.0f;
        for (int k = 0; k < nd; k++)
            sum = sum + to_float(dtype, grads[(int64_t)k * rank_stride + i]);
        float mean = sum / (float)nd;
        uint16_t q = from_float(dtype, mean);            /* what crosses the link */
        float gi = to_float(dtype, q) / loss_scale;      /* unscaled on the host  */
        if (!isfinite(gi)) bad = 1;
        g16[i] = q;
        g[i] = gi;
    }
    return bad;
}

int zo_step_offload(int nd, int64_t n, int dtype, const uint16_t* grads,
                    float* master, float* m, float* v, uint16_t* params,
                    const zo_hparams* hp, zo_scalars* st, zo_result* res)
{
    size_t cnt = (size_t)(n > 0 ? n : 1);
    float* g = (float*)malloc(cnt * sizeof(float));
    uint16_t* q = (uint16_t*)malloc(cnt * sizeof(uint16_t));
    if (!g || !q) {
        free(g);
        free(q);
        return -1;
    }
    int bad = zo_reduce16(nd, n, dtype, grads, n, st->loss_scale, q, g);
    res->grad_norm = sqrt(zo_sumsq(n, g));
    res->clip_coef = zo_clip_coef(res->grad_norm, hp->clip_norm);
    zo_advance(hp, st, bad, res);
    if (!res->skipped)
        zo_adam(n, g, res->clip_coef, master, m, v, params, dtype, hp, res->bc1, res->bc2);
    free(g);
    free(q);
    return 0;
}
