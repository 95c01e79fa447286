/*
 * zero_oracle.h -- plain CPU oracle for the ZeRO-DP sharded mixed-precision
 * optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the slow, obviously-correct statement of
 * what the GPU path must compute.  Only the test suite, the smoke check of the
 * package entry point and the CPU-baseline leg of the benchmark may load it.
 * It shares no code, header, table or helper with the CUDA library: the
 * 16-bit conversions, the reduce, the norm, the Adam update, the partition
 * layout and the memory ledger are all restated here from the pages.
 *
 * Pages cited (title as printed; section numbers are the page's own):
 *   [L18]  "第 18 讲 · Memory Optimization in Distributed Training: ZeRO"
 *          (CMU 11-868 lecture notes)
 *   [Z026] "026｜ZeRO：数据并行中，没必要让每张卡保存全部训练状态"
 *   [L32]  "L3.2 显存优化与 ZeRO"
 *   [ZL8]  "图解分布式训练（八）—— ZeRO 学习"
 *   [PZ]   "ZeRO:" (ZeRO paper digest; 0x05 Deep Dive into ZeRO-DP,
 *          0x07 ZeRO-DP Communication Volume)
 *
 * Floating point: every fp32 operation is a single IEEE-754 round-to-nearest
 * operation in the order written; the library is compiled with
 * -ffp-contract=off so no multiply-add is fused.
 *
 * Parity pins: every function here is pinned by the not-gpu tests against
 * values the pages print, closed forms, library routines or invariants; none
 * is marked "parity unpinned".
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- 16-bit storage formats (IEEE 754-2008 binary16; bfloat16 = the upper
 *      half of binary32).  Round-to-nearest, ties to even. ---------------- */
float    zo_half_to_float(uint16_t h);
uint16_t zo_float_to_half(float x);
float    zo_bf16_to_float(uint16_t b);
uint16_t zo_float_to_bf16(float x);
/* dtype: 0 = fp16, 1 = bf16 (bulk versions for the tests) */
void zo_to_float_n(int dtype, const uint16_t* in, float* out, int64_t n);
void zo_from_float_n(int dtype, const float* in, uint16_t* out, int64_t n);

/* ---- memory ledger and communication volume ([L18] sec. 1.2, 2.1, 3.1;
 *      [Z026] sec. 2; [L32] sec. 2.1-2.3; [PZ] sec. 0x05, 0x07) ---------- */
/* bytes of model state held by one data-parallel rank:
 *   stage 0 (DP)   (2 + 2 + K) Psi
 *   stage 1        4 Psi + K Psi / Nd
 *   stage 2        2 Psi + (2 + K) Psi / Nd
 *   stage 3        (4 + K) Psi / Nd                                     */
double zo_state_bytes(double psi, double nd, int stage, double K);
/* elements each rank sends per step: 2 Psi for stages 0-2, 3 Psi for
 * stage 3; exact = 1 multiplies by (Nd - 1) / Nd                         */
double zo_comm_volume(double psi, double nd, int stage, int exact);
/* largest Psi whose model state fits in mem_bytes per rank              */
double zo_max_params(double mem_bytes, double nd, int stage, double K);

/* ---- flat partition ([L18] sec. 3.2 flat vector split evenly;
 *      [ZL8] sec. 8.4 flatten, each rank finds its contiguous piece) --- */
/* elements per rank: ceil(psi / nd) rounded up to a multiple of 64      */
int64_t zo_shard_elems(int64_t psi, int nd);

/* ---- optimizer description ------------------------------------------- */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int   decoupled_wd;     /* 1: AdamW decay p *= (1 - lr wd); 0: g += wd p */
    float clip_norm;        /* 0: no clipping                               */
    int   dynamic_scale;    /* 1: an overflow skips the step and backs the
                               loss scale off; growth after good steps     */
    float backoff;          /* scale multiplier on overflow                 */
    int   growth_interval;  /* good steps before the scale doubles; <=0 off */
    int   skip_on_overflow; /* 1: an overflow skips the step under a static
                               scale too (the scale is left as it is); 0:
                               under a static scale the flag is only
                               reported and the step goes ahead            */
} zo_hparams;

typedef struct {            /* optimizer scalars carried across steps       */
    float   loss_scale;
    int32_t good_steps;
    int64_t t;              /* completed (non-skipped) steps                */
    double  beta1_pow;      /* beta1^t, by repeated multiplication          */
    double  beta2_pow;
} zo_scalars;

typedef struct {            /* what one step reports                        */
    int32_t skipped;
    int32_t overflow;
    double  grad_norm;
    float   clip_coef;
    float   bc1, bc2;
} zo_result;

/* ---- the stages, each a plain loop ----------------------------------- */
/* stage 1 + 2: g[i] = ((sum_{r=0..nd-1} (float)grad[r][i]) / nd) / loss_scale,
 * the sum a left fold from 0.0f in rank order.  Returns 1 if any g[i] is
 * not finite.  grads[r * rank_stride + i].                               */
int zo_reduce(int nd, int64_t n, int dtype, const uint16_t* grads,
              int64_t rank_stride, float loss_scale, float* g);
/* stage 3a: sum of squares in double, sequential in index order          */
double zo_sumsq(int64_t n, const float* g);
/* stage 3b: c = clip / norm if norm > clip, else 1 (clip 0 = off)        */
float zo_clip_coef(double norm, float clip);
/* scalar bookkeeping: skip decision, loss-scale backoff/growth, t, bias
 * corrections.  Fills res->skipped, overflow, bc1, bc2.                  */
void zo_advance(const zo_hparams* hp, zo_scalars* st, int overflow, zo_result* res);
/* stages 4 + 5 (+ the write-back into the flat 16-bit buffer)            */
void zo_adam(int64_t n, const float* g, float c, float* master, float* m, float* v,
             uint16_t* params, int dtype, const zo_hparams* hp, float bc1, float bc2);

/* ---- the whole step -------------------------------------------------- */
/* Unsharded definition: one model, the averaged gradient, one update.
 * grads: [nd][n] (rank stride n).  Returns 0, or -1 on allocation failure. */
int zo_step(int nd, int64_t n, int dtype, const uint16_t* grads,
            float* master, float* m, float* v, uint16_t* params,
            const zo_hparams* hp, zo_scalars* st, zo_result* res);
/* Sharded execution of the same step: rank r owns [r*shard, (r+1)*shard)
 * of the flat vector, reduces only its slice, contributes one double
 * partial of the squared norm (combined in rank order), and updates only
 * its slice.  nthreads host threads run the ranks.  grads: [nd][n].       */
int zo_step_sharded(int nd, int64_t n, int64_t shard, int dtype, const uint16_t* grads,
                    float* master, float* m, float* v, uint16_t* params,
                    const zo_hparams* hp, zo_scalars* st, zo_result* res, int nthreads);

/* ---- ZeRO-3 unit gather ([L18] sec. 2.4; [ZL8] sec. 8.4) -------------- */
/* A unit of len elements is split into nd slices of slice elements each
 * (the tail zero-padded).  Gather writes the unit back: out[j] for
 * j < len is element j % slice of rank j / slice's slice.                */
void zo_gather_unit(int nd, int64_t len, int64_t slice,
                    const uint16_t* const* slices, uint16_t* out);
/* the inverse: split a unit into nd padded slices (slices[k][0..slice))  */
void zo_shard_unit(int nd, int64_t len, int64_t slice,
                   const uint16_t* unit, uint16_t* const* slices);

/* ---- ZeRO++ quantized weight gather, qwZ ([L18] 4.5: block-wise
 *      quantization, one scale per block, so a few large values only coarsen
 *      their own block) ------------------------------------------------------
 * Symmetric absmax quantization to `bits` (8 or 4) bits, qmax = 2^(bits-1)-1,
 * blocks of `block` consecutive elements (the last one may be short):
 *   scale_b = (max_i |x_i|) / qmax                       (binary32 division)
 *   q_i     = clamp(round_half_even(x_i / scale_b), -qmax, qmax); 0 if scale_b = 0
 *   x'_i    = (float)q_i * scale_b                       (binary32 product)
 * 4-bit codes are packed two per byte, element 2k in the low nibble. */
void zo_quantize_f32(const float* x, int64_t n, int bits, int64_t block,
                     uint8_t* q, float* scales);
void zo_dequantize_f32(const uint8_t* q, const float* scales, int64_t n, int bits,
                       int64_t block, float* out);
/* The same on 16-bit values (dtype 0 fp16, 1 bf16); dequantized values are
 * rounded to that 16-bit type. */
void zo_quantize_16(int dtype, const uint16_t* x, int64_t n, int bits, int64_t block,
                    uint8_t* q, float* scales);
void zo_dequantize_16(int dtype, const uint8_t* q, const float* scales, int64_t n, int bits,
                      int64_t block, uint16_t* out);
/* Gather of a unit from nd quantized shards: rank k's slice of the unit starts
 * at element `offset` of its shard; its codes and scales cover the whole shard
 * (blocks counted from the shard's start).  out[j] for j < len is element
 * offset + j % slice of rank j / slice's shard, dequantized. */
void zo_gather_unit_q(int dtype, int nd, int64_t len, int64_t slice, int64_t offset, int bits,
                      int64_t block, const uint8_t* const* q, const float* const* scales,
                      uint16_t* out);

/* ---- ZeRO-Offload ([L18] sec. 4.4: the fp32 master, m and v and the Adam
 *      update live on the host; each step moves the 16-bit gradients to the
 *      host, 2 Psi, and the 16-bit parameters back, 2 Psi; [ZL8] sec. 6.2, 7:
 *      the device runs forward and backward, the host the parameter update) --
 * The reduced gradient crosses the link in the 16-bit type: the rank-order
 * fp32 fold divided by nd is rounded to the 16-bit type (that is what is
 * copied), and the host unscales the copied value:
 *   g16[i] = to16(fold_i / nd);   g[i] = (float)g16[i] / loss_scale.
 * Returns 1 if any g[i] is inf or NaN.  grads: [nd][rank_stride]. */
int zo_reduce16(int nd, int64_t n, int dtype, const uint16_t* grads, int64_t rank_stride,
                float loss_scale, uint16_t* g16, float* g);
/* One offloaded step: zo_reduce16, then the norm, clip, skip decision and
 * Adam exactly as zo_step, on the host's master, m, v; params receives the
 * 16-bit parameters copied back to the device. */
int zo_step_offload(int nd, int64_t n, int dtype, const uint16_t* grads,
                    float* master, float* m, float* v, uint16_t* params,
                    const zo_hparams* hp, zo_scalars* st, zo_result* res);

/* ---- sharded checkpoint: ownership regrouped for another rank count
 *      ([Z026] sec. 5: restoring at a different degree of parallelism must
 *      reorganise which rank owns what while keeping the parameter order and
 *      each element's moments together; [L32] sec. 4.3: the checkpoint holds
 *      the sharded optimizer state) --------------------------------------------
 * A layout of psi flat elements over nd ranks: nunits units of len[u]
 * consecutive flat elements (stages 0-2: one unit, len[0] = psi; stage 3: the
 * ZeRO-3 units in order).  Unit u is cut into nd slices of
 * S_u = zo_shard_elems(len[u], nd) elements; rank r's shard is the
 * concatenation, in unit order, of element r*S_u .. (r+1)*S_u - 1 of every
 * unit (positions past len[u] are padding). */
typedef struct {
    int nd;
    int nunits;
    const int64_t* len;
} zo_layout;

/* elements of one rank's shard: the sum of the S_u */
int64_t zo_layout_shard_len(const zo_layout* L);
/* flat index held at position j of rank r's shard; -1 for padding */
int64_t zo_layout_global(const zo_layout* L, int r, int64_t j);
/* Regroup: old_shards[r] (layout A, elem_bytes-wide elements) -> new_shards[r]
 * (layout B): each position of B takes the element of A that holds the same
 * flat index; padding positions of B are zero.  Both layouts cover the same psi. */
void zo_reshard(const zo_layout* A, const void* const* old_shards, const zo_layout* B,
                void* const* new_shards, int elem_bytes);

#ifdef __cplusplus
}
#endif
#endif
