/*
 * zero_b200.h -- C ABI of libzero_b200: the ZeRO-DP sharded mixed-precision
 * optimizer step on one GPU (sm_103a), with Nd data-parallel ranks emulated in
 * that GPU's own memory.
 *
 * Pages cited (title as printed; section numbers are each page's own):
 *   [L18]  "第 18 讲 · Memory Optimization in Distributed Training: ZeRO"
 *   [Z026] "026｜ZeRO：数据并行中，没必要让每张卡保存全部训练状态"
 *   [L32]  "L3.2 显存优化与 ZeRO"
 *   [ZL8]  "图解分布式训练（八）—— ZeRO 学习"
 *   [PZ]   "ZeRO:" (ZeRO paper digest)
 *
 * One step, per element of the flat parameter vector ([L18] 2.2-2.4):
 *   (1) reduce-scatter: the Nd ranks' 16-bit local gradients are summed in
 *       fixed rank order (0..Nd-1, fp32, from 0.0f) and divided by Nd
 *       ([L18] 2.2, 2.5; [PZ] 5.2);
 *   (2) unscale by the loss scale; any inf/NaN sets the overflow flag, which
 *       under dynamic loss scaling skips the step and halves the scale
 *       ([L32] 4.3);
 *   (3) global gradient norm over every shard and clip-by-norm
 *       ([L32] 4.2 "gradient_clipping");
 *   (4) Adam / AdamW with bias correction on each shard's fp32 master, m, v
 *       ([L18] 2.1-2.2: Adam is elementwise, a rank needs only its slice);
 *   (5) cast to fp16/bf16 ([L18] 2.2);
 *   (6) all-gather of the 16-bit parameters: for ZeRO-1/2 every shard writes
 *       into one flat full-parameter buffer ([L18] 2.2; [L32] 2.3); for
 *       ZeRO-3 zero_gather_layer assembles one unit from its Nd slices
 *       ([L18] 2.4, 3.3; [ZL8] 8.4).
 *
 * Conventions for every entry point:
 *   - Errors: every call returns a zero_status_t and never aborts; arguments
 *     are validated before anything is launched.  CUDA failures return
 *     ZERO_ECUDA.  A skipped step is not an error.
 *   - Ownership: the caller allocates and owns every device buffer and the
 *     stream; the library borrows raw device pointers for the duration of a
 *     call.  A plan owns only its host bookkeeping and a small device block
 *     (optimizer scalars, step status, per-block partials: about 100 KB,
 *     allocated by zero_plan_create on the current device).
 *   - Device pointers must be 16-byte aligned.  Streams are cudaStream_t
 *     passed as void* (NULL = the legacy default stream).
 *   - Steps of one plan must be ordered (same stream, or ordered by events):
 *     they share the plan's device block.
 */
#ifndef ZERO_B200_H
#define ZERO_B200_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct zero_plan* zero_plan_t;

typedef enum {
    ZERO_OK       = 0,
    ZERO_EINVAL   = 1,   /* an argument is out of range, null or misaligned   */
    ZERO_ENOMEM   = 2,   /* host or device allocation failed                  */
    ZERO_ECUDA    = 3,   /* a CUDA call or kernel launch failed                */
    ZERO_ETIMEOUT = 4    /* a bounded device-side wait gave up                 */
} zero_status_t;

typedef enum { ZERO_FP16 = 0, ZERO_BF16 = 1 } zero_dtype_t;

/* Optimizer and mixed-precision settings ([L32] 3.2 and 4.2 DeepSpeed config:
 * optimizer lr, fp16 loss scaling, gradient_clipping).
 *   lr, beta1, beta2, eps    Adam; bias-corrected with 1 - beta^t.
 *   weight_decay             0 = none.  decoupled_wd = 1: AdamW, the master is
 *                            multiplied by (1 - lr wd) before the update;
 *                            0: L2, wd * master is added to the gradient.
 *   clip_norm                clip by global norm; 0 = off.
 *   loss_scale               initial loss scale S (the gradients arrive
 *                            multiplied by S); 1 = none.
 *   dynamic_scale            1: an overflow skips the step (state untouched,
 *                            t unchanged) and multiplies S by backoff; after
 *                            growth_interval good steps in a row S doubles
 *                            (growth_interval <= 0: never).  Requires fp16.
 *                            0: static S; the overflow flag is reported but
 *                            does not skip. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int   decoupled_wd;
    float clip_norm;
    float loss_scale;
    int   dynamic_scale;
    float backoff;
    int   growth_interval;
} zero_hparams_t;

/* ---- plans ------------------------------------------------------------ */

/* Create a plan for a model of psi parameters made of ntensors tensors whose
 * shapes are given in list order: tensor i has ndims[i] dimensions, taken in
 * order from dims.  psi must equal the sum of the tensor sizes.
 * nd: emulated data-parallel ranks (1..1024).  stage: 0 = plain DP, 1, 2, 3.
 * dtype: format of the gradients and of the 16-bit parameters.
 * Layout ([L18] 3.2 flat partition; [ZL8] 8.4):
 *   stages 0-2: all tensors flattened into one vector and split into nd equal
 *     contiguous shards of S = ceil(psi/nd) rounded up to 64 elements; rank r
 *     owns [r S, (r+1) S); the flat length is nd S (the tail is padding).
 *   stage 3: each ZeRO-3 unit (here: one unit per tensor; see
 *     zero_plan_create_units) is flattened and split into nd slices of
 *     S_u = ceil(len_u/nd) rounded up to 64; a rank's shard is the
 *     concatenation of its slice of every unit in unit order.
 * The plan copies everything it needs; dims/ndims/hp may be freed afterwards.
 * Allocates the plan's device block on the current device.
 * Errors: ZERO_EINVAL (bad sizes, psi mismatch, dynamic_scale with bf16,
 * nd or stage out of range), ZERO_ENOMEM, ZERO_ECUDA. */
zero_status_t zero_plan_create(uint64_t psi, int nd, int stage, zero_dtype_t dtype,
                               const int64_t* dims, const int* ndims, int ntensors,
                               const zero_hparams_t* hp, zero_plan_t* out);

/* As zero_plan_create, with the ZeRO-3 unit of each tensor given explicitly:
 * unit_of_tensor[i] is tensor i's unit; units are numbered 0..U-1 in the
 * order their tensors appear and each unit's tensors are contiguous in the
 * list (e.g. embedding, one unit per transformer layer, final norm + head:
 * [L18] 3.3 the FSDP unit is usually one Transformer layer).  Ignored for
 * stages 0-2. */
zero_status_t zero_plan_create_units(uint64_t psi, int nd, int stage, zero_dtype_t dtype,
                                     const int64_t* dims, const int* ndims, int ntensors,
                                     const int* unit_of_tensor, const zero_hparams_t* hp,
                                     zero_plan_t* out);

/* Free the plan and its device block.  NULL is accepted. */
zero_status_t zero_plan_destroy(zero_plan_t plan);

/* Layout of the buffers zero_step expects (any output pointer may be NULL):
 *   shard_elems     S (stages 0-2), or the length of one rank's shard (stage 3)
 *   padded_elems    stages 0-2: nd * S, the flat parameter/state length;
 *                   stage 3: one rank's shard length (= shard_elems)
 *   nunits          ZeRO-3 units (stage 3), else 0
 *   workspace_bytes device scratch zero_step needs (0 when none). */
zero_status_t zero_plan_layout(zero_plan_t plan, uint64_t* shard_elems, uint64_t* padded_elems,
                               int* nunits, uint64_t* workspace_bytes);

/* Stage 3: unit u's length, slice length S_u and the slice's offset inside a
 * rank's shard. */
zero_status_t zero_plan_unit(zero_plan_t plan, int unit, uint64_t* len, uint64_t* slice_elems,
                             uint64_t* offset);

/* ---- the step ----------------------------------------------------------- */

/* One optimizer step, asynchronous on `stream` (no host synchronisation).
 * Stages 0-2 (every emulated rank's shard is updated):
 *   grads      [nd][nd*S] 16-bit: rank r's full local gradient at
 *              grads + r*nd*S; elements at flat index >= psi are ignored.
 *   master,m,v [nd*S] fp32, updated in place (elements >= psi untouched).
 *   params     [nd*S] 16-bit flat full-parameter buffer: every shard's updated
 *              parameters are written at their flat offset (the all-gather
 *              write-back); elements >= psi untouched.
 * Stage 3 (one rank's shard is resident):
 *   grads      [nd][L] 16-bit, L = that rank's shard length: the nd ranks'
 *              contributions to that shard;
 *   master,m,v,params [L] that rank's shard.  The overflow flag and the norm
 *              cover the resident shard (the scalar all-reduce over ranks has
 *              a single participant here).
 * workspace: zero_plan_layout's workspace_bytes of device scratch (NULL when 0).
 * On a skipped step nothing but the plan's loss scale changes.
 * Errors: ZERO_EINVAL (null or misaligned pointer), ZERO_ECUDA. */
zero_status_t zero_step(zero_plan_t plan, const void* grads, float* master, float* m, float* v,
                        void* params, void* workspace, void* stream);

/* Wait for the plan's last step and report it (any pointer may be NULL):
 * skipped (1 if the overflow skipped it), grad_norm (global L2 norm of the
 * unscaled averaged gradient, before clipping), clip_coef (the factor applied,
 * 1 when not clipped), loss_scale (the scale the next step uses), t (completed
 * steps).  Before any step: skipped 0, grad_norm 0, clip_coef 1, the initial
 * loss scale and t = 0.  Errors: ZERO_EINVAL (null plan), ZERO_ECUDA. */
zero_status_t zero_step_result(zero_plan_t plan, int* skipped, double* grad_norm,
                               float* clip_coef, float* loss_scale, int64_t* t);

/* The overflow flag of the plan's last step (1 if any gradient element was
 * inf/NaN after unscaling); waits like zero_step_result. */
zero_status_t zero_step_overflow(zero_plan_t plan, int* overflow);

/* ---- ZeRO-3 gather ------------------------------------------------------ */

/* Assemble unit `unit` of a stage-3 plan ([L18] 2.4: the owners send their
 * pieces before the unit is used; [ZL8] 8.4: one contiguous buffer per
 * module).  shard_ptrs[k] (k < nd, host array of device pointers) is rank k's
 * whole 16-bit parameter shard; out receives the unit's len elements:
 * out[k*S_u + j] = shard_k[off_u + j] for k*S_u + j < len.  Asynchronous.
 * Errors: ZERO_EINVAL (not stage 3, unit out of range, null or misaligned
 * pointer), ZERO_ECUDA. */
zero_status_t zero_gather_layer(zero_plan_t plan, int unit, const void* const* shard_ptrs,
                                void* out, void* stream);

/* ---- constant-size gradient buckets ------------------------------------------ */

/* [L18] 2.3 (ZeRO-2: as soon as the backward pass has a segment's gradients they
 * are reduced to the segment's owner and dropped, so each rank keeps only a
 * buffer for the segment in flight; the segment reduces together are one
 * reduce-scatter) and [L18] 4.3 / [PZ] 6.2 (a constant-size buffer worked
 * through piece by piece instead of one flat buffer that grows with the model).
 * A bucketed step takes the ranks' gradients bucket by bucket: bucket b covers
 * elements [b*B, min((b+1)*B, n)) of the flat vector (stage 3: of the resident
 * shard), B = bucket_elems (a multiple of 64).
 *   zero_plan_set_bucket   turns bucketed steps on (B > 0) or off (B = 0) and
 *                          reports the workspace they need: the fp32 reduced
 *                          gradient (n floats) plus one norm partial and one
 *                          flag per bucket.  Waits for the plan's last step.
 *   zero_step_bucket       reduces bucket b: bucket_grads is [nd][B] 16-bit
 *                          (rank stride B; a short last bucket uses its first
 *                          count columns); buckets may come in any order, each
 *                          exactly once per step (ZERO_EINVAL otherwise); the
 *                          bucket buffer may be reused once this call's work
 *                          on `stream` is done.
 *   zero_step_apply        after every bucket: the global norm from the bucket
 *                          partials (summed in bucket order), clip, skip
 *                          decision, Adam, cast, write-back; ZERO_EINVAL if a
 *                          bucket is missing.  zero_step_result reports it.
 * Reduced gradients are bit-identical to zero_step's; the norm agrees to
 * 1e-5 (its partial sums are grouped by bucket).  Calls of one plan must be
 * ordered on one stream. */
zero_status_t zero_plan_set_bucket(zero_plan_t plan, uint64_t bucket_elems,
                                   uint64_t* workspace_bytes);
zero_status_t zero_step_bucket(zero_plan_t plan, uint64_t bucket, const void* bucket_grads,
                               void* workspace, void* stream);
zero_status_t zero_step_apply(zero_plan_t plan, float* master, float* m, float* v, void* params,
                              void* workspace, void* stream);

/* ---- ZeRO++ quantized weight gather (qwZ) ---------------------------------- */

/* [L18] 4.5 ZeRO++: the parameters a ZeRO-3 gather moves are quantized block
 * by block, one scale per block, so a few large weights coarsen only their own
 * block.  A rank's 16-bit shard of n elements is cut into blocks of 256
 * elements counted from the shard's start; for each block
 *   scale = max|x| / qmax  (qmax = 127 for bits = 8, 7 for bits = 4; binary32)
 *   code  = round_half_even(x / scale) clamped to [-qmax, qmax]; 0 if scale = 0.
 * codes: n bytes (bits 8, two's complement) or ceil(n/2) bytes (bits 4, two
 * codes per byte, the even element in the low nibble), 16-byte aligned;
 * scales: ceil(n/256) floats.  Asynchronous.  Errors: ZERO_EINVAL, ZERO_ECUDA. */
zero_status_t zero_quantize_shard(zero_dtype_t dtype, const void* shard, uint64_t n, int bits,
                                  void* codes, float* scales, void* stream);

/* The ZeRO-3 gather of unit `unit` from the nd ranks' quantized shards
 * (code_ptrs[k], scale_ptrs[k]: rank k's whole-shard codes and scales, as
 * zero_quantize_shard writes them): out[k*S_u + j] = 16-bit rounding of
 * code_k[off_u + j] * scale_k[(off_u + j) / 256] for k*S_u + j < len.  Moves
 * 1 (bits 8) or 0.5 (bits 4) bytes per element in instead of 2.  Errors:
 * ZERO_EINVAL (not stage 3, unit or bits out of range, null or misaligned
 * pointer), ZERO_ECUDA. */
zero_status_t zero_gather_layer_q(zero_plan_t plan, int unit, int bits,
                                  const void* const* code_ptrs, const float* const* scale_ptrs,
                                  void* out, void* stream);

/* ---- gradient norm without allocating ------------------------------------ */

/* No counterpart on the pages: a convenience for callers that may not
 * allocate device memory (code running under another framework's memory pool
 * or allocator hooks, or code that only holds pre-allocated buffers and so
 * cannot create a plan, whose creation allocates).
 * Computes what zero_step's reduce pass reports: the global L2 norm of the
 * averaged, unscaled gradient g_i = (sum_r grads[r][i] / nd) / loss_scale (the
 * sum in rank order, fp32) and whether any g_i is inf/NaN.
 *   grads        [nd][rank_stride] 16-bit device array, 16-byte aligned; the
 *                first n elements of each rank's row are used.
 *   rank_stride  >= n, a multiple of 8.
 *   norm_out     device pointer to one double (8-byte aligned): the norm.
 *   overflow_out device pointer to one int: 1 if any g_i is inf/NaN, else 0.
 * Asynchronous on `stream`.  Allocates nothing: its scratch (one partial per
 * 2^17-element tile plus a counter, 196,864 bytes) is a fixed device array in
 * the library that every GPU loading the library keeps until process exit;
 * hence n is limited to 2^31 elements (ZERO_EINVAL beyond).  The first call on
 * a device looks up that array's device address (cudaGetSymbolAddress); make
 * the first call on each device before any stream capture.  Every call shares
 * the array, so calls whose executions overlap on the GPU (e.g. on two
 * concurrent streams) race and give wrong results; order them.  The norm
 * agrees with zero_step's within 1e-5 relative (the partial sums are grouped
 * differently); the flag is identical.
 * Errors: ZERO_EINVAL (sizes, alignment, null output), ZERO_ECUDA. */
zero_status_t zero_grad_norm_noalloc(const void* grads, int nd, uint64_t n, uint64_t rank_stride,
                                     zero_dtype_t dtype, float loss_scale, double* norm_out,
                                     int* overflow_out, void* stream);

/* ---- memory ledger and communication volume ------------------------------- */

/* Bytes of model state one rank holds ([L18] 1.2, 2.1; [Z026] 2; [L32] 2.1,
 * 2.3): K bytes of optimizer state per parameter (12 for Adam; 16 in the
 * slides' count that keeps an fp32 gradient) plus 2 + 2 for the 16-bit
 * parameters and gradients:
 *   stage 0 (4+K) psi;  1: 4 psi + K psi/nd;  2: 2 psi + (2+K) psi/nd;
 *   stage 3 (4+K) psi/nd.  Divisions round up.  0 on invalid arguments. */
uint64_t zero_state_bytes(uint64_t psi, uint64_t nd, int stage, int K);

/* Elements each rank sends per step ([L18] 3.1; [L32] 2.3; [PZ] 0x07):
 * stages 0-2: 2 psi (reduce-scatter + all-gather); stage 3: 3 psi (the
 * parameters are gathered again for the backward pass).  exact = 1 keeps
 * only the (nd - 1)/nd share that is not already local (rounded up).
 * 0 on invalid arguments. */
uint64_t zero_comm_volume(uint64_t psi, uint64_t nd, int stage, int exact);

/* Largest psi whose model state fits in mem_bytes per rank ([L18] 2.6). */
uint64_t zero_max_params(uint64_t mem_bytes, uint64_t nd, int stage, int K);

/* ---- diagnostics ----------------------------------------------------------- */

/* Static string naming a status code. */
const char* zero_status_string(zero_status_t status);

/* Per-kernel timing: when enabled, zero_step records CUDA events around each
 * of its kernels on the step's stream; zero_plan_kernel_times waits for the
 * last step and returns the accumulated milliseconds of the reduce pass
 * (pass 1, or the fused pass), of the update pass (0 for the fused path), the
 * number of timed steps and the number of kernels the plan has launched.
 * enable = 0 turns timing off; enable = 1 also clears the accumulators. */
zero_status_t zero_plan_profile(zero_plan_t plan, int enable);
zero_status_t zero_plan_kernel_times(zero_plan_t plan, double* reduce_ms, double* update_ms,
                                     int64_t* steps, int64_t* launches);

/* Which kernel path the plan runs: 0 = fused single pass (no clip, no dynamic
 * scale), 1 = two passes through an fp32 gradient in the workspace, 2 = two
 * passes that re-read the 16-bit gradients (clip or dynamic scale, nd < 4). */
int zero_plan_path(zero_plan_t plan);

/* Which kernel runs the reduce pass of a two-pass plan: 0 = 128-bit loads of
 * the rank rows (the default, measured fastest at nd = 16), 1 = TMA bulk
 * staging (cp.async.bulk of each rank's 2 KB row slice into a ring of shared-
 * memory stages, a producer warp and eight consumer warps).  Both compute the
 * same reduced gradient bit for bit; the norm's partial sums are grouped
 * differently.  Kind 1 needs the two-pass path with the fp32 workspace and
 * 4 <= nd <= 48 (ZERO_EINVAL otherwise).  Waits for the plan's last step.
 * A bounded wait in kind 1 that gives up makes zero_step_result return
 * ZERO_ETIMEOUT from then on. */
zero_status_t zero_plan_set_reduce_kernel(zero_plan_t plan, int kind);

#ifdef __cplusplus
}
#endif
#endif
