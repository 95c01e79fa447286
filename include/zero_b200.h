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
 *       ([L32] 4.3), and under a static scale skips it when the caller asks
 *       (zero_hparams_t.skip_on_overflow);
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

/* Every entry point reports through its return value and never throws: a C++
 * exception inside the library (a host allocation or a worker thread that
 * cannot be had) comes back as ZERO_ENOMEM, or ZERO_EIO inside checkpoint IO. */
typedef enum {
    ZERO_OK       = 0,
    ZERO_EINVAL   = 1,   /* an argument is out of range, null or misaligned   */
    ZERO_ENOMEM   = 2,   /* host or device allocation failed                  */
    ZERO_ECUDA    = 3,   /* a CUDA call or kernel launch failed                */
    ZERO_ETIMEOUT = 4,   /* a bounded device-side wait gave up                 */
    ZERO_ENOENT   = 5,   /* a checkpoint file is missing or cannot be opened   */
    ZERO_ECORRUPT = 6,   /* a checkpoint file is truncated, fails a checksum,
                            or does not belong with the other files           */
    ZERO_EIO      = 7,   /* reading, writing or flushing a file failed         */
    ZERO_ESTATE   = 8    /* a failed checkpoint load left the plan's state
                            incomplete; steps are refused until a load succeeds */
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
 *                            0: static S (see skip_on_overflow).
 *   skip_on_overflow         with a static S: 1 = an overflow skips the step
 *                            (state untouched, t and S unchanged); 0 = the
 *                            flag is reported and the step goes ahead.
 *                            Ignored under dynamic_scale (which always skips).
 *
 * Overflow under a static scale (dynamic_scale 0, skip_on_overflow 0): the
 * skip belongs to loss scaling ([L32] 4.3 ties a NaN loss to the fp16
 * loss_scale setting), and a step that nothing global gates is what lets the
 * update run as one fused pass over the data.  The consequences of a non-finite
 * averaged gradient element i in such a step:
 *   - without clipping, only element i is affected: its master, m and v
 *     become NaN (or inf) and stay so; every other element is updated exactly
 *     as if element i's gradient had been finite;
 *   - with clipping, the norm is inf, the clip coefficient tau/inf = 0, so
 *     every finite element takes a zero-gradient step (m *= beta1,
 *     v *= beta2, the master moves by the remaining momentum) and element i
 *     becomes NaN (inf * 0).
 * A caller who wants such steps dropped sets skip_on_overflow = 1; the plan
 * then runs two passes (the flag must be known before any update), which
 * costs the fp32 gradient's write and read (8 bytes per element) on the
 * paths that would otherwise fuse. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int   decoupled_wd;
    float clip_norm;
    float loss_scale;
    int   dynamic_scale;
    float backoff;
    int   growth_interval;
    int   skip_on_overflow;
} zero_hparams_t;

/* ---- plans ------------------------------------------------------------ */

/* Largest psi a plan accepts (2^48 elements): far above any GPU's memory, and
 * small enough that every element index times nd fits the kernels' 64-bit
 * arithmetic. */
#define ZERO_MAX_PSI (1ull << 48)

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
 * Errors: ZERO_EINVAL (bad sizes, psi mismatch, psi > ZERO_MAX_PSI,
 * dynamic_scale with bf16, nd or stage out of range), ZERO_ENOMEM, ZERO_ECUDA. */
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
 * grads may also lie in page-locked host memory that the device can address
 * (cudaHostAlloc, or cudaHostRegister; under unified addressing the host address
 * is the device address): the passes then read it in place over the host link,
 * with the same results; the caller must not rewrite it before the step is done
 * (zero_step_result waits for it).  Every other buffer is device memory.
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
 *                          flag per block of each bucket's reduce.  Waits for
 *                          the plan's last step.
 *   zero_step_bucket       reduces bucket b: bucket_grads is [nd][B] 16-bit
 *                          (rank stride B; a short last bucket uses its first
 *                          count columns); buckets may come in any order, each
 *                          exactly once per step (ZERO_EINVAL otherwise); the
 *                          bucket buffer may be reused once this call's work
 *                          on `stream` is done.
 *   zero_step_apply        after every bucket: the global norm from the bucket
 *                          reduces' block partials (summed in bucket, then
 *                          block, order), clip, skip decision, Adam, cast,
 *                          write-back; ZERO_EINVAL if a bucket is missing.
 *                          zero_step_result reports it.
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

/* One ZeRO-3 optimizer step (exactly zero_step's, same arguments) whose update
 * pass also quantizes the resident shard's updated 16-bit parameters for the
 * qwZ gather ([L18] 4.5): codes and scales receive what
 * zero_quantize_shard(dtype, params, L, bits, codes, scales) would write after
 * the step, L being the shard length, but the parameters are quantized from
 * the update's registers as they are written instead of being read back
 * (2 bytes per element and one launch saved).  On a skipped step the
 * unchanged parameters are quantized, so the codes are valid whatever the
 * buffers held.  codes: L bytes (bits 8) or L/2 bytes (bits 4), 16-byte
 * aligned; scales: ceil(L/256) floats.  Asynchronous.  Errors: ZERO_EINVAL
 * (not stage 3, bits not 4 or 8, null or misaligned pointer), ZERO_ESTATE,
 * ZERO_ECUDA. */
zero_status_t zero_step_qwz(zero_plan_t plan, const void* grads, float* master, float* m, float* v,
                            void* params, void* workspace, int bits, void* codes, float* scales,
                            void* stream);

/* ---- ping-pong step ------------------------------------------------------- */

/* One optimizer step as a single pass over the data even when an overflow may
 * skip it (dynamic loss scaling or skip_on_overflow, without a clip): the
 * caller keeps two sets of master, m, v; the step reads the current set and
 * writes the other, and only a step that is not skipped makes the other set
 * current, so a skipped step leaves the current state untouched without having
 * to know the overflow before the update.  The 16-bit parameters are written by
 * the pass; when the step is skipped, a small pass after it rewrites them from
 * the current set's master (4 + 2 bytes per element, on skipped steps only).
 * The arithmetic is zero_step's: the same state, parameters and report.
 *   set 0: master0, m0, v0; set 1: master1, m1, v1; each laid out as zero_step's
 *          master, m, v (stages 0-2: [nd*S]; stage 3: the resident shard).
 *   grads, params: as zero_step.
 * zero_plan_state_set reports which set is current after the plan's last step
 * (waiting for it): 0 after zero_plan_create and after zero_checkpoint_load
 * (load a checkpoint into set 0); checkpoint the current set.  A plan may mix
 * zero_step and zero_step_pingpong only if the caller passes the current set
 * to zero_step.  Asynchronous.  Errors: ZERO_EINVAL (clip_norm > 0, null or
 * misaligned pointer), ZERO_ESTATE, ZERO_ECUDA. */
zero_status_t zero_step_pingpong(zero_plan_t plan, const void* grads, float* master0, float* m0,
                                 float* v0, float* master1, float* m1, float* v1, void* params,
                                 void* stream);
zero_status_t zero_plan_state_set(zero_plan_t plan, int* set);

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
 * a device looks up that array's device address (cudaGetSymbolAddress) and
 * keeps it per device context: after the device's primary context is reset
 * (cudaDeviceReset), the next call looks it up again.  Every call shares
 * the array, so calls whose executions overlap on the GPU (e.g. on two
 * concurrent streams) race and give wrong results; order them.  The norm
 * agrees with zero_step's within 1e-5 relative (the partial sums are grouped
 * differently); the flag is identical.
 * Errors: ZERO_EINVAL (sizes, alignment, null output), ZERO_ECUDA. */
zero_status_t zero_grad_norm_noalloc(const void* grads, int nd, uint64_t n, uint64_t rank_stride,
                                     zero_dtype_t dtype, float loss_scale, double* norm_out,
                                     int* overflow_out, void* stream);

/* ---- sharded checkpoint ------------------------------------------------------ */
/* [Z026] sec. 5: with the state sharded, each rank holds only its part of the
 * weights and optimizer state; a restore at another degree of parallelism
 * must regroup ownership while keeping the parameter order and each
 * element's moments together, and a rank's missing file must make the
 * restore fail explicitly rather than produce an incomplete model.
 * [L32] sec. 4.3: a resumable checkpoint holds the sharded optimizer state,
 * not the weights alone.
 *
 * A checkpoint is a directory holding manifest.zck and one file per rank of
 * the saving plan, shard_<rank>_of_<nd>.zck (5-digit decimal, zero-padded).
 * Each rank file holds, for the flat elements that rank owns (padding
 * excluded): master, m and v (fp32) and the 16-bit parameters.  The file
 * records those elements as segments [global_start, global_start + count) of
 * the flat parameter vector, so a checkpoint does not depend on the saving
 * plan's rank count or stage: a plan of any nd and stage over the same tensor
 * list can load it, each of its ranks taking the elements it owns.
 *
 * Format (all integers little-endian):
 *   manifest.zck, 88 bytes: "ZEROMAN1", u32 version (1), u32 size (88),
 *     u64 psi, i32 nd, i32 stage, i32 dtype, i32 0, u64 model_hash,
 *     scalars (32 bytes: f32 loss_scale, i32 good_steps, i64 t, f64 beta1^t,
 *     f64 beta2^t), u64 zck64 of bytes 0..79.
 *   shard file: a 4096-byte header: "ZEROSHD1", u32 version (1),
 *     u32 4096, u64 psi, i32 nd, i32 stage, i32 dtype, i32 rank,
 *     u64 model_hash, scalars (32 bytes, as above), u64 nseg, u64 n (elements
 *     held = sum of the segment counts), u64 block_elems (2^20), u64 nblocks
 *     (ceil(n / block_elems)), u64 table_offset (4096), u64 array_offset[4]
 *     (master, m, v, params), u64 file_bytes, u64 meta_hash; zeros up to 4096.
 *     At table_offset: nseg pairs {u64 global_start, u64 count} in shard
 *     order, then 4 x nblocks u64 block checksums (array a, block b at
 *     a * nblocks + b).  Each array holds its n values in segment order and
 *     starts on a 4096-byte boundary.  meta_hash = zck64 of header bytes
 *     0..159 plus zck64 of the table, mod 2^64.
 *   zck64 of a byte string whose first 8-byte word has index w0 within its
 *     array: the sum mod 2^64, over its 8-byte words x_i (the last one
 *     zero-padded), of mix(x_i + (w0 + i + 1) * 0x9E3779B97F4A7C15), where
 *     mix is the SplitMix64 finaliser (z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *     z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31).  Block b of an
 *     array covers elements [b * 2^20, min((b + 1) * 2^20, n)), w0 = its byte
 *     offset / 8.
 *   model_hash: FNV-1a 64 over the little-endian bytes of the int64 values
 *     ntensors, then for each tensor its ndims and its dims.
 */

/* flags of zero_checkpoint_save */
#define ZERO_CKPT_FSYNC      1   /* flush every file and the directory to storage  */
#define ZERO_CKPT_DROP_CACHE 2   /* with FSYNC: then drop the files' cached pages  */

/* Save rank `rank`'s state, or every rank's (rank = -1; stages 0-2 only).
 * Buffers: as zero_step.  Stages 0-2: the flat [nd*S] master, m, v, params;
 * stage 3: rank `rank`'s resident shard.  Writes shard_<rank>_of_<nd>.zck
 * (through a temporary name, renamed when complete) for each rank saved, and
 * manifest.zck when rank is 0 or -1, creating `dir` if it does not exist.
 * The scalars (loss scale, good steps, t, beta powers) are the plan's after
 * its last step.  Synchronous: waits for `stream` and the plan's last step,
 * returns when the files are written.  Host staging is pinned memory the plan
 * keeps until it is destroyed.
 * Errors: ZERO_EINVAL (null, misaligned or out-of-range argument), ZERO_EIO
 * (a file could not be created, written or flushed; no partial file is left
 * under the final name), ZERO_ENOMEM, ZERO_ECUDA. */
zero_status_t zero_checkpoint_save(zero_plan_t plan, const char* dir, int rank,
                                   const float* master, const float* m, const float* v,
                                   const void* params, int flags, void* stream);

/* Load rank `rank`'s state, or every rank's (rank = -1; stages 0-2 only), from
 * the checkpoint in `dir`, whatever rank count and stage saved it; the
 * elements of the plan's layout past each unit's or the model's end are set
 * to zero.  Buffers: as zero_checkpoint_save.  On success the plan's scalars
 * are the checkpoint's and its last-step report is reset.  Synchronous.
 * Checks, before any device memory is written: the manifest and every one of
 * the saving plan's rank files exist (ZERO_ENOENT), their headers are intact
 * and agree with each other, their segments cover the flat vector exactly once
 * (ZERO_ECORRUPT), and the model is the plan's: same psi, tensor shape list
 * and 16-bit type (ZERO_EINVAL); the buffers are then untouched.  Every data
 * block read is checked against its checksum; a mismatch or read error after
 * device writes began returns ZERO_ECORRUPT or ZERO_EIO and leaves the plan
 * refusing steps and gathers (ZERO_ESTATE) until a load succeeds.
 * Other errors: ZERO_ENOMEM, ZERO_ECUDA. */
zero_status_t zero_checkpoint_load(zero_plan_t plan, const char* dir, int rank, float* master,
                                   float* m, float* v, void* params, void* stream);

/* ---- ZeRO-Offload: the Adam update on the host ------------------------------- */
/* [L18] sec. 4.4: the device keeps the 16-bit parameters and gradients; the
 * host keeps the fp32 master, m and v and runs Adam, multithreaded and
 * vectorised; each step copies the 16-bit gradients to the host (2 psi bytes)
 * and the updated 16-bit parameters back (2 psi).  [ZL8] sec. 6.2, 7: the
 * device runs forward and backward, the host the parameter update. */

/* One offloaded step of a stages 0-2 plan.  On the device: the rank-order fp32
 * fold of the nd contributions divided by nd, rounded to the plan's 16-bit
 * type (the copied value; written to `workspace`), the overflow flag and the
 * global norm of that value divided by the loss scale, and the step's
 * scalars (skip, clip coefficient, loss-scale update, t, bias corrections), as
 * zero_step.  On the host, unless the step is skipped: g = copied value / S,
 * times the clip coefficient, then Adam/AdamW on master, m, v exactly as
 * zero_step's update, and the 16-bit parameters copied to `params`.
 *   grads      device [nd][nd*S] 16-bit, as zero_step.
 *   master,m,v HOST fp32 arrays of at least psi elements (elements >= psi
 *              untouched); pageable or pinned.
 *   params     device [nd*S] 16-bit flat parameters (elements >= psi untouched).
 *   workspace  device scratch of at least 2*psi bytes, 16-byte aligned.
 *   nthreads   host threads (<= 0: one per hardware thread).
 * The copies stream through the plan's pinned staging in 2^24-element chunks
 * overlapped with the host arithmetic.  Synchronous: returns when the
 * parameters are on the device.  zero_step_result reports the step.
 * Errors: ZERO_EINVAL (stage 3, null or misaligned pointer), ZERO_ESTATE,
 * ZERO_ENOMEM, ZERO_ECUDA. */
zero_status_t zero_offload_step(zero_plan_t plan, const void* grads, float* master, float* m,
                                float* v, void* params, void* workspace, int nthreads,
                                void* stream);

/* The host Adam alone, on host memory: for i < n, g = grads16[i] (the 16-bit
 * type `dtype`) / loss_scale * clip_coef, then Adam/AdamW with the bias
 * corrections bc1 = 1 - beta1^t and bc2 = 1 - beta2^t of this step, each
 * operation one binary32 rounding in the order of zero_step's update; master,
 * m, v updated in place, params16[i] = master[i] rounded to the 16-bit type.
 * nthreads <= 0: one thread per hardware thread.  Needs no GPU.
 * Errors: ZERO_EINVAL (null pointer, dtype, loss_scale/bc1/bc2 not > 0),
 * ZERO_ENOMEM. */
zero_status_t zero_cpu_adam(const void* grads16, zero_dtype_t dtype, uint64_t n, float loss_scale,
                            float clip_coef, float bc1, float bc2, const zero_hparams_t* hp,
                            float* master, float* m, float* v, void* params16, int nthreads);

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
 * scale, no skip_on_overflow), 1 = two passes through an fp32 gradient in the
 * workspace, 2 = two passes that re-read the 16-bit gradients (clip, dynamic
 * scale or skip_on_overflow, nd < 4). */
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
