/*
 * zero_step.h - C ABI of the GB300 ZeRO-1/2 mixed-precision AdamW step.
 *
 * One optimizer step of data-parallel training with ZeRO stage 1 or 2,
 * with R data-parallel ranks emulated as R separate buffers in one GPU's
 * memory:
 *
 *   1. reduce-scatter + average: rank r owns shard r of the flat parameter
 *      vector and receives the fp32 sum, in fixed rank order, of every
 *      rank's bf16 gradients (each rank first accumulates its M
 *      micro-batches), divided by R*M;
 *   2. AdamW on the owned shard of the fp32 master weights and moments;
 *   3. cast to bf16 and all-gather into every rank's full replica.
 *
 * Sources (lecture pages on distributed training):
 *   - gradient accumulation g = (1/M) sum_j grad_j: CS25 V6 Lecture 4 notes,
 *     "single-GPU baseline and gradient accumulation";
 *     LLM infra 06 (3D parallelism), section 7.2
 *   - DP averaging g = (1/P) sum_r g_r: CS25 V6 Lecture 4 notes, "replicate
 *     the model, split the batch"; CS324 Lecture 9 notes, section 3.1
 *   - ZeRO-1 / ZeRO-2 (shard the optimizer state, then the gradients; each
 *     rank updates its shard; all-gather the new parameters): CS25 V6
 *     Lecture 4 notes, "ZeRO-1" and "ZeRO-2"; CS324 Lecture 9 notes,
 *     section 3.4; CS336 Lecture 7 summary, Q2
 *   - reduce-scatter / all-gather semantics: CS336 Lecture 7 book,
 *     sections 2.3 and 4.3 (reduce_scatter_tensor, all_gather_into_tensor);
 *     LLM infra 06, section 2.0
 *   - 16 bytes/param state (bf16 param + bf16 grad + fp32 master, m, v):
 *     CS324 Lecture 9 notes, section 2.1; CS336 Lecture 7 summary, Q3
 *   - fp32 reduction of gradients: LLM infra 06, section 15.3
 *
 * Arithmetic (the pages leave it open; this library fixes it and the CPU
 * oracle in the repository follows the same definition):
 *   acc_r = G[r][0][i] + G[r][1][i] + ... (fp32, micro-batches ascending)
 *   acc   = acc_0 + acc_1 + ... + acc_{R-1} (fp32, ranks ascending)
 *   g     = acc / (float)(R*M)              (IEEE division)
 *   torch.optim.AdamW's algorithm, every float operation rounded on its own
 *   (no fused multiply-add):
 *   w = W[i]*(1-lr*wd); m = b1*m + (1-b1)*g; v = b2*v + ((1-b2)*g)*g;
 *   W[i] = w - (lr/(1-b1^t)) * (m / (sqrt(v)/sqrt(1-b2^t) + eps));
 *   P[r][i] = bf16(W[i]) for every r (round to nearest even; every NaN
 *   becomes 0x7FC0).  The scalars lr/(1-b1^t), sqrt(1-b2^t), 1-lr*wd, 1-b1
 *   and 1-b2 are computed once per step in double and rounded to float.
 *
 * Conventions for every entry point:
 *   - Returns a zero_status; ZERO_OK (0) on success.  Argument, plan,
 *     alignment, size and overlap errors are returned synchronously and
 *     nothing is launched.  ZERO_ERR_CUDA means a launch or copy failed
 *     (cudaGetLastError after the launches).  Conditions found on the device
 *     are OR-ed into an optional caller-owned device status word.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and is asynchronous with respect to the host.
 *   - The caller allocates and owns every device buffer (PyTorch in the
 *     bundled binding).  The library allocates only the host-side plan.
 *   - bf16 buffers are passed as uint16_t* (raw bf16 bits).  Device buffers
 *     must be 16-byte aligned.
 *   - No exceptions and no global state cross the ABI; entry points are
 *     thread-safe for distinct buffers.
 *   - A plan with N = 0 is a no-op for the step entry points: once the
 *     plan, hyper-parameters, flags and scalar arguments have passed their
 *     checks, the call returns ZERO_OK without reading a buffer pointer,
 *     launching anything or writing dev_status / dev_sumsq.  (The one
 *     exception: zero_step_onebit checks its residual pointers first.)
 */
#ifndef ZERO_STEP_H
#define ZERO_STEP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZERO_ABI_VERSION 1
#define ZERO_MAX_R 64        /* emulated ranks */
#define ZERO_MAX_RM 256      /* gradient buffers (ranks x micro-batches) */

typedef enum {
    ZERO_OK = 0,
    ZERO_ERR_INVALID_ARG = -1,     /* R, M, stage, step, variant, hparams, ... */
    ZERO_ERR_NULL = -2,            /* a required pointer is NULL              */
    ZERO_ERR_ALIGN = -3,           /* a device pointer is not 16-byte aligned  */
    ZERO_ERR_SIZE = -4,            /* sizes beyond the limits / scratch too small */
    ZERO_ERR_OVERLAP = -5,         /* an output overlaps another buffer        */
    ZERO_ERR_CUDA = -6,            /* a CUDA launch or copy failed             */
    ZERO_ERR_DEVICE_TIMEOUT = -7,  /* a bounded device wait ran out (zero_get_device_status) */
    ZERO_ERR_NONFINITE = -8,       /* a non-finite gradient or norm (zero_get_device_status) */
    ZERO_ERR_IO = -9,              /* a checkpoint file could not be written/read */
    ZERO_ERR_CORRUPT = -10         /* a checkpoint header or checksum is wrong  */
} zero_status;

/* Bits OR-ed into the optional device status word. */
#define ZERO_DEV_NONFINITE 1       /* an averaged gradient (or the norm) was Inf or NaN */
#define ZERO_DEV_TIMEOUT 2         /* a bounded device wait ran out (TMA variant) */
#define ZERO_DEV_SKIPPED 4         /* zero_step_clipped skipped the update      */
/* Set with ZERO_DEV_TIMEOUT when, after a wait ran out, the block's own
 * bounded wait for the copies it had already issued ran out as well: the
 * block left with copies in flight into its shared memory, so treat the CUDA
 * context as suspect (finish or reset it) rather than continue training. */
#define ZERO_DEV_DRAIN_FAILED 8

/* Flags for zero_step / zero_rs_avg. */
#define ZERO_FLAG_CHECK_FINITE 1   /* set ZERO_DEV_NONFINITE when g is non-finite */
#define ZERO_FLAG_SKIP_NONFINITE 2 /* zero_step_clipped: skip the update on a non-finite norm */
/* Test-only, ZERO_VARIANT_FUSED_TMA: every bounded device wait gives up at
 * once, so the timeout path runs: the kernel drains its copies, sets
 * ZERO_DEV_TIMEOUT and returns without updating anything it had not
 * reached.  Needs dev_status. */
#define ZERO_FLAG_DEBUG_EXPIRE_WAITS (1 << 30)

/* Variants for zero_step. */
#define ZERO_VARIANT_FUSED 0       /* one pass: rs -> adamw -> ag per element  */
#define ZERO_VARIANT_STAGED 1      /* rs_avg, adamw_shard, ag_cast, fp32 g in scratch */
#define ZERO_VARIANT_FUSED_TMA 2   /* one pass, tiles staged by TMA bulk copies (R*M <= 16) */
#define ZERO_TMA_MAX_RM 16

/*
 * Shard layout of a flat parameter vector (the tensors concatenated in the
 * given order, no per-tensor padding): N = sum of numels,
 * S = roundup(ceil(N / R), align_elems), owner(i) = i / S.  The fp32 state
 * arrays (master, m, v) hold padded = R*S floats with shard r at offset r*S,
 * so element i lives at index i; pad elements [N, R*S) are never read or
 * written.  Replicas and gradient buffers hold exactly N elements.
 * Byte accounting per rank (CS25 V6 Lecture 4 notes, ZeRO-1/ZeRO-2 memory
 * equations; CS324 Lecture 9 notes, exercise 1), with b_p = b_g = 2 bytes
 * (bf16) and b_o = 12 bytes (fp32 master, m, v), sharded parts counted with
 * the padded shard S:
 *   dp = N(b_p + b_g + b_o); z1 = N(b_p + b_g) + S b_o;
 *   z2 = N b_p + S(b_g + b_o); z3 = S(b_p + b_g + b_o).
 */
typedef struct {
    int64_t N;                     /* real parameter count                     */
    int64_t S;                     /* shard length (elements)                  */
    int64_t padded;                /* R * S                                    */
    int32_t R, M;                  /* ranks, micro-batches                     */
    int32_t stage;                 /* 1 or 2 (same numbers; accounting only)   */
    int32_t align_elems;           /* shard alignment, a multiple of 4         */
    int32_t n_tensors;
    const int64_t* tensor_offsets; /* n_tensors + 1 entries, owned by the plan */
    int64_t bytes_per_rank_dp, bytes_per_rank_z1, bytes_per_rank_z2, bytes_per_rank_z3;
    int64_t bytes_per_rank;        /* the one for `stage`                      */
    int64_t scratch_bytes_staged;  /* scratch the staged variant needs: 4*R*S  */
} zero_plan_t;

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
} zero_adamw_hparams;

/* ABI version (ZERO_ABI_VERSION). */
int32_t zero_abi_version(void);

/* Static, human-readable name of a status code. */
const char* zero_status_string(zero_status s);

/*
 * Build the shard layout for n_tensors tensors of the given element counts
 * (host array, read only), R ranks (1..ZERO_MAX_R), M micro-batches
 * (R*M <= ZERO_MAX_RM), ZeRO stage 1 or 2, shard alignment align_elems
 * (0 -> 64; otherwise a positive multiple of 4).  Host only: needs no GPU.
 * On success *out owns a new plan (free with zero_plan_destroy).
 * Errors: ZERO_ERR_NULL, ZERO_ERR_INVALID_ARG (a negative numel, R, M,
 * stage or alignment out of range), ZERO_ERR_SIZE (N overflows).
 */
zero_status zero_plan_create(const int64_t* tensor_numels, int32_t n_tensors, int32_t R,
                             int32_t M, int32_t stage, int32_t align_elems, zero_plan_t** out);

/* Free a plan (NULL is ignored). */
void zero_plan_destroy(zero_plan_t* plan);

/* Rank owning element i (i / S), or -1 if i is outside [0, N). */
int32_t zero_plan_owner(const zero_plan_t* plan, int64_t i);

/*
 * One optimizer step (see the top of this file for the arithmetic).
 *   rank_grads  host array of R*M device pointers, entry r*M + j = rank r,
 *               micro-batch j; each N bf16, read only (entries may alias
 *               one another), except in the staged ZeRO-2 mode without
 *               scratch described under `scratch`.
 *   master, m, v  device, plan->padded floats each, updated in place.
 *   rank_params host array of R device pointers, each N bf16, written.
 *   hp          AdamW hyper-parameters (0 <= beta1, beta2 < 1; lr, eps,
 *               weight_decay finite; eps >= 0).
 *   step        the step count t >= 1 used for bias correction.
 *   variant     ZERO_VARIANT_FUSED, ZERO_VARIANT_STAGED, or
 *               ZERO_VARIANT_FUSED_TMA (the fused pass with each tile's
 *               gradient and state streams brought into shared memory by
 *               cp.async.bulk copies completing on an mbarrier, and the
 *               replicas written back by bulk stores; R*M <= 16; every
 *               device wait is bounded and reports ZERO_DEV_TIMEOUT).
 *   scratch     device scratch of scratch_bytes bytes; the staged variant
 *               needs plan->scratch_bytes_staged (fp32 reduced gradient of
 *               every shard); ignored (may be NULL) for the fused variant.
 *               ZeRO-2 gives up the gradients once they are reduced (CS25 V6
 *               Lecture 4 notes, "ZeRO-2"): with plan->stage == 2 and
 *               R*M >= 2 the staged variant accepts scratch = NULL and then
 *               keeps the reduced gradient in rank_grads[0] and
 *               rank_grads[1] (the low and high 16 bits of each element's
 *               fp32 value), whose contents are unspecified afterwards (the
 *               next backward must write them again: read as gradients they
 *               are arbitrary bits); those two buffers are then outputs and
 *               may alias no other buffer.
 *   flags       0, ZERO_FLAG_CHECK_FINITE, and for the TMA variant
 *               ZERO_FLAG_DEBUG_EXPIRE_WAITS (test only).
 *   dev_status  optional device int32 the kernels OR ZERO_DEV_* bits into.
 * Outputs (master, m, v, replicas, scratch) must not overlap one another or
 * any gradient buffer (ZERO_ERR_OVERLAP).  All variants give identical
 * bits.
 */
zero_status zero_step(const zero_plan_t* plan, const uint16_t* const* rank_grads,
                      float* master, float* m, float* v, uint16_t* const* rank_params,
                      const zero_adamw_hparams* hp, int64_t step, int32_t variant,
                      void* scratch, int64_t scratch_bytes, int32_t flags,
                      int32_t* dev_status, void* stream);

/*
 * Read the device status word after the steps that wrote it (failure
 * detection: find and report a failed step instead of hanging or going on
 * silently; LLM infra 06, section 15.4).
 *   dev_status  the caller's device int32 passed to the steps (4-byte
 *               aligned).  It is read, not cleared: zero it before the next
 *               steps that should report afresh.
 *   stream      the stream the steps ran on: the call enqueues the read of
 *               the word on it and waits for the stream to finish (so it is
 *               a host-side call, not for a stream being captured).
 *   out         optional host int32: receives the word (ZERO_DEV_* bits).
 * Returns ZERO_ERR_DEVICE_TIMEOUT when ZERO_DEV_TIMEOUT is set (with or
 * without ZERO_DEV_DRAIN_FAILED), else ZERO_ERR_NONFINITE when
 * ZERO_DEV_NONFINITE is set (zero_step_clipped's ZERO_DEV_SKIPPED comes with
 * it), else ZERO_OK; ZERO_ERR_NULL for a NULL dev_status, ZERO_ERR_ALIGN for
 * a misaligned one, ZERO_ERR_CUDA when the copy or the wait fails (*out is
 * then not written).
 */
zero_status zero_get_device_status(const int32_t* dev_status, void* stream, int32_t* out);

/*
 * Staged step 1, reduce-scatter + average: for each rank r and each element
 * i of shard r, g_shards[i] = (ordered fp32 sum of the R*M gradients at i) /
 * (R*M).  g_shards: device, plan->padded floats (shard r at r*S); elements
 * [N, padded) are not written.  Same pointer rules as zero_step.
 */
zero_status zero_rs_avg(const zero_plan_t* plan, const uint16_t* const* rank_grads,
                        float* g_shards, int32_t flags, int32_t* dev_status, void* stream);

/*
 * Staged step 2, AdamW on every rank's shard: reads g_shards (from
 * zero_rs_avg) and updates master, m, v in place at the N real elements.
 */
zero_status zero_adamw_shard(const zero_plan_t* plan, const float* g_shards, float* master,
                             float* m, float* v, const zero_adamw_hparams* hp, int64_t step,
                             void* stream);

/*
 * Staged step 3, cast + all-gather: every rank r casts its shard of master
 * to bf16 and writes it into all R replicas.
 */
zero_status zero_ag_cast(const zero_plan_t* plan, const float* master,
                         uint16_t* const* rank_params, void* stream);

/*
 * Step with global gradient-norm clipping (the training recipe "AdamW +
 * gradient clipping", CS324 Lecture 9 notes, section 7.4; fp32 gradient
 * reduction, LLM infra 06, section 15.3).  After the reduce-scatter and
 * average, the squared global norm is the fp32 pairwise (binary-tree) sum of
 * the squares g_i*g_i with the leaves padded by zeros to a power of two (one
 * fixed order, identical for any grid); norm = sqrt(sumsq) and
 * coef = max_norm / (norm + 1e-6) in double; when coef < 1 every averaged
 * gradient is multiplied by (float)coef, then AdamW and the all-gather run as
 * in zero_step.  A non-finite squared norm sets ZERO_DEV_NONFINITE in
 * dev_status; with ZERO_FLAG_SKIP_NONFINITE the update is skipped (state and
 * replicas untouched) and ZERO_DEV_SKIPPED is set.
 *   max_norm   > 0 and finite.
 *   scratch    device, 16-byte aligned, at least zero_clip_scratch_bytes(plan)
 *              bytes: the fp32 averaged gradients and one tree partial per
 *              group of tiles (any contents on entry; nothing persists
 *              between calls).
 * Two launches: the reduce-scatter with the tree up to one partial per group
 * of tiles, then the update, whose blocks each finish the tree, derive the
 * coefficient and run AdamW with the all-gather.
 *   dev_sumsq  optional device double: receives the squared norm.
 * Traffic: 2RM + 4 bytes/param (reduce-scatter, gradient stash) plus
 * 4 + 24 + 2R (update and all-gather); the tree's partials (at most 32 KB)
 * are read from L2.
 */
zero_status zero_step_clipped(const zero_plan_t* plan, const uint16_t* const* rank_grads,
                              float* master, float* m, float* v, uint16_t* const* rank_params,
                              const zero_adamw_hparams* hp, int64_t step, float max_norm,
                              void* scratch, int64_t scratch_bytes, int32_t flags,
                              int32_t* dev_status, double* dev_sumsq, void* stream);

/* Scratch bytes zero_step_clipped needs for this plan (-1 for a bad plan). */
int64_t zero_clip_scratch_bytes(const zero_plan_t* plan);

/*
 * Replica consistency check, a silent-data-corruption detector (LLM infra
 * 06, section 15.4: a GPU that flips a bit is found by comparing what two
 * ranks computed on the same data).  After the all-gather every replica must
 * hold the same bits; this counts the elements where any replica differs
 * from rank 0's.
 *   dev_count  device int64 (8-byte aligned): receives the count (zeroed
 *              first, on `stream`).
 *   dev_first  optional device int64: receives the first such index, or
 *              INT64_MAX when there is none.
 * Reads 2R bytes per parameter.
 */
zero_status zero_check_replicas(const zero_plan_t* plan, uint16_t* const* rank_params,
                                int64_t* dev_count, int64_t* dev_first, void* stream);

/* Codecs for zero_step_compressed. */
#define ZERO_COMP_FP16 1           /* binary16, round to nearest even: 2 bytes sent a param */
#define ZERO_COMP_INT8 2           /* per 128-element block: 1 byte + a 4-byte scale */
#define ZERO_COMP_SIGN 3           /* per 128-element block: 1 bit + a 4-byte magnitude */

/*
 * Step with a compressed gradient reduce-scatter (CS324 Lecture 9 notes,
 * section 7.4: each card compresses what it sends - fp16, int8 quantised per
 * block, sign only - optionally with error feedback, each card keeping what
 * the compression dropped and adding it to its next gradient).  Rank r's
 * locally accumulated gradient x_r (+ its residual e_r) is compressed over
 * aligned blocks of 128 elements of the flat vector (the last may be short):
 *   FP16: d = binary16(x) (round to nearest even)
 *   INT8: s = max|x| / 127 per block; d = 0 if s == 0, else
 *         clamp(rint(x / s), -127, 127) * s
 *   SIGN: s = (pairwise fp32 sum of |x| over the block) / count;
 *         d = (x < 0) ? -s : s
 * The owner sums the d_r in rank order, divides by R*M, and AdamW and the
 * all-gather follow as in zero_step.
 *   residuals  NULL (no error feedback), or a host array of R device
 *              pointers, N floats each (16-byte aligned), read and updated
 *              in place: e_r <- x_r - d_r.  Start them at zero.
 * Traffic: 2RM + 24 + 2R bytes/param, plus 8R with error feedback (the
 * compressed message itself lives in registers, never in memory).
 */
zero_status zero_step_compressed(const zero_plan_t* plan, const uint16_t* const* rank_grads,
                                 float* master, float* m, float* v, uint16_t* const* rank_params,
                                 const zero_adamw_hparams* hp, int64_t step, int32_t kind,
                                 float* const* residuals, void* stream);

/*
 * 1-bit Adam step (CS324 Lecture 9 notes, section 7.4: error feedback alone
 * does not carry over to Adam, so warm up with plain Adam, then freeze the
 * variance into a fixed preconditioner and send 1 bit per value).
 *   step <= freeze_step (the warm-up): exactly zero_step's fused step; v is
 *     updated and the residuals are not touched.
 *   step > freeze_step, for every element i and rank r:
 *     gl_r = (sum_j G[r][j][i]) / M;  x_r = beta1*m[i] + (1-beta1)*gl_r + E_r[i]
 *     d_r  = sign codec of x_r (ZERO_COMP_SIGN, 128-element blocks of the
 *            flat vector);  E_r[i] = x_r - d_r
 *     y    = (d_0 + ... + d_{R-1}) / R + Es[i]   (ranks ascending)
 *     ds   = sign codec of y over the same blocks, which lie inside one
 *            owner's shard;  Es[i] = y - ds;  m[i] = ds
 *     W[i] = W[i]*(1-lr*wd) - lr/(1-beta1^t) * ds / (sqrt(v[i]) /
 *            sqrt(1-beta2^freeze_step) + eps);  v is read, not written;
 *     every replica receives bf16(W[i]).
 *   Each float operation is rounded on its own.
 *   freeze_step  >= 1, else ZERO_ERR_INVALID_ARG.
 *   plan->S      must be a multiple of 128 (make the plan with align_elems
 *                a multiple of 128) so that every owner's compression block
 *                is a block of the flat vector; else ZERO_ERR_INVALID_ARG.
 *   worker_residuals  host array of R device pointers, N floats each
 *                (16-byte aligned), read and updated in place; start at 0.
 *   server_residual   device, plan->padded floats in the state layout
 *                (element i at index i, the pad never touched); start at 0.
 * Traffic after the warm-up: 2RM + 10R + 28 bytes/param (grads 2RM, worker
 * residuals 8R, replicas 2R, W/m/Es read and written 24, v read 4).
 */
zero_status zero_step_onebit(const zero_plan_t* plan, const uint16_t* const* rank_grads,
                             float* master, float* m, float* v, uint16_t* const* rank_params,
                             const zero_adamw_hparams* hp, int64_t step, int64_t freeze_step,
                             float* const* worker_residuals, float* server_residual,
                             void* stream);

/*
 * ZeRO-3 step (CS25 V6 Lecture 4 notes, "ZeRO-3 / FSDP": the parameters are
 * sharded as well and materialised per unit just before use; CS324 Lecture
 * 9 notes, section 3.4: bit-identical to plain DP).  The reduce-scatter,
 * average and AdamW of zero_step, then each rank casts its updated shard to
 * bf16 into its own parameter shard; there is no all-gather in the step.
 *   param_shards  device, plan->padded bf16 in the padded layout of the
 *                 state (shard r at r*S, element i at index i); the pad is
 *                 never written.
 * Traffic: 2RM + 24 + 2 bytes/param.  Other arguments as zero_step.
 */
zero_status zero3_step(const zero_plan_t* plan, const uint16_t* const* rank_grads,
                       float* master, float* m, float* v, uint16_t* param_shards,
                       const zero_adamw_hparams* hp, int64_t step, int32_t flags,
                       int32_t* dev_status, void* stream);

/*
 * ZeRO-3 all-gather of one unit (a layer, or any range of the flat vector)
 * before its use: outs[o][i - lo] = param_shards[i] for i in [lo, hi), where
 * element i comes from the shard of rank i / S, for each of the n_out
 * transient buffers (the ranks that materialise the unit, 1 <= n_out <= R).
 *   0 <= lo <= hi <= N; lo may be any element (units start at arbitrary
 *   tensor offsets).  outs: host array of n_out device pointers, each
 *   (hi - lo) bf16, 16-byte aligned, not overlapping each other or the
 *   shards.  Traffic: 2 + 2 n_out bytes per element.
 */
zero_status zero3_gather(const zero_plan_t* plan, const uint16_t* param_shards, int64_t lo,
                         int64_t hi, uint16_t* const* outs, int32_t n_out, void* stream);

/*
 * ZeRO-3 all-gather of a table of units in one launch: for every entry k,
 * units[k].out[i - lo] = param_shards[i] for i in [units[k].lo, units[k].hi),
 * exactly as zero3_gather of that unit with one destination.  Built for the
 * many small units of a per-tensor schedule, whose separate launches would
 * leave the GPU idle between them (CS25 V6 Lecture 4 notes, "ZeRO-3 / FSDP":
 * each unit is materialised just before use; LLM infra 06, section 3.1).
 *   units    host array of n_units entries, read during the call only (the
 *            table travels with the launch, so it may be reused at once).
 *            Each: 0 <= lo <= hi <= N, any lo; out device, hi - lo bf16,
 *            16-byte aligned (may be NULL when lo == hi).  Outputs must not
 *            overlap each other or the shards (ZERO_ERR_OVERLAP); the units'
 *            source ranges may overlap.  To write one unit into several
 *            buffers, list it once per buffer.
 *   n_units  0 .. ZERO_MAX_GATHER_UNITS (0 is a no-op).
 * Traffic: 2 + 2 bytes per element of every unit.
 */
#define ZERO_MAX_GATHER_UNITS 1024
typedef struct {
    int64_t lo, hi;
    uint16_t* out;
} zero_gather_unit;
zero_status zero3_gather_units(const zero_plan_t* plan, const uint16_t* param_shards,
                               const zero_gather_unit* units, int32_t n_units, void* stream);

/*
 * ZeRO-3 gradient reduce-scatter of one unit, right after that unit's
 * backward (CS25 V6 Lecture 4 notes, "ZeRO-3 / FSDP": the backward
 * materialises each unit's parameters again and reduce-scatters its
 * gradient; LLM infra 06, section 3.1).  For every element i in [lo, hi):
 *   grad_shards[i] = (ordered fp32 sum over r, j of unit_grads[r*M + j][i - lo])
 *                    / (R*M)
 * with the sum order and the division of zero_step, written into the owner's
 * gradient shard.  Elements outside [lo, hi) are not touched.
 *   unit_grads   host array of R*M device pointers, each hi - lo bf16 (the
 *                unit's gradient of rank r, micro-batch j), 16-byte aligned.
 *   grad_shards  device, plan->padded floats in the state layout (element i
 *                at index i, pad never written); must not overlap the inputs.
 *   0 <= lo <= hi <= N, any lo.  flags: 0 or ZERO_FLAG_CHECK_FINITE (then
 *   dev_status is required, as in zero_step).
 * Traffic: 2RM + 4 bytes per element of the unit.
 */
zero_status zero3_rs_unit(const zero_plan_t* plan, const uint16_t* const* unit_grads, int64_t lo,
                          int64_t hi, float* grad_shards, int32_t flags, int32_t* dev_status,
                          void* stream);

/*
 * ZeRO-3 shard update from reduce-scattered gradients: AdamW of every
 * element i < N from grad_shards[i], then param_shards[i] = bf16(master[i]),
 * the rank's own parameter shard.  After zero3_rs_unit over units that cover
 * [0, N) once, in any order, the result is zero3_step's, bit for bit.
 *   grad_shards  device, plan->padded floats (read only).  Other arguments
 *                as zero3_step.
 * Traffic: 4 + 24 + 2 bytes per element.
 */
zero_status zero3_update(const zero_plan_t* plan, const float* grad_shards, float* master,
                         float* m, float* v, uint16_t* param_shards,
                         const zero_adamw_hparams* hp, int64_t step, void* stream);

/*
 * End-to-end step from host memory.  host_grads: R*M host pointers to the
 * gradient buffers (N bf16 each); host_params_out: host, N bf16, receives
 * replica 0 (every replica holds the same bits).  Two modes:
 *   dev_grads == NULL (zero-copy): the fused kernel reads the gradients
 *     straight from host memory over the host link and writes replica 0's
 *     bits to host_params_out as well as to the R device replicas, so the
 *     transfers overlap the HBM work.  The host buffers must be reachable by
 *     the GPU: pinned memory (cudaHostAlloc / cudaHostRegister), or any host
 *     memory on systems where the GPU uses the host page tables; otherwise
 *     ZERO_ERR_INVALID_ARG.
 *   dev_grads != NULL (copy engine): R*M cudaMemcpyAsync copies into
 *     dev_grads (device, N bf16 each, must not overlap), the fused step,
 *     then one copy of replica 0 to host_params_out.
 * All on `stream`; the host buffers must stay valid until the stream has
 * finished.  Same argument rules as zero_step otherwise.
 */
zero_status zero_step_host(const zero_plan_t* plan, const uint16_t* const* host_grads,
                           uint16_t* const* dev_grads, float* master, float* m, float* v,
                           uint16_t* const* rank_params, uint16_t* host_params_out,
                           const zero_adamw_hparams* hp, int64_t step, int32_t flags,
                           int32_t* dev_status, void* stream);

/*
 * Staged step that allocates nothing and takes no scratch argument.
 * (The lecture pages have no counterpart; this entry point exists for
 * callers, not for the method.)  Some callers cannot allocate device memory
 * at all: a host runtime that has already reserved the GPU's memory for its
 * own pool and forbids other allocations, or a latency-critical caller for
 * which cudaMalloc, which can synchronize the device, is not allowed.  They
 * can still run the staged step through this call.  The fp32 reduced
 * gradient lives in a fixed array of ZERO_NOALLOC_MAX_ELEMS floats (16 MiB)
 * that this library places in device memory; every GPU that loads the
 * library holds that array until the process exits.
 *   - The plan must have plan->padded <= ZERO_NOALLOC_MAX_ELEMS, else
 *     ZERO_ERR_SIZE is returned and nothing is launched.
 *   - The first call on a device looks up the array's device address
 *     (once per device, with that device current, and again if the
 *     device's context has been replaced since, e.g. by cudaDeviceReset);
 *     make that first call before any stream capture.  A failed lookup
 *     returns ZERO_ERR_CUDA.
 *   - `stream` must belong to the current device (the array's address is
 *     that device's), else ZERO_ERR_INVALID_ARG.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents; nothing needs clearing, because the reduce-scatter
 *     writes every element the AdamW kernel then reads.  Calls that overlap
 *     on the GPU (e.g. on two streams at once) race on the array: order
 *     them on one stream.
 * Arguments, results and errors are otherwise those of zero_step with
 * variant ZERO_VARIANT_STAGED; the bits are the same.
 */
#define ZERO_NOALLOC_MAX_ELEMS (4 * 1024 * 1024)
zero_status zero_step_staged_noalloc(const zero_plan_t* plan, const uint16_t* const* rank_grads,
                                     float* master, float* m, float* v,
                                     uint16_t* const* rank_params, const zero_adamw_hparams* hp,
                                     int64_t step, int32_t flags, int32_t* dev_status,
                                     void* stream);

/* ------------------------------------------------------------------------
 * Sharded optimizer-state checkpoints and R -> R' resharding.
 * One file per rank shard, "<dir>/shard-RRRRR-of-NNNNN.zck": a 128-byte
 * header (layout R, rank, N, S, lo, len; step; AdamW hyper-parameters;
 * Fletcher-64 checksums of payload and header), then the rank's elements
 * [lo, lo+len) as bf16 params, fp32 master, m, v: 14 bytes per parameter,
 * BLOOM's checkpoint layout (CS324 Lecture 9 notes, section 2.1).  Each file
 * is written to "<name>.tmp", fsync'ed and renamed (sharded, atomic writes:
 * LLM infra 06, section 15.4); one checkpoint per directory.  Loading under
 * another plan (another R', same N) reads, for each new shard, the byte
 * ranges of the old shards that overlap it: the merge a different card
 * count needs (CS324 Lecture 9 notes, exercise 11).  A save followed by a
 * load reproduces every bit, so training resumes bit-identically (section
 * 3.1, PaLM).
 * ---------------------------------------------------------------------- */

typedef struct zero_ckpt_job zero_ckpt_job;

/*
 * Host layer (no GPU needed).  params: host, N bf16 (element i at [i]);
 * master, m, v: host, element i at [i] (plan->padded or at least N floats).
 * Writes every shard of `plan` into dir (created if missing), n_threads
 * files at a time.  Errors: ZERO_ERR_NULL, ZERO_ERR_INVALID_ARG, ZERO_ERR_IO.
 */
zero_status zero_ckpt_write_host(const zero_plan_t* plan, const uint16_t* params,
                                 const float* master, const float* m, const float* v,
                                 int64_t step, const zero_adamw_hparams* hp, const char* dir,
                                 int32_t n_threads);

/*
 * Host layer: read the checkpoint in dir into the layout of `plan` (same N,
 * any R).  rank = -1 fills every element [0, N); rank = r fills only the
 * elements of the new shard r (what rank r would load on its own GPU).
 * The old shards touched are checksum-verified first.  step_out / hp_out may
 * be NULL.  Errors: ZERO_ERR_IO (missing/short file), ZERO_ERR_CORRUPT (bad
 * magic, header or payload checksum, inconsistent shards), ZERO_ERR_SIZE
 * (the checkpoint has another N).
 */
zero_status zero_ckpt_read_host(const zero_plan_t* plan, const char* dir, int32_t rank,
                                uint16_t* params, float* master, float* m, float* v,
                                int64_t* step_out, zero_adamw_hparams* hp_out);

/*
 * Device layer, asynchronous save: enqueues device-to-host copies of the
 * state (dev_params: N bf16, e.g. replica 0 or the ZeRO-3 shard buffer;
 * dev_master/m/v: element i at [i]) into a pinned staging buffer on
 * `stream`, then writes the shard files on a background thread once the
 * copies have landed.  Later work on `stream` is ordered after the copies,
 * so training can continue at once.  *job must be passed to
 * zero_ckpt_job_wait, which joins the writer, frees the staging buffer and
 * returns the write status.  The library allocates the staging buffer
 * (14 bytes/param of pinned host memory).
 */
zero_status zero_ckpt_save_async(const zero_plan_t* plan, const uint16_t* dev_params,
                                 const float* dev_master, const float* dev_m, const float* dev_v,
                                 int64_t step, const zero_adamw_hparams* hp, const char* dir,
                                 int32_t n_threads, void* stream, zero_ckpt_job** job);

/* Wait for an asynchronous save; frees the job.  Returns its status. */
zero_status zero_ckpt_job_wait(zero_ckpt_job* job);

/*
 * Device layer, load: reads the checkpoint in dir (any R) into the layout
 * of `plan` and copies it to the device: dev_master/m/v element i at [i] (the
 * pad is not written), the bf16 params into each of the n_params device
 * buffers dev_params[k] (N bf16: the R replicas, or one ZeRO-3 shard
 * buffer).  Synchronizes `stream` before returning.  Errors as
 * zero_ckpt_read_host, plus ZERO_ERR_CUDA.
 */
zero_status zero_ckpt_load(const zero_plan_t* plan, const char* dir, uint16_t* const* dev_params,
                           int32_t n_params, float* dev_master, float* dev_m, float* dev_v,
                           int64_t* step_out, zero_adamw_hparams* hp_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif
