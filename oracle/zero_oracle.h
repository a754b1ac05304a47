/*
 * zero_oracle.h - CPU oracle for the ZeRO-1/2 mixed-precision AdamW step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  This is the plain, slow, single
 * threaded definition that the CUDA path is checked against.  Only the test
 * suite, __graft_entry__.smoke() and the cpu_baseline / reference leg of
 * bench.py may load it.  The product library (zero_optimizer_step_rs_gb300)
 * neither links nor calls it, and the two share no source: the seeded input
 * generator in zgen/ is the only module both sides use, and it holds none of
 * the step's arithmetic.
 *
 * What it computes (sources are the five lecture pages on distributed
 * training this project is built from):
 *   - gradient accumulation g = (1/M) sum_j grad_j
 *       [CS25 V6 Lecture 4 notes, "single-GPU baseline and gradient
 *        accumulation", accumulation equation; LLM infra 06, section 7.2]
 *   - data-parallel averaging g = (1/P) sum_r g_r, identical update per rank
 *       [CS25 V6 Lecture 4 notes, "replicate the model, split the batch",
 *        DP equation; CS324 Lecture 9 notes, section 3.1]
 *   - reduce-scatter / all-gather, AllReduce = ReduceScatter + AllGather
 *       [CS336 Lecture 7 book, sections 2.3 and 4.3; LLM infra 06, 2.0]
 *   - ZeRO-1/2: each rank updates only its shard of the fp32 master weights
 *     and Adam moments, then all-gathers the new parameters; bit-identical to
 *     plain DP because AdamW is elementwise
 *       [CS324 Lecture 9 notes, section 3.4; CS25 V6 Lecture 4 notes,
 *        "ZeRO-1" and "ZeRO-2"; CS336 Lecture 7 summary, Q2]
 *   - 16 bytes/param mixed-precision state: bf16 param 2 + bf16 grad 2 +
 *     fp32 master 4 + m 4 + v 4
 *       [CS324 Lecture 9 notes, section 2.1; CS336 Lecture 7 summary, Q3]
 *   - ring all-reduce demo and its per-card send volume 2(p-1)/p
 *       [CS324 Lecture 9 notes, section 3.2]
 *   - per-device model-state formulas M_DP, M_Z1, M_Z2 (and Z3)
 *       [CS25 V6 Lecture 4 notes, "ZeRO-1" and "ZeRO-2" memory equations;
 *        CS324 Lecture 9 notes, exercises 1 and 7]
 *
 * Readings where the pages leave a step open:
 *   R1 AdamW is torch.optim.AdamW's documented algorithm (decoupled decay
 *      w*(1-lr*wd) first, then m/v EMA, bias correction, eps added after
 *      the bias-corrected square root).
 *   R2 every float operation is rounded to nearest-even on its own; no fused
 *      multiply-add; the exact sequence is the one in oracle_adamw_elem().
 *   R3 each rank first sums its M micro-batch gradients (j ascending), then
 *      the rank sums are added in ascending rank order; each sum starts from
 *      its first term (no +0.0 seed).
 *   R4 one IEEE division of the fp32 sum by (float)(R*M) after summation.
 *   R5 weight decay applies to every element.
 *   R6 shard length S = roundup(ceil(N/R), ALIGN); owner(i) = i / S; state
 *      arrays hold R*S floats with shard r at r*S; pad elements are never
 *      read or written; replicas hold exactly N elements.
 *   R7 bf16 cast: round to nearest, ties to even; +-Inf kept; overflow to
 *      +-Inf; every NaN becomes the one quiet NaN 0x7FC0 (IEEE 754 fixes
 *      neither the sign nor the payload of a NaN an operation produces).
 *   R8 non-finite gradients propagate IEEE-wise (no skip).
 *   R9 ZeRO-1 and ZeRO-2 compute the same numbers; the stage changes only
 *      which buffers stay resident (the byte accounting).
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* AdamW hyper-parameters as a user gives them. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
} oracle_hparams;

/* The per-step float scalars of the update, each computed once in double
 * from the hyper-parameters and the step count t, then rounded to float. */
typedef struct {
    float step_size;   /* lr / (1 - beta1^t)              */
    float bc2_sqrt;    /* sqrt(1 - beta2^t)               */
    float decay;       /* 1 - lr * weight_decay           */
    float beta1, beta2;
    float one_minus_beta1, one_minus_beta2;
    float eps;
    float denom_rm;    /* (float)(R * M)                  */
} oracle_scalars;

/* bf16 <-> float, written from the format definition (sign, 8-bit exponent,
 * 7-bit fraction = the high half of an IEEE binary32). */
uint16_t oracle_bf16_rne(float x);
float    oracle_bf16_to_float(uint16_t h);

/* Per-step scalars (reading R1, R4). step >= 1. */
void oracle_make_scalars(const oracle_hparams* hp, int64_t step, int32_t R,
                         int32_t M, oracle_scalars* out);

/* One AdamW update of one element (reading R1, R2). g is the averaged
 * gradient; w, m, v are updated in place. */
void oracle_adamw_elem(const oracle_scalars* s, float g, float* w, float* m,
                       float* v);

/* Averaged gradient of element i over R ranks x M micro-batches (R3, R4).
 * G is an array of R*M pointers, entry r*M+j = rank r, micro-batch j. */
float oracle_avg_grad(const uint16_t* const* G, int32_t R, int32_t M,
                      int64_t i, float denom_rm);

/* Unsharded data-parallel step: every rank all-reduces the gradients and
 * applies the same AdamW update to a full copy of the state; the result is
 * written to every rank's replica P[r] (R pointers, n bf16 each).
 * W, m, v hold n floats.  Returns 0, or -1 on a bad argument. */
int oracle_dp_step(int64_t n, int32_t R, int32_t M,
                   const uint16_t* const* G, float* W, float* m, float* v,
                   uint16_t* const* P, const oracle_hparams* hp, int64_t step);

/* Same as oracle_dp_step, split over nthreads element ranges (the step is
 * elementwise, so the result is bit-identical).  Used to time the oracle on
 * all host cores; nthreads <= 0 means 1. */
int oracle_dp_step_mt(int64_t n, int32_t R, int32_t M,
                      const uint16_t* const* G, float* W, float* m, float* v,
                      uint16_t* const* P, const oracle_hparams* hp,
                      int64_t step, int32_t nthreads);

/* Shard length S = roundup(ceil(n/R), align) (reading R6). align >= 1. */
int64_t oracle_shard_len(int64_t n, int32_t R, int32_t align);

/* ZeRO-1/2 step emulated card by card, each card a separate buffer:
 *   1. reduce-scatter: card r receives, from every rank r', a copy of the
 *      bf16 gradient chunk r of each of r's M micro-batches, and sums them
 *      (R3) into its fp32 gradient shard, then divides by R*M (R4);
 *   2. card r updates its own slice [r*S, r*S+len_r) of W, m, v (R*S floats
 *      each, reading R6) with AdamW;
 *   3. all-gather: card r casts its updated shard to bf16 (R7) and copies it
 *      into every card's replica P[r'] (n bf16 each).
 * Returns 0, -1 on a bad argument, -2 if a buffer cannot be allocated. */
int oracle_zero_step(int64_t n, int32_t R, int32_t M, int64_t S,
                     const uint16_t* const* G, float* W, float* m, float* v,
                     uint16_t* const* P, const oracle_hparams* hp,
                     int64_t step);

/* Reduce-scatter alone (sum, no division): card r ends with chunk r of the
 * element-wise sum over ranks; out[r] points to S floats (only the first
 * len_r are written).  in[r] points to n floats.  Sum order as R3. */
int oracle_reduce_scatter_sum(int64_t n, int32_t R, int64_t S,
                              const float* const* in, float* const* out);

/* Ring all-reduce over p cards (CS324 Lecture 9 notes, section 3.2): the
 * arrays are cut into p chunks; p-1 reduce-scatter steps in which every card
 * sends one chunk to the next card, which adds it to its own copy, then p-1
 * all-gather steps in which the completed chunks are passed on and
 * overwrite.  cards[k] points to n floats, updated in place; sent[k]
 * receives the count of numbers card k sent.  Returns 0 or -1. */
int oracle_ring_allreduce(float* const* cards, int32_t p, int64_t n,
                          int64_t* sent);

/* Per-device model-state bytes for N params on P ranks with b_p, b_g, b_o
 * bytes of parameter, gradient and optimizer state per param:
 *   out[0] DP = N(b_p + b_g + b_o)
 *   out[1] Z1 = N(b_p + b_g) + N b_o / P
 *   out[2] Z2 = N b_p + N(b_g + b_o) / P
 *   out[3] Z3 = N(b_p + b_g + b_o) / P
 * (CS25 V6 Lecture 4 notes, ZeRO-1/ZeRO-2 memory equations; Z3 from
 *  CS324 Lecture 9 notes, exercise 1). */
void oracle_zero_bytes(double N, int32_t P, double bp, double bg, double bo,
                       double out[4]);

/* ------------------------------------------------------------------------
 * Global gradient-norm clipping with a non-finite check, before the update
 * (the training recipe of AdamW with gradient clipping, CS324 Lecture 9
 * notes, section 7.4; fp32 gradient reduction, LLM infra 06, section 15.3).
 * Readings:
 *   R10 the squared norm is the fp32 pairwise (binary-tree) sum of the
 *       leaves g_i * g_i (fp32 products), i < n, padded with zeros to the
 *       next power of two: one fixed order, so every implementation that
 *       follows the tree gets the same bits (fp32, the precision
 *       clip_grad_norm_ uses for fp32 gradients);
 *   R11 norm = sqrt(sumsq); coef = max_norm / (norm + 1e-6) in double (the
 *       clip_grad_norm_ formula); when coef < 1 every averaged gradient is
 *       multiplied by (float)coef, otherwise it is left alone;
 *   R12 a non-finite sumsq is reported; with skip_nonfinite the whole step
 *       is skipped (state and replicas untouched), otherwise the formula
 *       runs on as IEEE arithmetic gives it.
 * ---------------------------------------------------------------------- */

/* Pairwise fp32 sum of g[i]*g[i] over n leaves padded to a power of two
 * (returned widened to double). */
double oracle_grad_sumsq(const float* g, int64_t n);

/* Clip coefficient from the squared norm (norm = sqrt(sumsq) and the
 * quotient in double): returns the float multiplier and
 * sets *clip to 1 when coef < 1; otherwise (coef >= 1, or coef NaN because
 * the norm is NaN) returns 1.0f and sets *clip to 0. */
float oracle_clip_coef(double sumsq, float max_norm, int32_t* clip);

/* DP step with global-norm clipping: averaged gradients (as oracle_dp_step),
 * squared norm (R10), coefficient (R11), non-finite handling (R12), then the
 * AdamW update and the replica write of oracle_dp_step.  *sumsq_out (may be
 * NULL) receives the squared norm; *skipped_out (may be NULL) is set to 1 when
 * the step was skipped.  Returns 0, -1 on a bad argument, -2 on allocation
 * failure. */
int oracle_dp_step_clipped(int64_t n, int32_t R, int32_t M,
                           const uint16_t* const* G, float* W, float* m, float* v,
                           uint16_t* const* P, const oracle_hparams* hp,
                           int64_t step, float max_norm, int32_t skip_nonfinite,
                           double* sumsq_out, int32_t* skipped_out);

/* ------------------------------------------------------------------------
 * ZeRO-3 (CS25 V6 Lecture 4 notes, "ZeRO-3 / FSDP": parameters are sharded
 * too and materialised per unit just before use; CS324 Lecture 9 notes,
 * section 3.4 and exercise 7: bit-identical to DP, per-card traffic
 * 3(p-1)/p Psi against 2(p-1)/p for DP / ZeRO-1 / ZeRO-2).
 * Reading R13: each card keeps its bf16 parameter shard in the same padded
 * layout as the fp32 state (R*S elements, shard r at r*S); the step is the
 * ZeRO-2 reduce-scatter and shard update followed by a cast into the
 * card's own shard, with no all-gather; a unit [lo, hi) of the flat vector
 * is all-gathered on demand into a card's transient buffer.
 * ---------------------------------------------------------------------- */

/* ZeRO-3 step emulated card by card.  Pshard holds R*S bf16 (shard r at
 * r*S).  recv (may be NULL, R entries) receives, per card, the count of
 * gradient numbers it got from other cards in the reduce-scatter: one per
 * other rank and element, since a rank sums its micro-batches before the
 * reduce-scatter.
 * Returns 0, -1 on a bad argument, -2 on allocation failure. */
int oracle_zero3_step(int64_t n, int32_t R, int32_t M, int64_t S,
                      const uint16_t* const* G, float* W, float* m, float* v,
                      uint16_t* Pshard, const oracle_hparams* hp, int64_t step,
                      int64_t* recv);

/* All-gather of the unit [lo, hi) for card `card`: out[i - lo] is copied
 * from the shard of owner(i).  *recv (may be NULL) receives the count of
 * numbers that came from other cards.  Returns 0 or -1. */
int oracle_zero3_gather(int64_t n, int32_t R, int64_t S, const uint16_t* Pshard,
                        int64_t lo, int64_t hi, int32_t card, uint16_t* out,
                        int64_t* recv);

/* ZeRO-3 backward, unit by unit (CS25 V6 Lecture 4 notes, "ZeRO-3 / FSDP":
 * the backward materialises each unit's parameters again and reduce-
 * scatters the unit's gradient; LLM infra 06, section 3.1: all-gather,
 * reduce-scatter and all-gather again, about 1.5 times DP's traffic).
 * Reading R16: right after a unit [lo, hi)'s backward, every rank holds the
 * unit's gradient for each of its micro-batches: Gu[r*M + j] holds hi - lo
 * bf16 values, element i at index i - lo.  Each card r receives, for the
 * elements of the unit it owns, the other ranks' local sums, and writes
 *   gshard[i] = (ordered sum as in oracle_avg_grad) / (R*M)
 * into its fp32 gradient shard (padded layout, element i at index i).
 * The step then updates every owned element from gshard and casts it into
 * the card's bf16 parameter shard (oracle_zero3_update).  Over any set of
 * units that covers [0, n) once, in any order, the result is that of
 * oracle_zero3_step.
 * recv (may be NULL, R entries) receives per card the count of numbers it
 * got from other cards for this unit: one per other rank and owned element.
 * Returns 0 or -1 (bad argument; 0 <= lo <= hi <= n). */
int oracle_zero3_rs_unit(int64_t n, int32_t R, int32_t M, int64_t S,
                         const uint16_t* const* Gu, int64_t lo, int64_t hi,
                         float* gshard, int64_t* recv);

/* ZeRO-3 shard update from reduce-scattered gradients: AdamW of every
 * element i < n from gshard[i], then Pshard[i] = bf16(W[i]).  Returns 0 or
 * -1. */
int oracle_zero3_update(int64_t n, int32_t R, int32_t M, int64_t S, const float* gshard,
                        float* W, float* m, float* v, uint16_t* Pshard,
                        const oracle_hparams* hp, int64_t step);

/* ------------------------------------------------------------------------
 * Compressed gradient reduce-scatter (CS324 Lecture 9 notes, section 7.4:
 * every card compresses the gradient it sends - fp16, int8, sign - with or
 * without error feedback, where each card keeps what compression dropped
 * and adds it back to its next gradient; real systems quantize int8 per
 * block rather than with one scale for the whole vector).
 * Reading R14: each rank compresses its locally accumulated gradient x_r
 * (after error feedback, x_r + e_r) over aligned blocks of 128 elements of
 * the flat vector (the last block may be short), and the owner sums the
 * decompressed values in rank order, then divides by R*M:
 *   fp16: d = (float)fp16_rne(x)                      (2 bytes/param sent)
 *   int8: a = max|x| over the block; s = a / 127; d = 0 when s == 0, else
 *         d = clamp(rint(x / s), -127, 127) * s        (1 + 4/128 bytes)
 *   sign: s = (pairwise fp32 tree sum of |x| over the block, zero padded to
 *         128) / count; d = (x < 0) ? -s : s          (1/8 + 4/128 bytes)
 * With error feedback the residual becomes e_r = x_r - d.
 * ---------------------------------------------------------------------- */

#define ORACLE_COMP_NONE 0
#define ORACLE_COMP_FP16 1
#define ORACLE_COMP_INT8 2
#define ORACLE_COMP_SIGN 3
#define ORACLE_COMP_BLOCK 128

/* binary16 round to nearest even from the format definition (NaN -> 0x7E00) */
uint16_t oracle_fp16_rne(float x);
float    oracle_fp16_to_float(uint16_t h);

/* Compress and decompress x[0..n) (blocks of 128 starting at element 0):
 * d[k] receives the value the receiver reconstructs. */
void oracle_compress(int32_t kind, const float* x, int64_t n, float* d);

/* DP step with a compressed reduce-scatter (R14).  E: NULL (no error
 * feedback) or R pointers to fp32 residuals of n elements, updated in
 * place.  Returns 0, -1, or -2 on allocation failure. */
int oracle_dp_step_compressed(int64_t n, int32_t R, int32_t M,
                              const uint16_t* const* G, float* W, float* m, float* v,
                              uint16_t* const* P, const oracle_hparams* hp,
                              int64_t step, int32_t kind, float* const* E);

/* ------------------------------------------------------------------------
 * 1-bit Adam (CS324 Lecture 9 notes, section 7.4: error feedback alone
 * does not carry over to Adam, because Adam is a non-linear function of the
 * gradient; the remedy is to warm up with plain Adam, then freeze the
 * variance into a fixed preconditioner and compress the communication to
 * 1 bit).
 * Reading R15 (the pages give the idea, not the formulas):
 *   - steps t <= T_w (the warm-up) are the plain step of oracle_dp_step,
 *     v is updated there, and the residuals are not touched;
 *   - at t > T_w, for each rank r and element i:
 *       gl_r = (sum_j G[r][j][i]) / (float)M       local average, j ascending
 *       ml_r = beta1*m[i] + (1-beta1)*gl_r          local momentum
 *       x_r  = ml_r + E[r][i]                       worker error feedback
 *       d_r  = sign codec of x_r over aligned 128-element blocks of the flat
 *              vector (R14's sign codec); E[r][i] = x_r - d_r
 *     and the owner of element i (rank i / S):
 *       a    = (((d_0 + d_1) + ...) + d_{R-1}) / (float)R
 *       y    = a + Es[i]                            server error feedback
 *       ds   = sign codec of y over blocks of 128 elements counted from the
 *              start of the owner's shard (the last block of a shard may be
 *              short); Es[i] = y - ds
 *       m[i] = ds                                   the momentum every rank
 *                                                   decompresses
 *       W[i] = W[i]*(1-lr*wd) - (lr/(1-beta1^t)) * (ds / den),
 *       den  = sqrt(v[i]) / sqrt(1-beta2^T_w) + eps
 *     v is not written: the frozen preconditioner is v and its bias
 *     correction as they stood at the end of the warm-up.  Every float
 *     operation is rounded on its own (R2); the replicas receive bf16(W).
 * ---------------------------------------------------------------------- */

/* One step of 1-bit Adam in the ZeRO layout.  S: shard length (the owner's
 * blocks start at multiples of S).  E: R pointers to n fp32 worker
 * residuals; Es: n fp32 server residuals (index i for element i); both are
 * updated in place at t > freeze_step and start at zero.  freeze_step >= 1.
 * v is updated in the warm-up only.
 * Returns 0, -1 (bad arguments) or -2 (allocation failure). */
int oracle_onebit_step(int64_t n, int64_t S, int32_t R, int32_t M,
                       const uint16_t* const* G, float* W, float* m, float* v,
                       uint16_t* const* P, const oracle_hparams* hp, int64_t step,
                       int64_t freeze_step, float* const* E, float* Es);

#ifdef __cplusplus
}
#endif
#endif
