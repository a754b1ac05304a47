/*
 * zero_oracle.c - CPU oracle for the ZeRO-1/2 mixed-precision AdamW step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE (see zero_oracle.h for who may load
 * it, the passages each function follows and the readings R1-R16).
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared
 * (-ffp-contract=off keeps every float * and + separately rounded, which is
 * reading R2; without -ffast-math gcc never reassociates float arithmetic).
 *
 * Parity pins (tests/test_oracle_pins.py, tests/test_oracle_collectives.py):
 *   oracle_bf16_rne        values fixed by the bf16 format (exact halfway
 *                          cases, Inf, NaN, overflow), and torch's bf16 cast
 *   oracle_make_scalars    closed forms at t=1 and t=2
 *   oracle_adamw_elem      hand-worked 3-element 2-step example; closed form
 *                          at step 1 with m=v=0; torch.optim.AdamW within
 *                          1e-6 over 20 steps; zero-gradient invariants
 *   oracle_avg_grad        identical micro-batches average exactly to the
 *                          gradient; exact small-integer sums against a
 *                          brute-force any-order sum
 *   oracle_dp_step(_mt)    the above, plus thread-count invariance
 *   oracle_zero_step       bit-identical to oracle_dp_step (the pages' ZeRO
 *                          == DP result), pad elements untouched
 *   oracle_reduce_scatter_sum  the worked 4-rank example 6/10/14/18
 *   oracle_ring_allreduce  the 4-card demo 10*[0..7] and send volume
 *                          2(p-1)/p
 *   oracle_zero_bytes      the pages' exercises (7B/8 ranks, 7.5B/64 ranks,
 *                          p=8 per-card units)
 *   oracle_shard_len       hand-computed layouts (uneven 100,000,007 / 7)
 *   oracle_zero3_rs_unit / oracle_zero3_update  (tests/test_oracle_zero3.py)
 *                          composed over random unit partitions in random
 *                          order == oracle_zero3_step bit for bit; the
 *                          worked 4-rank reduce-scatter example as one unit;
 *                          per-card receive counts add up to the step's
 *   oracle_onebit_step     (tests/test_oracle_onebit.py) warm-up == the
 *                          plain step; a hand-worked two-rank example; the
 *                          plain step whenever the sign codec is lossless
 *                          and beta2 = 0; a closed form for the frozen
 *                          preconditioner; codec and error-feedback
 *                          invariants on random inputs
 */
#define _POSIX_C_SOURCE 200809L
#include "zero_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 -- */

static uint32_t f2u(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float u2f(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* Round a binary32 to the nearest bf16, ties to even (reading R7).  A bf16
 * is the high 16 bits of a binary32, so rounding is: add half of the dropped
 * range, plus one more when the kept part is odd (ties to even), then drop
 * the low 16 bits.  A carry out of the fraction correctly bumps the exponent,
 * and a carry out of the largest finite value gives Inf. */
uint16_t oracle_bf16_rne(float x)
{
    uint32_t u = f2u(x);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)0x7FC0u;                     /* any NaN -> 0x7FC0 */
    uint32_t kept_lsb = (u >> 16) & 1u;
    u += 0x7FFFu + kept_lsb;
    return (uint16_t)(u >> 16);
}

float oracle_bf16_to_float(uint16_t h) { return u2f((uint32_t)h << 16); }

/* ------------------------------------------------------------- scalars -- */

void oracle_make_scalars(const oracle_hparams* hp, int64_t step, int32_t R,
                         int32_t M, oracle_scalars* out)
{
    double t = (double)step;
    double b1 = (double)hp->beta1, b2 = (double)hp->beta2;
    double lr = (double)hp->lr, wd = (double)hp->weight_decay;
    double bc1 = 1.0 - pow(b1, t);          /* bias correction of m */
    double bc2 = 1.0 - pow(b2, t);          /* bias correction of v */
    out->step_size = (float)(lr / bc1);
    out->bc2_sqrt = (float)sqrt(bc2);
    out->decay = (float)(1.0 - lr * wd);
    out->beta1 = hp->beta1;
    out->beta2 = hp->beta2;
    out->one_minus_beta1 = (float)(1.0 - b1);
    out->one_minus_beta2 = (float)(1.0 - b2);
    out->eps = hp->eps;
    out->denom_rm = (float)((double)R * (double)M);
}

/* ------------------------------------------------------- AdamW element -- */

/* torch.optim.AdamW's algorithm for one element (reading R1), each float
 * operation rounded on its own (reading R2):
 *   w  <- w * (1 - lr*wd)                 decoupled weight decay
 *   m  <- beta1*m + (1-beta1)*g           first moment
 *   v  <- beta2*v + ((1-beta2)*g)*g       second moment
 *   den = sqrt(v) / sqrt(1-beta2^t) + eps
 *   w  <- w - (lr/(1-beta1^t)) * (m / den)                                 */
void oracle_adamw_elem(const oracle_scalars* s, float g, float* w, float* m,
                       float* v)
{
    float wd = *w * s->decay;
    float a = s->beta1 * *m;
    float b = s->one_minus_beta1 * g;
    float m1 = a + b;
    float c = s->beta2 * *v;
    float d = s->one_minus_beta2 * g;
    float e = d * g;
    float v1 = c + e;
    float root = sqrtf(v1);
    float q = root / s->bc2_sqrt;
    float den = q + s->eps;
    float ratio = m1 / den;
    float upd = s->step_size * ratio;
    *w = wd - upd;
    *m = m1;
    *v = v1;
}

/* ----------------------------------------------------- gradient average -- */

float oracle_avg_grad(const uint16_t* const* G, int32_t R, int32_t M,
                      int64_t i, float denom_rm)
{
    float acc = 0.0f;
    for (int32_t r = 0; r < R; ++r) {
        /* local gradient accumulation of rank r, micro-batches in order */
        float local = oracle_bf16_to_float(G[(int64_t)r * M + 0][i]);
        for (int32_t j = 1; j < M; ++j)
            local = local + oracle_bf16_to_float(G[(int64_t)r * M + j][i]);
        /* ranks folded in ascending order */
        acc = (r == 0) ? local : acc + local;
    }
    return acc / denom_rm;
}

/* -------------------------------------------------------------- DP step -- */

static int check_args(int64_t n, int32_t R, int32_t M, const void* G,
                      const void* W, const void* m, const void* v,
                      const void* P, const void* hp, int64_t step)
{
    if (n < 0 || R < 1 || M < 1 || step < 1) return -1;
    if (!hp) return -1;
    if (n > 0 && (!G || !W || !m || !v || !P)) return -1;
    return 0;
}

int oracle_dp_step(int64_t n, int32_t R, int32_t M,
                   const uint16_t* const* G, float* W, float* m, float* v,
                   uint16_t* const* P, const oracle_hparams* hp, int64_t step)
{
    if (check_args(n, R, M, G, W, m, v, P, hp, step)) return -1;
    oracle_scalars s;
    oracle_make_scalars(hp, step, R, M, &s);
    for (int64_t i = 0; i < n; ++i) {
        /* all-reduce: every rank sees the same averaged gradient */
        float g = oracle_avg_grad(G, R, M, i, s.denom_rm);
        oracle_adamw_elem(&s, g, &W[i], &m[i], &v[i]);
        uint16_t p = oracle_bf16_rne(W[i]);
        for (int32_t r = 0; r < R; ++r) P[r][i] = p;
    }
    return 0;
}

typedef struct {
    int64_t lo, hi;
    int32_t R, M;
    const uint16_t* const* G;
    float *W, *m, *v;
    uint16_t* const* P;
    const oracle_hparams* hp;
    int64_t step;
    int rc;
} mt_job;

static void* mt_run(void* arg)
{
    mt_job* jb = (mt_job*)arg;
    int32_t RM = jb->R * jb->M;
    const uint16_t** g = (const uint16_t**)malloc(sizeof(void*) * (size_t)RM);
    uint16_t** p = (uint16_t**)malloc(sizeof(void*) * (size_t)jb->R);
    if (!g || !p) { free(g); free(p); jb->rc = -2; return NULL; }
    for (int32_t k = 0; k < RM; ++k) g[k] = jb->G[k] + jb->lo;
    for (int32_t r = 0; r < jb->R; ++r) p[r] = jb->P[r] + jb->lo;
    jb->rc = oracle_dp_step(jb->hi - jb->lo, jb->R, jb->M,
                            (const uint16_t* const*)g, jb->W + jb->lo,
                            jb->m + jb->lo, jb->v + jb->lo,
                            (uint16_t* const*)p, jb->hp, jb->step);
    free(g);
    free(p);
    return NULL;
}

int oracle_dp_step_mt(int64_t n, int32_t R, int32_t M,
                      const uint16_t* const* G, float* W, float* m, float* v,
                      uint16_t* const* P, const oracle_hparams* hp,
                      int64_t step, int32_t nthreads)
{
    if (check_args(n, R, M, G, W, m, v, P, hp, step)) return -1;
    if (nthreads <= 1 || n < nthreads)
        return oracle_dp_step(n, R, M, G, W, m, v, P, hp, step);
    mt_job* jobs = (mt_job*)calloc((size_t)nthreads, sizeof(mt_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    char* started = (char*)calloc((size_t)nthreads, 1);
    if (!jobs || !th || !started) { free(jobs); free(th); free(started); return -2; }
    for (int32_t k = 0; k < nthreads; ++k) {
        mt_job* jb = &jobs[k];
        jb->lo = n * k / nthreads;
        jb->hi = n * (k + 1) / nthreads;
        jb->R = R; jb->M = M; jb->G = G; jb->W = W; jb->m = m; jb->v = v;
        jb->P = P; jb->hp = hp; jb->step = step; jb->rc = 0;
        if (pthread_create(&th[k], NULL, mt_run, jb) == 0)
            started[k] = 1;
        else
            mt_run(jb);                  /* run this range on this thread */
    }
    int rc = 0;
    for (int32_t k = 0; k < nthreads; ++k) {
        if (started[k]) pthread_join(th[k], NULL);
        if (jobs[k].rc) rc = jobs[k].rc;
    }
    free(jobs);
    free(th);
    free(started);
    return rc;
}

/* ------------------------------------------------------------ ZeRO step -- */

int64_t oracle_shard_len(int64_t n, int32_t R, int32_t align)
{
    if (n < 0 || R < 1 || align < 1) return -1;
    int64_t per = (n + R - 1) / R;                       /* ceil(n / R) */
    return (per + align - 1) / align * align;            /* roundup     */
}

int oracle_zero_step(int64_t n, int32_t R, int32_t M, int64_t S,
                     const uint16_t* const* G, float* W, float* m, float* v,
                     uint16_t* const* P, const oracle_hparams* hp,
                     int64_t step)
{
    if (check_args(n, R, M, G, W, m, v, P, hp, step)) return -1;
    if (S < 0 || S * R < n) return -1;
    oracle_scalars s;
    oracle_make_scalars(hp, step, R, M, &s);
    int32_t RM = R * M;
    int rc = 0;
    for (int32_t r = 0; r < R && rc == 0; ++r) {        /* card r */
        int64_t lo = (int64_t)r * S;
        int64_t len = n - lo < S ? n - lo : S;
        if (len <= 0) continue;                          /* empty shard  */
        /* 1. reduce-scatter: card r receives chunk r of every rank's
         *    micro-batch gradients (explicit copies, as in the pages' CPU
         *    walkthrough where each card is a separate list element). */
        uint16_t* recv = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)RM * (size_t)len);
        const uint16_t** recv_ptr = (const uint16_t**)malloc(sizeof(void*) * (size_t)RM);
        float* gshard = (float*)malloc(sizeof(float) * (size_t)len);
        uint16_t* pshard = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)len);
        if (!recv || !recv_ptr || !gshard || !pshard) {
            rc = -2;
        } else {
            for (int32_t k = 0; k < RM; ++k) {
                memcpy(recv + (int64_t)k * len, G[k] + lo, sizeof(uint16_t) * (size_t)len);
                recv_ptr[k] = recv + (int64_t)k * len;
            }
            for (int64_t k = 0; k < len; ++k)
                gshard[k] = oracle_avg_grad((const uint16_t* const*)recv_ptr, R, M, k,
                                            s.denom_rm);
            /* 2. card r updates only its own slice of the fp32 state. */
            for (int64_t k = 0; k < len; ++k) {
                oracle_adamw_elem(&s, gshard[k], &W[lo + k], &m[lo + k], &v[lo + k]);
                pshard[k] = oracle_bf16_rne(W[lo + k]);
            }
            /* 3. all-gather: the bf16 shard is copied into every replica. */
            for (int32_t q = 0; q < R; ++q)
                memcpy(P[q] + lo, pshard, sizeof(uint16_t) * (size_t)len);
        }
        free(recv);
        free(recv_ptr);
        free(gshard);
        free(pshard);
    }
    return rc;
}

int oracle_reduce_scatter_sum(int64_t n, int32_t R, int64_t S,
                              const float* const* in, float* const* out)
{
    if (n < 0 || R < 1 || S < 0 || S * R < n || !in || !out) return -1;
    for (int32_t r = 0; r < R; ++r) {
        int64_t lo = (int64_t)r * S;
        int64_t len = n - lo < S ? n - lo : S;
        for (int64_t k = 0; k < len; ++k) {
            float acc = in[0][lo + k];
            for (int32_t q = 1; q < R; ++q) acc = acc + in[q][lo + k];
            out[r][k] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------ ring demo -- */

int oracle_ring_allreduce(float* const* cards, int32_t p, int64_t n,
                          int64_t* sent)
{
    if (p < 1 || n < 0 || !cards || !sent) return -1;
    for (int32_t k = 0; k < p; ++k) sent[k] = 0;
    if (p == 1 || n == 0) return 0;
    int64_t csz = (n + p - 1) / p;                       /* chunk length */
    float* msg = (float*)malloc(sizeof(float) * (size_t)csz * (size_t)p);
    if (!msg) return -2;
#define CH_LO(c) ((int64_t)(c) * csz < n ? (int64_t)(c) * csz : n)
#define CH_HI(c) ((int64_t)((c) + 1) * csz < n ? (int64_t)((c) + 1) * csz : n)
    /* reduce-scatter half: in step s card k sends chunk (k - s) mod p to
     * card k+1, which adds it to its own copy of that chunk.  All cards send
     * at once, so the messages are staged first. */
    for (int32_t s = 0; s < p - 1; ++s) {
        for (int32_t k = 0; k < p; ++k) {
            int32_t c = ((k - s) % p + p) % p;
            int64_t lo = CH_LO(c), hi = CH_HI(c);
            memcpy(msg + (int64_t)k * csz, cards[k] + lo, sizeof(float) * (size_t)(hi - lo));
            sent[k] += hi - lo;
        }
        for (int32_t k = 0; k < p; ++k) {
            int32_t dst = (k + 1) % p;
            int32_t c = ((k - s) % p + p) % p;
            int64_t lo = CH_LO(c), hi = CH_HI(c);
            for (int64_t e = lo; e < hi; ++e)
                cards[dst][e] = cards[dst][e] + msg[(int64_t)k * csz + (e - lo)];
        }
    }
    /* now card k holds the full sum of chunk (k + 1) mod p.  All-gather half:
     * in step s card k passes chunk (k + 1 - s) mod p on; the receiver
     * overwrites its copy. */
    for (int32_t s = 0; s < p - 1; ++s) {
        for (int32_t k = 0; k < p; ++k) {
            int32_t c = ((k + 1 - s) % p + p) % p;
            int64_t lo = CH_LO(c), hi = CH_HI(c);
            memcpy(msg + (int64_t)k * csz, cards[k] + lo, sizeof(float) * (size_t)(hi - lo));
            sent[k] += hi - lo;
        }
        for (int32_t k = 0; k < p; ++k) {
            int32_t dst = (k + 1) % p;
            int32_t c = ((k + 1 - s) % p + p) % p;
            int64_t lo = CH_LO(c), hi = CH_HI(c);
            memcpy(cards[dst] + lo, msg + (int64_t)k * csz, sizeof(float) * (size_t)(hi - lo));
        }
    }
#undef CH_LO
#undef CH_HI
    free(msg);
    return 0;
}

/* ----------------------------------------------------------- accounting -- */

void oracle_zero_bytes(double N, int32_t P, double bp, double bg, double bo,
                       double out[4])
{
    out[0] = N * (bp + bg + bo);
    out[1] = N * (bp + bg) + N * bo / P;
    out[2] = N * bp + N * (bg + bo) / P;
    out[3] = N * (bp + bg + bo) / P;
}

/* ------------------------------------------------------------ clipping -- */

/* the pairwise tree over [lo, lo + len), len a power of two; every leaf is
 * the fp32 product g*g and every node an fp32 sum (reading R10) */
static float sumsq_tree(const float* g, int64_t n, int64_t lo, int64_t len)
{
    if (len == 1) {
        if (lo >= n) return 0.0f;
        float x = g[lo];
        return x * x;
    }
    int64_t half = len / 2;
    if (lo >= n) return 0.0f;                      /* an all-padding subtree */
    float left = sumsq_tree(g, n, lo, half);
    float right = sumsq_tree(g, n, lo + half, half);
    return left + right;
}

double oracle_grad_sumsq(const float* g, int64_t n)
{
    if (n <= 0) return 0.0;
    int64_t len = 1;
    while (len < n) len *= 2;
    return (double)sumsq_tree(g, n, 0, len);
}

float oracle_clip_coef(double sumsq, float max_norm, int32_t* clip)
{
    double norm = sqrt(sumsq);
    double coef = (double)max_norm / (norm + 1e-6);
    if (coef < 1.0) {
        *clip = 1;
        return (float)coef;
    }
    *clip = 0;                 /* also when coef is NaN: no clipping applied */
    return 1.0f;
}

int oracle_dp_step_clipped(int64_t n, int32_t R, int32_t M,
                           const uint16_t* const* G, float* W, float* m, float* v,
                           uint16_t* const* P, const oracle_hparams* hp,
                           int64_t step, float max_norm, int32_t skip_nonfinite,
                           double* sumsq_out, int32_t* skipped_out)
{
    if (check_args(n, R, M, G, W, m, v, P, hp, step)) return -1;
    oracle_scalars s;
    oracle_make_scalars(hp, step, R, M, &s);
    float* g = (float*)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    if (!g) return -2;
    for (int64_t i = 0; i < n; ++i) g[i] = oracle_avg_grad(G, R, M, i, s.denom_rm);
    double sumsq = oracle_grad_sumsq(g, n);
    if (sumsq_out) *sumsq_out = sumsq;
    int32_t skipped = 0;
    if (!isfinite(sumsq) && skip_nonfinite) skipped = 1;
    if (skipped_out) *skipped_out = skipped;
    if (!skipped) {
        int32_t clip = 0;
        float coef = oracle_clip_coef(sumsq, max_norm, &clip);
        for (int64_t i = 0; i < n; ++i) {
            float gi = clip ? g[i] * coef : g[i];
            oracle_adamw_elem(&s, gi, &W[i], &m[i], &v[i]);
            uint16_t p = oracle_bf16_rne(W[i]);
            for (int32_t r = 0; r < R; ++r) P[r][i] = p;
        }
    }
    free(g);
    return 0;
}

/* --------------------------------------------------------------- ZeRO-3 -- */

int oracle_zero3_step(int64_t n, int32_t R, int32_t M, int64_t S,
                      const uint16_t* const* G, float* W, float* m, float* v,
                      uint16_t* Pshard, const oracle_hparams* hp, int64_t step,
                      int64_t* recv)
{
    if (check_args(n, R, M, G, W, m, v, (const void*)Pshard, hp, step)) return -1;
    if (S < 0 || S * R < n) return -1;
    oracle_scalars s;
    oracle_make_scalars(hp, step, R, M, &s);
    int32_t RM = R * M;
    int rc = 0;
    for (int32_t r = 0; r < R && rc == 0; ++r) {        /* card r */
        int64_t lo = (int64_t)r * S;
        int64_t len = n - lo < S ? n - lo : S;
        if (recv) recv[r] = 0;
        if (len <= 0) continue;
        /* reduce-scatter: card r receives chunk r of every rank's gradients
         * (its own M micro-batches stay local) */
        uint16_t* buf = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)RM * (size_t)len);
        const uint16_t** ptr = (const uint16_t**)malloc(sizeof(void*) * (size_t)RM);
        if (!buf || !ptr) {
            rc = -2;
        } else {
            for (int32_t k = 0; k < RM; ++k) {
                memcpy(buf + (int64_t)k * len, G[k] + lo, sizeof(uint16_t) * (size_t)len);
                ptr[k] = buf + (int64_t)k * len;
                /* traffic: one number per other rank and element (a rank sums
                 * its micro-batches locally before the reduce-scatter) */
                if (recv && k % M == 0 && k / M != r) recv[r] += len;
            }
            /* shard update, then the cast into the card's own parameter shard */
            for (int64_t k = 0; k < len; ++k) {
                float g = oracle_avg_grad((const uint16_t* const*)ptr, R, M, k, s.denom_rm);
                oracle_adamw_elem(&s, g, &W[lo + k], &m[lo + k], &v[lo + k]);
                Pshard[lo + k] = oracle_bf16_rne(W[lo + k]);
            }
        }
        free(buf);
        free(ptr);
    }
    return rc;
}

int oracle_zero3_gather(int64_t n, int32_t R, int64_t S, const uint16_t* Pshard,
                        int64_t lo, int64_t hi, int32_t card, uint16_t* out,
                        int64_t* recv)
{
    if (n < 0 || R < 1 || S < 0 || S * R < n || !Pshard || !out) return -1;
    if (lo < 0 || hi < lo || hi > n || card < 0 || card >= R) return -1;
    int64_t from_others = 0;
    for (int64_t i = lo; i < hi; ++i) {
        int32_t owner = (int32_t)(i / S);
        out[i - lo] = Pshard[i];          /* the owner's shard holds element i */
        if (owner != card) ++from_others;
    }
    if (recv) *recv = from_others;
    return 0;
}

/* Reading R16 (zero_oracle.h): the unit's reduce-scatter, card by card. */
int oracle_zero3_rs_unit(int64_t n, int32_t R, int32_t M, int64_t S,
                         const uint16_t* const* Gu, int64_t lo, int64_t hi,
                         float* gshard, int64_t* recv)
{
    if (n < 0 || R < 1 || M < 1 || S < 0 || S * R < n) return -1;
    if (lo < 0 || hi < lo || hi > n) return -1;
    if (hi > lo && (!Gu || !gshard)) return -1;
    float denom_rm = (float)((double)R * (double)M);
    int32_t RM = R * M;
    const uint16_t** ptr = (const uint16_t**)malloc(sizeof(void*) * (size_t)RM);
    if (!ptr) return -1;
    for (int32_t r = 0; r < R; ++r) {                   /* card r */
        int64_t own_lo = (int64_t)r * S, own_hi = own_lo + S;
        if (own_hi > n) own_hi = n;
        int64_t a = lo > own_lo ? lo : own_lo;          /* the unit's part card r owns */
        int64_t b = hi < own_hi ? hi : own_hi;
        if (recv) recv[r] = 0;
        if (b <= a) continue;
        /* every rank's gradient values for [a, b): rank q's buffers hold
         * element i at index i - lo */
        for (int32_t k = 0; k < RM; ++k) {
            ptr[k] = Gu[k] + (a - lo);
            if (recv && k % M == 0 && k / M != r) recv[r] += b - a;
        }
        for (int64_t i = a; i < b; ++i)
            gshard[i] = oracle_avg_grad((const uint16_t* const*)ptr, R, M, i - a, denom_rm);
    }
    free(ptr);
    return 0;
}

int oracle_zero3_update(int64_t n, int32_t R, int32_t M, int64_t S, const float* gshard,
                        float* W, float* m, float* v, uint16_t* Pshard,
                        const oracle_hparams* hp, int64_t step)
{
    if (n < 0 || R < 1 || M < 1 || S < 0 || S * R < n || !hp || step < 1) return -1;
    if (n > 0 && (!gshard || !W || !m || !v || !Pshard)) return -1;
    oracle_scalars s;
    oracle_make_scalars(hp, step, R, M, &s);
    for (int64_t i = 0; i < n; ++i) {        /* each card updates the elements it owns */
        oracle_adamw_elem(&s, gshard[i], &W[i], &m[i], &v[i]);
        Pshard[i] = oracle_bf16_rne(W[i]);
    }
    return 0;
}

/* ----------------------------------------------------------- compression -- */

uint16_t oracle_fp16_rne(float x)
{
    uint32_t u = f2u(x);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);       /* NaN */
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);      /* >= 65520: Inf */
    if (a <= 0x33000000u) return (uint16_t)sign;                  /* <= 2^-25: 0 */
    int32_t e = (int32_t)(a >> 23) - 127;
    if (e >= -14) {
        /* normal: keep 10 of the 23 fraction bits, ties to even; a carry
         * moves into the exponent; re-bias the exponent from 127 to 15 */
        uint32_t r = a + 0xFFFu + ((a >> 13) & 1u);
        r >>= 13;
        return (uint16_t)(sign | (r - ((127u - 15u) << 10)));
    }
    /* subnormal: value / 2^-24 rounded to an integer, ties to even */
    uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;     /* value = mant * 2^(e-23) */
    int32_t shift = -e - 1;                          /* 14 .. 24 */
    uint32_t q = mant >> shift;
    uint32_t rem = mant & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) ++q;
    return (uint16_t)(sign | q);
}

float oracle_fp16_to_float(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu, f = h & 0x3FFu;
    if (e == 0x1F) return u2f(sign | 0x7F800000u | (f << 13));
    if (e == 0) {                                    /* zero or subnormal: f * 2^-24 */
        float v = (float)f * 5.9604644775390625e-08f;
        return sign ? -v : v;
    }
    return u2f(sign | ((e + 127u - 15u) << 23) | (f << 13));
}

/* pairwise fp32 sum of |x| over one block of up to 128 leaves, zero padded */
static float abs_tree(const float* x, int64_t count, int64_t lo, int64_t len)
{
    if (len == 1) return lo < count ? fabsf(x[lo]) : 0.0f;
    if (lo >= count) return 0.0f;
    float a = abs_tree(x, count, lo, len / 2);
    float b = abs_tree(x, count, lo + len / 2, len / 2);
    return a + b;
}

void oracle_compress(int32_t kind, const float* x, int64_t n, float* d)
{
    for (int64_t b0 = 0; b0 < n; b0 += ORACLE_COMP_BLOCK) {
        int64_t cnt = n - b0 < ORACLE_COMP_BLOCK ? n - b0 : ORACLE_COMP_BLOCK;
        const float* xb = x + b0;
        float* db = d + b0;
        if (kind == ORACLE_COMP_FP16) {
            for (int64_t k = 0; k < cnt; ++k) db[k] = oracle_fp16_to_float(oracle_fp16_rne(xb[k]));
        } else if (kind == ORACLE_COMP_INT8) {
            float amax = 0.0f;
            for (int64_t k = 0; k < cnt; ++k) {
                float a = fabsf(xb[k]);
                if (a != a || a > amax) amax = a;   /* a NaN wins, like an unsigned compare */
                if (amax != amax) break;
            }
            float s = amax / 127.0f;
            for (int64_t k = 0; k < cnt; ++k) {
                if (s == 0.0f) {
                    db[k] = 0.0f;
                } else {
                    float q = rintf(xb[k] / s);
                    q = fminf(fmaxf(q, -127.0f), 127.0f);
                    db[k] = q * s;
                }
            }
        } else if (kind == ORACLE_COMP_SIGN) {
            float s = abs_tree(xb, cnt, 0, ORACLE_COMP_BLOCK) / (float)cnt;
            for (int64_t k = 0; k < cnt; ++k) db[k] = xb[k] < 0.0f ? -s : s;
        } else {
            for (int64_t k = 0; k < cnt; ++k) db[k] = xb[k];
        }
    }
}

int oracle_dp_step_compressed(int64_t n, int32_t R, int32_t M,
                              const uint16_t* const* G, float* W, float* m, float* v,
                              uint16_t* const* P, const oracle_hparams* hp,
                              int64_t step, int32_t kind, float* const* E)
{
    if (check_args(n, R, M, G, W, m, v, P, hp, step)) return -1;
    if (kind < ORACLE_COMP_NONE || kind > ORACLE_COMP_SIGN) return -1;
    oracle_scalars s;
    oracle_make_scalars(hp, step, R, M, &s);
    size_t nn = (size_t)(n > 0 ? n : 1);
    float* x = (float*)malloc(sizeof(float) * nn);
    float* d = (float*)malloc(sizeof(float) * nn);
    float* acc = (float*)malloc(sizeof(float) * nn);
    if (!x || !d || !acc) { free(x); free(d); free(acc); return -2; }
    for (int32_t r = 0; r < R; ++r) {
        /* rank r: local accumulation of its micro-batches, error feedback */
        for (int64_t i = 0; i < n; ++i) {
            float loc = oracle_bf16_to_float(G[(int64_t)r * M][i]);
            for (int32_t j = 1; j < M; ++j)
                loc = loc + oracle_bf16_to_float(G[(int64_t)r * M + j][i]);
            x[i] = E ? loc + E[r][i] : loc;
        }
        oracle_compress(kind, x, n, d);
        for (int64_t i = 0; i < n; ++i) {
            if (E) E[r][i] = x[i] - d[i];
            /* the owner adds the decompressed contributions in rank order */
            acc[i] = (r == 0) ? d[i] : acc[i] + d[i];
        }
    }
    for (int64_t i = 0; i < n; ++i) {
        float g = acc[i] / s.denom_rm;
        oracle_adamw_elem(&s, g, &W[i], &m[i], &v[i]);
        uint16_t p = oracle_bf16_rne(W[i]);
        for (int32_t r = 0; r < R; ++r) P[r][i] = p;
    }
    free(x);
    free(d);
    free(acc);
    return 0;
}

/* ------------------------------------------------------------ 1-bit Adam -- */

/* Reading R15 (zero_oracle.h).  The warm-up is the plain step; afterwards
 * the ranks' local momenta are sign-compressed with error feedback, the
 * owner averages them and compresses its shard again with its own error
 * feedback, and the update divides by the frozen preconditioner.  Names
 * follow R15: xr/dr a worker's input and decompressed message, y/ds the
 * server's. */
int oracle_onebit_step(int64_t n, int64_t S, int32_t R, int32_t M,
                       const uint16_t* const* G, float* W, float* m, float* v,
                       uint16_t* const* P, const oracle_hparams* hp, int64_t step,
                       int64_t freeze_step, float* const* E, float* Es)
{
    if (freeze_step < 1 || S < 1 || !E || !Es) return -1;
    if (n > 0 && S * (int64_t)R < n) return -1;
    if (step <= freeze_step)
        return oracle_dp_step(n, R, M, G, W, m, v, P, hp, step);
    if (check_args(n, R, M, G, W, m, v, P, hp, step)) return -1;
    oracle_scalars s;            /* beta1 and lr's bias correction at t */
    oracle_scalars sf;           /* the frozen bias correction of v, at T_w */
    oracle_make_scalars(hp, step, R, M, &s);
    oracle_make_scalars(hp, freeze_step, R, M, &sf);
    size_t nn = (size_t)(n > 0 ? n : 1);
    float* xr = (float*)malloc(sizeof(float) * nn);
    float* dr = (float*)malloc(sizeof(float) * nn);
    float* dsum = (float*)malloc(sizeof(float) * nn);
    if (!xr || !dr || !dsum) { free(xr); free(dr); free(dsum); return -2; }
    float denom_m = (float)M, denom_r = (float)R;
    for (int32_t r = 0; r < R; ++r) {
        /* worker r: local momentum, error feedback, 1-bit compression */
        for (int64_t i = 0; i < n; ++i) {
            float loc = oracle_bf16_to_float(G[(int64_t)r * M][i]);
            for (int32_t j = 1; j < M; ++j)
                loc = loc + oracle_bf16_to_float(G[(int64_t)r * M + j][i]);
            float gl = loc / denom_m;
            float ml = s.beta1 * m[i] + s.one_minus_beta1 * gl;
            xr[i] = ml + E[r][i];
        }
        oracle_compress(ORACLE_COMP_SIGN, xr, n, dr);
        for (int64_t i = 0; i < n; ++i) {
            E[r][i] = xr[i] - dr[i];
            dsum[i] = (r == 0) ? dr[i] : dsum[i] + dr[i];
        }
    }
    /* server: the owner of each shard averages, adds its residual and
     * compresses again, blocks counted from the shard's start */
    float* y = xr;
    float* ds = dr;
    for (int64_t i = 0; i < n; ++i) y[i] = dsum[i] / denom_r + Es[i];
    for (int32_t r = 0; r < R; ++r) {
        int64_t lo = (int64_t)r * S;
        if (lo >= n) break;
        int64_t len = n - lo < S ? n - lo : S;
        oracle_compress(ORACLE_COMP_SIGN, y + lo, len, ds + lo);
    }
    for (int64_t i = 0; i < n; ++i) {
        Es[i] = y[i] - ds[i];
        float mi = ds[i];
        float wd = W[i] * s.decay;
        float root = sqrtf(v[i]);
        float q = root / sf.bc2_sqrt;
        float den = q + s.eps;
        float ratio = mi / den;
        float upd = s.step_size * ratio;
        W[i] = wd - upd;
        m[i] = mi;
        uint16_t p = oracle_bf16_rne(W[i]);
        for (int32_t r = 0; r < R; ++r) P[r][i] = p;
    }
    free(xr);
    free(dr);
    free(dsum);
    return 0;
}
