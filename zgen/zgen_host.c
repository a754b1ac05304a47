/*
 * zgen_host.c - host fill routines of the seeded input generator (zgen.h).
 * Plain C; the values are bit-identical to zgen_dev.cu's device fills.
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared
 */
#include "zgen.h"

/* out[k] = gradient element i0 + k, k < n */
void zgen_fill_grad_bf16(uint16_t* out, int64_t i0, int64_t n, uint64_t seed,
                         uint64_t stream, float scale, float outlier,
                         uint32_t outlier_pct)
{
    uint64_t key = zgen_key(seed, stream);
    for (int64_t k = 0; k < n; ++k)
        out[k] = zgen_grad_bf16(key, i0 + k, scale, outlier, outlier_pct);
}

/* out[k] = gradient element idx[k] */
void zgen_gather_grad_bf16(uint16_t* out, const int64_t* idx, int64_t n,
                           uint64_t seed, uint64_t stream, float scale,
                           float outlier, uint32_t outlier_pct)
{
    uint64_t key = zgen_key(seed, stream);
    for (int64_t k = 0; k < n; ++k)
        out[k] = zgen_grad_bf16(key, idx[k], scale, outlier, outlier_pct);
}

void zgen_fill_state_f32(float* out, int64_t i0, int64_t n, uint64_t seed,
                         uint64_t stream, float scale, int32_t square)
{
    uint64_t key = zgen_key(seed, stream);
    for (int64_t k = 0; k < n; ++k)
        out[k] = zgen_state_f32(key, i0 + k, scale, square);
}

void zgen_gather_state_f32(float* out, const int64_t* idx, int64_t n,
                           uint64_t seed, uint64_t stream, float scale,
                           int32_t square)
{
    uint64_t key = zgen_key(seed, stream);
    for (int64_t k = 0; k < n; ++k)
        out[k] = zgen_state_f32(key, idx[k], scale, square);
}

/* raw 64-bit draw number `draw` of stream (seed, stream): used for the
 * workload recipes' integer draws (tensor sizes of the uneven workload). */
uint64_t zgen_draw_u64(uint64_t seed, uint64_t stream, int64_t draw)
{
    return zgen_h(zgen_key(seed, stream), draw, 3);
}
