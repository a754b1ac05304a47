/*
 * zgen.h - seeded, counter-based input generator for the ZeRO AdamW step.
 *
 * This module makes the synthetic inputs (bf16 gradients, fp32 master
 * weights and Adam moments).  It is the one module that both the CUDA path's
 * tests/benchmark (device fill kernels, zgen_dev.cu) and the CPU oracle's
 * callers (host fill routines, zgen_host.c) use, so it holds none of the
 * optimizer step's arithmetic: no summation, no AdamW, no bf16 rounding.
 *
 * Every value is a pure function of (seed, stream, index), so any element
 * of any buffer can be produced on its own, on the host or on the device,
 * with identical bits:
 *
 *   key      = SplitMix64 finaliser of (seed * GAMMA + stream + 1)
 *   h_k(i)   = SplitMix64 finaliser of (key + (4*i + k + 1) * GAMMA), k = 0..3
 *
 * i.e. h_k(i) is output 4i+k of a SplitMix64 generator seeded with `key`
 * (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014: the generator adds GAMMA to its state and passes the state
 * through the 64-bit finaliser below).
 *
 * Normal-like values use the Irwin-Hall construction: the eight 16-bit
 * lanes of h_0 and h_1 are summed, centred and scaled,
 *   s = 2 * (sum of lanes) - 8 * 65535     (an odd integer, |s| < 2^20)
 *   x = (float)s * scale,                  scale = sigma / ZGEN_IH_STD
 * which has mean 0, standard deviation sigma, and is bounded by about
 * 4.9 sigma.  Only exactly rounded operations are used (an integer to float
 * conversion that is exact, and one IEEE multiply), so host and device agree
 * bit for bit.  bf16 values are the high half of the float (truncation), and
 * an optional outlier replaces the value with +-outlier when h_2 mod 100 is
 * below the requested percentage.
 */
#ifndef ZGEN_H
#define ZGEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define ZGEN_HD __host__ __device__ __forceinline__
#else
#define ZGEN_HD static inline
#endif

#define ZGEN_GAMMA 0x9E3779B97F4A7C15ull
/* standard deviation of s = 2*sum(8 uniform 16-bit lanes) - 8*65535:
 * sqrt(8 * 4 * (65536^2 - 1) / 12) */
#define ZGEN_IH_STD 107019.57184877197

ZGEN_HD uint64_t zgen_mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

ZGEN_HD uint64_t zgen_key(uint64_t seed, uint64_t stream)
{
    return zgen_mix64(seed * ZGEN_GAMMA + stream + 1ull);
}

ZGEN_HD uint64_t zgen_h(uint64_t key, int64_t i, int k)
{
    return zgen_mix64(key + ((uint64_t)i * 4ull + (uint64_t)k + 1ull) * ZGEN_GAMMA);
}

/* centred Irwin-Hall integer of element i (odd, |s| <= 524280) */
ZGEN_HD int32_t zgen_ih(uint64_t key, int64_t i)
{
    uint64_t a = zgen_h(key, i, 0), b = zgen_h(key, i, 1);
    int32_t sum = 0;
    for (int l = 0; l < 4; ++l) {
        sum += (int32_t)((a >> (16 * l)) & 0xFFFFu);
        sum += (int32_t)((b >> (16 * l)) & 0xFFFFu);
    }
    return 2 * sum - 8 * 65535;
}

ZGEN_HD float zgen_mul(float a, float b)
{
#if defined(__CUDA_ARCH__)
    return __fmul_rn(a, b);
#else
    return a * b;
#endif
}

ZGEN_HD uint32_t zgen_f2u(float x)
{
#if defined(__CUDA_ARCH__)
    return (uint32_t)__float_as_uint(x);
#else
    union { float f; uint32_t u; } c;
    c.f = x;
    return c.u;
#endif
}

/* fp32 normal-like value of element i: (float)s * scale */
ZGEN_HD float zgen_normal(uint64_t key, int64_t i, float scale)
{
    return zgen_mul((float)zgen_ih(key, i), scale);
}

/* bf16 bits of a gradient element: the normal-like value, or +-outlier with
 * probability outlier_pct/100, truncated to its high 16 bits. */
ZGEN_HD uint16_t zgen_grad_bf16(uint64_t key, int64_t i, float scale,
                                float outlier, uint32_t outlier_pct)
{
    float x = zgen_normal(key, i, scale);
    if (outlier_pct) {
        uint64_t c = zgen_h(key, i, 2);
        if ((uint32_t)(c % 100ull) < outlier_pct)
            x = (c >> 63) ? -outlier : outlier;
    }
    return (uint16_t)(zgen_f2u(x) >> 16);
}

/* fp32 value of a state element; square != 0 returns x*x (a non-negative
 * second-moment-like value). */
ZGEN_HD float zgen_state_f32(uint64_t key, int64_t i, float scale, int square)
{
    float x = zgen_normal(key, i, scale);
    return square ? zgen_mul(x, x) : x;
}

#endif
