/*
 * zgen_dev.cu - device fill kernels of the seeded input generator (zgen.h).
 * The values are bit-identical to zgen_host.c's host fills.  Each thread
 * writes elements i0 + k for k = tid, tid + stride, ... < n: every store is
 * inside [out, out + n).
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "zgen.h"

static __global__ void k_fill_grad(uint16_t* __restrict__ out, int64_t i0, int64_t n,
                                   uint64_t key, float scale, float outlier,
                                   uint32_t pct)
{
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride)
        out[k] = zgen_grad_bf16(key, i0 + k, scale, outlier, pct);
}

static __global__ void k_fill_state(float* __restrict__ out, int64_t i0, int64_t n,
                                    uint64_t key, float scale, int32_t square)
{
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride)
        out[k] = zgen_state_f32(key, i0 + k, scale, square);
}

static __global__ void k_fill_const(float* __restrict__ out, int64_t n, float value)
{
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride)
        out[k] = value;
}

static unsigned grid_for(int64_t n)
{
    int64_t b = (n + 255) / 256;
    if (b > 152 * 32) b = 152 * 32;
    return (unsigned)(b < 1 ? 1 : b);
}

extern "C" int zgen_dev_fill_grad_bf16(uint16_t* out, int64_t i0, int64_t n, uint64_t seed,
                                       uint64_t stream, float scale, float outlier,
                                       uint32_t outlier_pct, void* cuda_stream)
{
    if (n <= 0) return 0;
    k_fill_grad<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
        out, i0, n, zgen_key(seed, stream), scale, outlier, outlier_pct);
    return (int)cudaGetLastError();
}

extern "C" int zgen_dev_fill_state_f32(float* out, int64_t i0, int64_t n, uint64_t seed,
                                       uint64_t stream, float scale, int32_t square,
                                       void* cuda_stream)
{
    if (n <= 0) return 0;
    k_fill_state<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
        out, i0, n, zgen_key(seed, stream), scale, square);
    return (int)cudaGetLastError();
}

extern "C" int zgen_dev_fill_const_f32(float* out, int64_t n, float value, void* cuda_stream)
{
    if (n <= 0) return 0;
    k_fill_const<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(out, n, value);
    return (int)cudaGetLastError();
}
