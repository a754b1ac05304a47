// zero_step.cu - sm_103a kernels and C-ABI entry points of the ZeRO-1/2
// mixed-precision AdamW step (declared in include/zero_step.h).
//
// The step is HBM-bound elementwise work (under 1 flop per byte), so there
// is no tensor-core contraction here: the kernels stream 16-byte/8-byte
// coalesced vectors through registers with evict-first cache hints, run a
// persistent grid of (SM count x resident blocks), and keep the fp32
// arithmetic in the fixed order the header defines, every operation
// rounded on its own (__fadd_rn / __fmul_rn / __fdiv_rn / __fsqrt_rn keep
// nvcc from contracting into FMA).
//
// Kernels
//   k_fused      reduce-scatter + average, AdamW and bf16 all-gather of each
//                element in one pass: 2RM + 24 + 2R bytes per parameter.
//   k_rs_avg     staged step 1: per shard, ordered fp32 sum / (R*M) into an
//                fp32 scratch shard (2RM + 4 bytes per parameter).
//   k_adamw      staged step 2: AdamW of each shard from the scratch
//                gradient (4 + 24 bytes per parameter).
//   k_ag_cast    staged step 3: bf16 cast of each shard written into all R
//                replicas (4 + 2R bytes per parameter).
//
// Work decomposition: a "vector" is 4 consecutive elements (8 bytes of each
// bf16 stream, 16 bytes of each fp32 stream), so one warp instruction moves
// 256 or 512 contiguous bytes.  The fused kernel walks tiles of
// 256 threads x 4 elements x U units per block (grid-stride over tiles);
// the last partial tile is done element by element.  The staged kernels
// give each rank r its own grid row (blockIdx.y = r) and grid-stride over
// the vectors of shard r, as rank r would on its own GPU.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>
#include <cmath>
#include <mutex>
#include <unordered_map>

#include "zero_step.h"

namespace {

constexpr int kThreads = 256;
constexpr int kVec = 4;                     // elements per thread per unit
constexpr int kUnit = kThreads * kVec;      // elements per block per unit

// ------------------------------------------------------------- scalars --

struct StepScalars {
    float step_size;      // lr / (1 - beta1^t)
    float bc2_sqrt;       // sqrt(1 - beta2^t)
    float decay;          // 1 - lr * wd
    float b1, b2;
    float omb1, omb2;     // 1 - beta1, 1 - beta2
    float eps;
    float denom_rm;       // (float)(R * M)
    float inv_rm;         // 1 / (R * M) when R*M is a power of two
    int32_t rm_pow2;      // dividing by 2^k equals multiplying by 2^-k exactly
};

StepScalars step_scalars(const zero_adamw_hparams& hp, int64_t step, int R, int M)
{
    StepScalars s;
    const double t = (double)step;
    const double b1 = hp.beta1, b2 = hp.beta2, lr = hp.lr, wd = hp.weight_decay;
    const double bias1 = 1.0 - std::pow(b1, t);
    const double bias2 = 1.0 - std::pow(b2, t);
    s.step_size = (float)(lr / bias1);
    s.bc2_sqrt = (float)std::sqrt(bias2);
    s.decay = (float)(1.0 - lr * wd);
    s.b1 = hp.beta1;
    s.b2 = hp.beta2;
    s.omb1 = (float)(1.0 - b1);
    s.omb2 = (float)(1.0 - b2);
    s.eps = hp.eps;
    const int rm = R * M;
    s.denom_rm = (float)rm;
    s.rm_pow2 = (rm & (rm - 1)) == 0;
    s.inv_rm = s.rm_pow2 ? 1.0f / (float)rm : 0.0f;
    return s;
}

// ------------------------------------------------------- kernel params --

struct GradPtrs { const uint16_t* p[ZERO_MAX_RM]; };
struct ReplicaPtrs { uint16_t* p[ZERO_MAX_R]; };

struct FusedArgs {
    GradPtrs g;
    ReplicaPtrs P;
    float* W;
    float* m;
    float* v;
    int64_t n;
    int32_t R, M;
    StepScalars s;
    int32_t* status;
    uint16_t* extra_rep;  // optional extra copy of the replica (e.g. in host memory)
    int32_t zero3;        // host-side dispatch: write one sharded buffer (P.p[0])
};

struct StagedArgs {
    GradPtrs g;
    ReplicaPtrs P;
    const float* gs;      // scratch gradient (rs_avg writes it, adamw reads it)
    float* gs_out;
    float* W;
    float* m;
    float* v;
    int64_t n, S;
    int32_t R, M;
    StepScalars s;
    int32_t* status;
};

// ------------------------------------------------------ device helpers --

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_bits(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Round to nearest even; every NaN becomes the quiet NaN 0x7FC0.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    uint32_t u = *reinterpret_cast<uint32_t*>(&h);
    if (lo != lo) u = (u & 0xFFFF0000u) | 0x7FC0u;
    if (hi != hi) u = (u & 0x0000FFFFu) | 0x7FC00000u;
    return u;
}

__device__ __forceinline__ uint16_t to_bf16(float x)
{
    if (x != x) return (uint16_t)0x7FC0u;
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float scale_grad(const StepScalars& s, float acc)
{
    return s.rm_pow2 ? __fmul_rn(acc, s.inv_rm) : __fdiv_rn(acc, s.denom_rm);
}

// AdamW on one element, in the header's operation order.
__device__ __forceinline__ void adamw(const StepScalars& s, float g, float& w, float& m,
                                      float& v)
{
    const float wd = __fmul_rn(w, s.decay);
    const float m1 = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
    const float v1 = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(__fmul_rn(s.omb2, g), g));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v1), s.bc2_sqrt), s.eps);
    w = __fsub_rn(wd, __fmul_rn(s.step_size, __fdiv_rn(m1, den)));
    m = m1;
    v = v1;
}

__device__ __forceinline__ uint2 ld_stream(const uint16_t* p)
{
    return __ldcs(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ float4 ld_stream(const float* p)
{
    return __ldcs(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ void st_stream(uint16_t* p, uint2 x)
{
    __stcs(reinterpret_cast<uint2*>(p), x);
}
__device__ __forceinline__ void st_stream(float* p, float4 x)
{
    __stcs(reinterpret_cast<float4*>(p), x);
}

__device__ __forceinline__ void fold4(float (&loc)[4], float (&tot)[4], uint2 x, int r, int j,
                                      int M)
{
    const float e[4] = {bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y)};
#pragma unroll
    for (int k = 0; k < 4; ++k) loc[k] = j == 0 ? e[k] : __fadd_rn(loc[k], e[k]);
    if (j == M - 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) tot[k] = r == 0 ? loc[k] : __fadd_rn(tot[k], loc[k]);
    }
}

// Ordered fp32 sum of the R*M gradients at the 4 elements starting at e:
// each rank's micro-batches first (j ascending), then ranks ascending.
// RC/MC are compile-time R and M, or 0 for run-time values; with both known
// every load is issued before the first add.
template <int RC, int MC>
__device__ __forceinline__ void grad_sum4(const GradPtrs& g, int R, int M, int64_t e,
                                          float (&tot)[4])
{
    float loc[4];
    if constexpr (RC > 0 && MC > 0) {
        uint2 x[RC * MC];
#pragma unroll
        for (int q = 0; q < RC * MC; ++q) x[q] = ld_stream(g.p[q] + e);
#pragma unroll
        for (int r = 0; r < RC; ++r)
#pragma unroll
            for (int j = 0; j < MC; ++j) fold4(loc, tot, x[r * MC + j], r, j, MC);
    } else {
        constexpr int B = 8;              // loads in flight per batch
        const int RM = R * M;
        int r = 0, j = 0;
        for (int q0 = 0; q0 < RM; q0 += B) {
            uint2 x[B];
#pragma unroll
            for (int b = 0; b < B; ++b)
                if (q0 + b < RM) x[b] = ld_stream(g.p[q0 + b] + e);
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (q0 + b < RM) {
                    fold4(loc, tot, x[b], r, j, M);
                    if (++j == M) { j = 0; ++r; }
                }
            }
        }
    }
}

__device__ __forceinline__ float grad_sum1(const GradPtrs& g, int R, int M, int64_t i)
{
    float tot = 0.0f;
    for (int r = 0; r < R; ++r) {
        float loc = bf16_bits(g.p[r * M][i]);
        for (int j = 1; j < M; ++j) loc = __fadd_rn(loc, bf16_bits(g.p[r * M + j][i]));
        tot = r == 0 ? loc : __fadd_rn(tot, loc);
    }
    return tot;
}

template <bool CHECK>
__device__ __forceinline__ void report_nonfinite(bool bad, int32_t* status)
{
    if constexpr (CHECK) {
        if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0 && status)
            atomicOr(status, ZERO_DEV_NONFINITE);
    }
}

// ------------------------------------------------------ launch helpers --

struct DevInfo {
    int sms = 0;
    std::unordered_map<const void*, int> occ;
};

std::mutex g_mu;
DevInfo g_dev[64];

int device_sms(int dev)
{
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo& d = g_dev[dev & 63];
    if (d.sms == 0) cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    return d.sms > 0 ? d.sms : 1;
}

int blocks_per_sm(int dev, const void* kernel)
{
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo& d = g_dev[dev & 63];
    auto it = d.occ.find(kernel);
    if (it != d.occ.end()) return it->second;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kThreads, 0) != cudaSuccess ||
        nb < 1)
        nb = 1;
    d.occ[kernel] = nb;
    return nb;
}

// persistent grid: every SM gets its resident blocks, capped by the work.
// quarter_blocks > 0 caps it further at quarter_blocks / 4 blocks per SM
// once every block has at least 4 work units: for some kernels a sweep of
// grid sizes on GB300 found HBM busier with fewer blocks than fit (the
// launch sites give the measured values), while smaller launches, bound by
// latency and ramp-up, run faster with every block that fits.
unsigned grid_for(const void* kernel, int64_t work_blocks, int quarter_blocks = 0)
{
    int dev = 0;
    cudaGetDevice(&dev);
    int64_t cap = (int64_t)device_sms(dev) * blocks_per_sm(dev, kernel);
    if (quarter_blocks > 0 && work_blocks >= 4 * cap) {
        const int64_t q = (int64_t)quarter_blocks * device_sms(dev) / 4;
        if (q >= 1 && q < cap) cap = q;
    }
    int64_t g = work_blocks < cap ? work_blocks : cap;
    return (unsigned)(g < 1 ? 1 : g);
}

// ---------------------------------------------------------- fused step --

// OUT selects where the bf16 result goes, as a template switch so the plain
// path carries no extra branch or register pressure:
//   0  the R replicas a.P.p[0..R)                       (ZeRO-1/2 all-gather)
//   1  the R replicas and a.extra_rep (the host-buffer entry point's
//      zero-copy mode writes replica 0 to host memory as well)
//   2  one buffer a.P.p[0] in the padded layout of the state: each rank
//      casts into its own parameter shard, no all-gather   (ZeRO-3)
template <int RC, int MC, int U, bool CHECK, int OUT>
__global__ void __launch_bounds__(kThreads) k_fused(const __grid_constant__ FusedArgs a)
{
    const int R = RC > 0 ? RC : a.R;
    const int M = MC > 0 ? MC : a.M;
    constexpr int T = kUnit * U;
    const int64_t n = a.n;
    const int64_t full_tiles = n / T;
    bool bad = false;

    for (int64_t tile = blockIdx.x; tile < full_tiles; tile += gridDim.x) {
        const int64_t e0 = tile * T + (int64_t)threadIdx.x * kVec;
        float acc[U][4];
        float4 w[U], mm[U], vv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t e = e0 + (int64_t)u * kUnit;
            w[u] = ld_stream(a.W + e);
            mm[u] = ld_stream(a.m + e);
            vv[u] = ld_stream(a.v + e);
            grad_sum4<RC, MC>(a.g, R, M, e, acc[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t e = e0 + (int64_t)u * kUnit;
            float* wp = &w[u].x;
            float* mp = &mm[u].x;
            float* vp = &vv[u].x;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float g = scale_grad(a.s, acc[u][k]);
                if (CHECK) bad |= !isfinite(g);
                adamw(a.s, g, wp[k], mp[k], vp[k]);
            }
            st_stream(a.W + e, w[u]);
            st_stream(a.m + e, mm[u]);
            st_stream(a.v + e, vv[u]);
            const uint2 p = make_uint2(pack_bf16x2(w[u].x, w[u].y), pack_bf16x2(w[u].z, w[u].w));
            if constexpr (OUT == 2) {
                st_stream(a.P.p[0] + e, p);
            } else if constexpr (RC > 0) {
#pragma unroll
                for (int r = 0; r < RC; ++r) st_stream(a.P.p[r] + e, p);
            } else {
                for (int r = 0; r < R; ++r) st_stream(a.P.p[r] + e, p);
            }
            if constexpr (OUT == 1) st_stream(a.extra_rep + e, p);
        }
    }

    // last partial tile, element by element, by the block that owns it
    const int64_t tail0 = full_tiles * T;
    if (tail0 < n && blockIdx.x == (unsigned)(full_tiles % gridDim.x)) {
        for (int64_t i = tail0 + threadIdx.x; i < n; i += kThreads) {
            const float g = scale_grad(a.s, grad_sum1(a.g, R, M, i));
            if (CHECK) bad |= !isfinite(g);
            float w = a.W[i], m = a.m[i], v = a.v[i];
            adamw(a.s, g, w, m, v);
            a.W[i] = w;
            a.m[i] = m;
            a.v[i] = v;
            const uint16_t p = to_bf16(w);
            if constexpr (OUT == 2) {
                a.P.p[0][i] = p;
            } else {
                for (int r = 0; r < R; ++r) a.P.p[r][i] = p;
            }
            if constexpr (OUT == 1) a.extra_rep[i] = p;
        }
    }
    report_nonfinite<CHECK>(bad, a.status);
}

// ----------------------------------------------------- fused dispatch --

// Blocks per SM (in quarters) of k_fused where fewer than the resident
// maximum measured faster: whole-step time against grid size on GB300
// (152 SMs) over the 1B- and 4B-shaped workloads and flat vectors of 0.4 to
// 2 G params.  R=2: 2 blocks/SM, 0.93-0.94 -> 0.98 of the copy peak (4
// resident).  R=4: 2.5, 0.94-0.95 -> 0.97 (4 resident).  ZeRO-3 output with
// R=8: 2.75, 0.95-0.96 -> 0.98; with R=4: 3, 0.95 -> 0.98 (4 resident).  0
// keeps the resident maximum (R=8 runs 2 blocks/SM, its maximum).
template <int RC, int MC, int OUT>
constexpr int fused_quarter_blocks()
{
    if (MC != 1) return 0;
    if (OUT == 0) return RC == 2 ? 8 : RC == 4 ? 10 : 0;
    if (OUT == 2) return RC == 8 ? 11 : RC == 4 ? 12 : 0;
    return 0;
}

template <int RC, int MC, bool CHECK, int OUT = 0>
cudaError_t launch_fused_t(const FusedArgs& a, cudaStream_t st)
{
    constexpr int U = 2;
    const void* k = reinterpret_cast<const void*>(&k_fused<RC, MC, U, CHECK, OUT>);
    const int64_t tiles = (a.n + kUnit * U - 1) / (kUnit * U);
    const unsigned grid = grid_for(k, tiles, fused_quarter_blocks<RC, MC, OUT>());
    k_fused<RC, MC, U, CHECK, OUT><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <bool CHECK, int OUT>
cudaError_t launch_fused_table(const FusedArgs& a, cudaStream_t st)
{
    const int R = a.R, M = a.M;
#define ZERO_CASE(r_, m_) \
    if (R == r_ && M == m_) return launch_fused_t<r_, m_, CHECK, OUT>(a, st);
    ZERO_CASE(8, 1) ZERO_CASE(4, 1) ZERO_CASE(2, 1) ZERO_CASE(1, 1) ZERO_CASE(16, 1)
    ZERO_CASE(4, 2) ZERO_CASE(7, 4) ZERO_CASE(8, 2) ZERO_CASE(4, 4) ZERO_CASE(2, 2)
#undef ZERO_CASE
    return launch_fused_t<0, 0, CHECK, OUT>(a, st);
}

template <bool CHECK>
cudaError_t launch_fused(const FusedArgs& a, cudaStream_t st)
{
    // the zero-copy host path is bound by the host link, not by HBM: one
    // run-time (R, M) instantiation serves it
    if (a.extra_rep) return launch_fused_t<0, 0, CHECK, 1>(a, st);
    if (a.zero3) return launch_fused_table<CHECK, 2>(a, st);
    return launch_fused_table<CHECK, 0>(a, st);
}

// ================================================== end of the fused path ==
// (everything above is what k_fused and its launch are compiled from)

// ------------------------------------------------------- staged steps --
// Shard r = blockIdx.y covers [r*S, r*S + len), len = min(S, n - r*S).
// S is a multiple of 4, so every shard starts on a vector boundary.
// k_rs_avg walks tiles of one or two units from the shard start, k_adamw
// 4-vectors, and k_ag_cast 8-element vectors that start on the shard's first
// multiple of 8 (one 16-byte store per replica), with the head and tail done
// element by element.

__device__ __forceinline__ int64_t shard_len(int64_t n, int64_t S, int r)
{
    const int64_t lo = (int64_t)r * S;
    const int64_t len = n - lo < S ? n - lo : S;
    return len > 0 ? len : 0;
}

template <int RC, int MC, bool CHECK>
__global__ void __launch_bounds__(kThreads) k_rs_avg(const __grid_constant__ StagedArgs a)
{
    const int R = RC > 0 ? RC : a.R;
    const int M = MC > 0 ? MC : a.M;
    const int r = blockIdx.y;
    const int64_t lo = (int64_t)r * a.S, len = shard_len(a.n, a.S, r);
    // two units per tile while R*M is small; with many source buffers one
    // unit already keeps R*M loads in flight per thread
    constexpr int U = (RC > 0 && RC * MC <= 16) ? 2 : 1;
    constexpr int T = kUnit * U;              // tiles of U*1024 elements from the shard start
    const int64_t full_tiles = len / T;
    bool bad = false;
    for (int64_t tile = blockIdx.x; tile < full_tiles; tile += gridDim.x) {
        const int64_t e0 = lo + tile * T + (int64_t)threadIdx.x * kVec;
        float acc[U][4];
#pragma unroll
        for (int u = 0; u < U; ++u) grad_sum4<RC, MC>(a.g, R, M, e0 + (int64_t)u * kUnit, acc[u]);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float4 o;
            o.x = scale_grad(a.s, acc[u][0]);
            o.y = scale_grad(a.s, acc[u][1]);
            o.z = scale_grad(a.s, acc[u][2]);
            o.w = scale_grad(a.s, acc[u][3]);
            if (CHECK) bad |= !(isfinite(o.x) && isfinite(o.y) && isfinite(o.z) && isfinite(o.w));
            st_stream(a.gs_out + e0 + (int64_t)u * kUnit, o);
        }
    }
    // the shard's last partial tile, element by element, by the block that owns it
    const int64_t tail0 = lo + full_tiles * T;
    if (tail0 < lo + len && blockIdx.x == (unsigned)(full_tiles % gridDim.x)) {
        for (int64_t i = tail0 + threadIdx.x; i < lo + len; i += kThreads) {
            const float g = scale_grad(a.s, grad_sum1(a.g, R, M, i));
            if (CHECK) bad |= !isfinite(g);
            a.gs_out[i] = g;
        }
    }
    report_nonfinite<CHECK>(bad, a.status);
}

__global__ void __launch_bounds__(kThreads) k_adamw(const __grid_constant__ StagedArgs a)
{
    const int r = blockIdx.y;
    const int64_t lo = (int64_t)r * a.S, len = shard_len(a.n, a.S, r);
    const int64_t nvec = len / kVec;
    for (int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x; q < nvec;
         q += (int64_t)gridDim.x * kThreads) {
        const int64_t e = lo + q * kVec;
        const float4 g = ld_stream(a.gs + e);
        float4 w = ld_stream(a.W + e), m = ld_stream(a.m + e), v = ld_stream(a.v + e);
        adamw(a.s, g.x, w.x, m.x, v.x);
        adamw(a.s, g.y, w.y, m.y, v.y);
        adamw(a.s, g.z, w.z, m.z, v.z);
        adamw(a.s, g.w, w.w, m.w, v.w);
        st_stream(a.W + e, w);
        st_stream(a.m + e, m);
        st_stream(a.v + e, v);
    }
    if (blockIdx.x == 0) {
        for (int64_t i = lo + nvec * kVec + threadIdx.x; i < lo + len; i += kThreads) {
            float w = a.W[i], m = a.m[i], v = a.v[i];
            adamw(a.s, a.gs[i], w, m, v);
            a.W[i] = w;
            a.m[i] = m;
            a.v[i] = v;
        }
    }
}

template <int RC>
__global__ void __launch_bounds__(kThreads) k_ag_cast(const __grid_constant__ StagedArgs a)
{
    // 8 elements per thread: two float4 loads of W, one 16-byte store per
    // replica.  A shard starts on a multiple of 4 elements only, so the vector
    // loop starts at the shard's first multiple of 8; the head before it and
    // the tail after the last full vector are done element by element.
    const int R = RC > 0 ? RC : a.R;
    const int r = blockIdx.y;
    const int64_t lo = (int64_t)r * a.S, len = shard_len(a.n, a.S, r);
    const int64_t hi = lo + len;
    const int64_t v0 = (lo + 7) / 8 * 8;                  // first 8-aligned element
    const int64_t n8 = hi > v0 ? (hi - v0) / 8 : 0;
    for (int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x; q < n8;
         q += (int64_t)gridDim.x * kThreads) {
        const int64_t e = v0 + q * 8;
        const float4 w0 = ld_stream(a.W + e), w1 = ld_stream(a.W + e + 4);
        const uint4 p = make_uint4(pack_bf16x2(w0.x, w0.y), pack_bf16x2(w0.z, w0.w),
                                   pack_bf16x2(w1.x, w1.y), pack_bf16x2(w1.z, w1.w));
        if constexpr (RC > 0) {
#pragma unroll
            for (int k = 0; k < RC; ++k) __stcs(reinterpret_cast<uint4*>(a.P.p[k] + e), p);
        } else {
            for (int k = 0; k < R; ++k) __stcs(reinterpret_cast<uint4*>(a.P.p[k] + e), p);
        }
    }
    if (blockIdx.x == 0) {
        const int64_t head_end = v0 < hi ? v0 : hi;
        for (int64_t i = lo + threadIdx.x; i < head_end; i += kThreads) {
            const uint16_t p = to_bf16(a.W[i]);
            for (int k = 0; k < R; ++k) a.P.p[k][i] = p;
        }
        for (int64_t i = v0 + n8 * 8 + threadIdx.x; i < hi; i += kThreads) {
            const uint16_t p = to_bf16(a.W[i]);
            for (int k = 0; k < R; ++k) a.P.p[k][i] = p;
        }
    }
}


template <bool CHECK>
cudaError_t launch_rs(const StagedArgs& a, cudaStream_t st)
{
    const int R = a.R, M = a.M;
    const int64_t work = (a.S + kUnit - 1) / kUnit;      // at most one block per unit of a shard
    // 4 blocks per SM (6 or 8 fit): 0.941 -> 0.957 of the copy peak for the
    // staged step on the R=7, M=4 workload, +0.3-0.5 % on the others (grid-size
    // sweep)
    auto go = [&](const void* k, auto kern) {
        const int64_t per_rank = (int64_t)grid_for(k, work * a.R, 16) / a.R;    // never past one wave
        dim3 grid((unsigned)(per_rank < 1 ? 1 : per_rank), (unsigned)a.R);
        kern<<<grid, kThreads, 0, st>>>(a);
        return cudaGetLastError();
    };
#define ZERO_CASE(r_, m_)                                                      \
    if (R == r_ && M == m_)                                                    \
        return go(reinterpret_cast<const void*>(&k_rs_avg<r_, m_, CHECK>),     \
                  k_rs_avg<r_, m_, CHECK>);
    ZERO_CASE(8, 1) ZERO_CASE(4, 1) ZERO_CASE(2, 1) ZERO_CASE(1, 1) ZERO_CASE(16, 1)
    ZERO_CASE(4, 2) ZERO_CASE(7, 4) ZERO_CASE(8, 2) ZERO_CASE(4, 4) ZERO_CASE(2, 2)
#undef ZERO_CASE
    return go(reinterpret_cast<const void*>(&k_rs_avg<0, 0, CHECK>), k_rs_avg<0, 0, CHECK>);
}

cudaError_t launch_adamw(const StagedArgs& a, cudaStream_t st)
{
    const void* k = reinterpret_cast<const void*>(&k_adamw);
    const int64_t work = (a.S / kVec + kThreads - 1) / kThreads;
    const int64_t per_rank = (int64_t)grid_for(k, work * a.R) / a.R;    // never past one wave
    dim3 grid((unsigned)(per_rank < 1 ? 1 : per_rank), (unsigned)a.R);
    k_adamw<<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_ag(const StagedArgs& a, cudaStream_t st)
{
    const int64_t work = (a.S / 8 + kThreads - 1) / kThreads;
    auto go = [&](const void* k, auto kern) {
        const int64_t per_rank = (int64_t)grid_for(k, work * a.R) / a.R;    // never past one wave
        dim3 grid((unsigned)(per_rank < 1 ? 1 : per_rank), (unsigned)a.R);
        kern<<<grid, kThreads, 0, st>>>(a);
        return cudaGetLastError();
    };
    switch (a.R) {
    case 8: return go(reinterpret_cast<const void*>(&k_ag_cast<8>), k_ag_cast<8>);
    case 4: return go(reinterpret_cast<const void*>(&k_ag_cast<4>), k_ag_cast<4>);
    case 2: return go(reinterpret_cast<const void*>(&k_ag_cast<2>), k_ag_cast<2>);
    default: return go(reinterpret_cast<const void*>(&k_ag_cast<0>), k_ag_cast<0>);
    }
}

// ---------------------------------------------------------- validation --

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

zero_status check_ptr(const void* p)
{
    if (!p) return ZERO_ERR_NULL;
    if (!aligned16(p)) return ZERO_ERR_ALIGN;
    return ZERO_OK;
}

zero_status check_hparams(const zero_adamw_hparams* hp, int64_t step)
{
    if (!hp) return ZERO_ERR_NULL;
    if (step < 1) return ZERO_ERR_INVALID_ARG;
    if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return ZERO_ERR_INVALID_ARG;
    if (!std::isfinite(hp->lr) || !std::isfinite(hp->weight_decay) || !std::isfinite(hp->eps) ||
        hp->eps < 0.0f)
        return ZERO_ERR_INVALID_ARG;
    return ZERO_OK;
}

struct Range {
    uintptr_t lo, hi;
    bool out;
};

// Outputs may not overlap anything; inputs may overlap inputs.
zero_status check_overlap(Range* r, int n)
{
    // insertion sort by start (n is at most a few hundred)
    for (int i = 1; i < n; ++i) {
        Range x = r[i];
        int j = i - 1;
        while (j >= 0 && r[j].lo > x.lo) { r[j + 1] = r[j]; --j; }
        r[j + 1] = x;
    }
    uintptr_t max_end_all = 0, max_end_out = 0;
    for (int i = 0; i < n; ++i) {
        if (r[i].hi <= r[i].lo) continue;
        if (r[i].out ? r[i].lo < max_end_all : r[i].lo < max_end_out) return ZERO_ERR_OVERLAP;
        if (r[i].hi > max_end_all) max_end_all = r[i].hi;
        if (r[i].out && r[i].hi > max_end_out) max_end_out = r[i].hi;
    }
    return ZERO_OK;
}

Range rng(const void* p, int64_t bytes, bool out)
{
    return Range{(uintptr_t)p, (uintptr_t)p + (uintptr_t)bytes, out};
}

zero_status check_plan(const zero_plan_t* plan)
{
    if (!plan) return ZERO_ERR_NULL;
    if (plan->R < 1 || plan->R > ZERO_MAX_R || plan->M < 1 ||
        (int64_t)plan->R * plan->M > ZERO_MAX_RM || plan->N < 0 || plan->S < 0 ||
        plan->S % 4 != 0 || plan->S * plan->R < plan->N)
        return ZERO_ERR_INVALID_ARG;
    return ZERO_OK;
}

zero_status check_grads(const zero_plan_t* plan, const uint16_t* const* grads, Range* rs, int& nr)
{
    if (!grads) return ZERO_ERR_NULL;
    const int RM = plan->R * plan->M;
    for (int q = 0; q < RM; ++q) {
        if (zero_status e = check_ptr(grads[q])) return e;
        rs[nr++] = rng(grads[q], 2 * plan->N, false);
    }
    return ZERO_OK;
}

zero_status check_replicas(const zero_plan_t* plan, uint16_t* const* P, Range* rs, int& nr)
{
    if (!P) return ZERO_ERR_NULL;
    for (int r = 0; r < plan->R; ++r) {
        if (zero_status e = check_ptr(P[r])) return e;
        rs[nr++] = rng(P[r], 2 * plan->N, true);
    }
    return ZERO_OK;
}

zero_status check_state(const zero_plan_t* plan, float* W, float* m, float* v, Range* rs, int& nr)
{
    for (const float* p : {W, m, v})
        if (zero_status e = check_ptr(p)) return e;
    for (float* p : {W, m, v}) rs[nr++] = rng(p, 4 * plan->padded, true);
    return ZERO_OK;
}

zero_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ZERO_OK : ZERO_ERR_CUDA; }

cudaError_t launch_fused_tma(const FusedArgs& a, bool expire_waits, bool check, cudaStream_t st);

void fill_grad_ptrs(GradPtrs& g, const zero_plan_t* plan, const uint16_t* const* grads)
{
    for (int q = 0; q < plan->R * plan->M; ++q) g.p[q] = grads[q];
}

void fill_replica_ptrs(ReplicaPtrs& P, const zero_plan_t* plan, uint16_t* const* rp)
{
    for (int r = 0; r < plan->R; ++r) P.p[r] = rp[r];
}

}  // namespace

// ======================================================== C entry points ==

extern "C" zero_status zero_step(const zero_plan_t* plan, const uint16_t* const* rank_grads,
                                 float* master, float* m, float* v,
                                 uint16_t* const* rank_params, const zero_adamw_hparams* hp,
                                 int64_t step, int32_t variant, void* scratch,
                                 int64_t scratch_bytes, int32_t flags, int32_t* dev_status,
                                 void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (zero_status e = check_hparams(hp, step)) return e;
    if (variant != ZERO_VARIANT_FUSED && variant != ZERO_VARIANT_STAGED &&
        variant != ZERO_VARIANT_FUSED_TMA)
        return ZERO_ERR_INVALID_ARG;
    if (variant == ZERO_VARIANT_FUSED_TMA && plan->R * plan->M > ZERO_TMA_MAX_RM)
        return ZERO_ERR_INVALID_ARG;
    const int32_t allowed = ZERO_FLAG_CHECK_FINITE |
                            (variant == ZERO_VARIANT_FUSED_TMA ? ZERO_FLAG_DEBUG_EXPIRE_WAITS : 0);
    if (flags & ~allowed) return ZERO_ERR_INVALID_ARG;
    if ((flags & (ZERO_FLAG_CHECK_FINITE | ZERO_FLAG_DEBUG_EXPIRE_WAITS)) && !dev_status)
        return ZERO_ERR_NULL;
    if (plan->N == 0) return ZERO_OK;

    Range rs[ZERO_MAX_RM + ZERO_MAX_R + 5];
    int nr = 0;
    if (zero_status e = check_grads(plan, rank_grads, rs, nr)) return e;
    if (zero_status e = check_replicas(plan, rank_params, rs, nr)) return e;
    if (zero_status e = check_state(plan, master, m, v, rs, nr)) return e;
    if (variant == ZERO_VARIANT_STAGED) {
        if (zero_status e = check_ptr(scratch)) return e;
        if (scratch_bytes < plan->scratch_bytes_staged) return ZERO_ERR_SIZE;
        rs[nr++] = rng(scratch, plan->scratch_bytes_staged, true);
    }
    if (dev_status) rs[nr++] = rng(dev_status, 4, true);
    if (zero_status e = check_overlap(rs, nr)) return e;

    const StepScalars s = step_scalars(*hp, step, plan->R, plan->M);
    const bool check = (flags & ZERO_FLAG_CHECK_FINITE) != 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (variant == ZERO_VARIANT_FUSED || variant == ZERO_VARIANT_FUSED_TMA) {
        FusedArgs a{};
        fill_grad_ptrs(a.g, plan, rank_grads);
        fill_replica_ptrs(a.P, plan, rank_params);
        a.W = master;
        a.m = m;
        a.v = v;
        a.n = plan->N;
        a.R = plan->R;
        a.M = plan->M;
        a.s = s;
        a.status = dev_status;
        if (variant == ZERO_VARIANT_FUSED_TMA)
            return cuda_status(launch_fused_tma(a, (flags & ZERO_FLAG_DEBUG_EXPIRE_WAITS) != 0,
                                                check, st));
        return cuda_status(check ? launch_fused<true>(a, st) : launch_fused<false>(a, st));
    }

    StagedArgs a{};
    fill_grad_ptrs(a.g, plan, rank_grads);
    fill_replica_ptrs(a.P, plan, rank_params);
    a.gs = static_cast<const float*>(scratch);
    a.gs_out = static_cast<float*>(scratch);
    a.W = master;
    a.m = m;
    a.v = v;
    a.n = plan->N;
    a.S = plan->S;
    a.R = plan->R;
    a.M = plan->M;
    a.s = s;
    a.status = dev_status;
    cudaError_t err = check ? launch_rs<true>(a, st) : launch_rs<false>(a, st);
    if (err == cudaSuccess) err = launch_adamw(a, st);
    if (err == cudaSuccess) err = launch_ag(a, st);
    return cuda_status(err);
}

extern "C" zero_status zero_rs_avg(const zero_plan_t* plan, const uint16_t* const* rank_grads,
                                   float* g_shards, int32_t flags, int32_t* dev_status,
                                   void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (flags & ~ZERO_FLAG_CHECK_FINITE) return ZERO_ERR_INVALID_ARG;
    if ((flags & ZERO_FLAG_CHECK_FINITE) && !dev_status) return ZERO_ERR_NULL;
    if (plan->N == 0) return ZERO_OK;
    Range rs[ZERO_MAX_RM + 2];
    int nr = 0;
    if (zero_status e = check_grads(plan, rank_grads, rs, nr)) return e;
    if (zero_status e = check_ptr(g_shards)) return e;
    rs[nr++] = rng(g_shards, 4 * plan->padded, true);
    if (dev_status) rs[nr++] = rng(dev_status, 4, true);
    if (zero_status e = check_overlap(rs, nr)) return e;
    StagedArgs a{};
    fill_grad_ptrs(a.g, plan, rank_grads);
    a.gs = g_shards;
    a.gs_out = g_shards;
    a.n = plan->N;
    a.S = plan->S;
    a.R = plan->R;
    a.M = plan->M;
    zero_adamw_hparams dummy{0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    a.s = step_scalars(dummy, 1, plan->R, plan->M);
    a.status = dev_status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool check = (flags & ZERO_FLAG_CHECK_FINITE) != 0;
    return cuda_status(check ? launch_rs<true>(a, st) : launch_rs<false>(a, st));
}

extern "C" zero_status zero_adamw_shard(const zero_plan_t* plan, const float* g_shards,
                                        float* master, float* m, float* v,
                                        const zero_adamw_hparams* hp, int64_t step, void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (zero_status e = check_hparams(hp, step)) return e;
    if (plan->N == 0) return ZERO_OK;
    Range rs[4];
    int nr = 0;
    if (zero_status e = check_ptr(g_shards)) return e;
    rs[nr++] = rng(g_shards, 4 * plan->padded, false);
    if (zero_status e = check_state(plan, master, m, v, rs, nr)) return e;
    if (zero_status e = check_overlap(rs, nr)) return e;
    StagedArgs a{};
    a.gs = g_shards;
    a.gs_out = nullptr;
    a.W = master;
    a.m = m;
    a.v = v;
    a.n = plan->N;
    a.S = plan->S;
    a.R = plan->R;
    a.M = plan->M;
    a.s = step_scalars(*hp, step, plan->R, plan->M);
    a.status = nullptr;
    return cuda_status(launch_adamw(a, static_cast<cudaStream_t>(stream)));
}

extern "C" zero_status zero_ag_cast(const zero_plan_t* plan, const float* master,
                                    uint16_t* const* rank_params, void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (plan->N == 0) return ZERO_OK;
    Range rs[ZERO_MAX_R + 1];
    int nr = 0;
    if (zero_status e = check_ptr(master)) return e;
    rs[nr++] = rng(master, 4 * plan->padded, false);
    if (zero_status e = check_replicas(plan, rank_params, rs, nr)) return e;
    if (zero_status e = check_overlap(rs, nr)) return e;
    StagedArgs a{};
    fill_replica_ptrs(a.P, plan, rank_params);
    a.W = const_cast<float*>(master);
    a.n = plan->N;
    a.S = plan->S;
    a.R = plan->R;
    a.M = plan->M;
    a.status = nullptr;
    return cuda_status(launch_ag(a, static_cast<cudaStream_t>(stream)));
}

// Device-side address of a host buffer the kernels may read or write over the
// host link: pinned (cudaHostAlloc / cudaHostRegister) memory maps to a
// device pointer; on systems where the GPU walks the host page tables any
// host pointer is usable as is.  Returns nullptr when the GPU cannot reach it.
static const void* device_view_of_host(const void* p, bool pageable_ok)
{
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return pageable_ok ? p : nullptr;
    }
    if (at.type == cudaMemoryTypeHost && at.devicePointer) return at.devicePointer;
    if (at.type == cudaMemoryTypeManaged) return p;
    if (at.type == cudaMemoryTypeUnregistered && pageable_ok) return p;
    return nullptr;
}

extern "C" zero_status zero_step_host(const zero_plan_t* plan, const uint16_t* const* host_grads,
                                      uint16_t* const* dev_grads, float* master, float* m,
                                      float* v, uint16_t* const* rank_params,
                                      uint16_t* host_params_out, const zero_adamw_hparams* hp,
                                      int64_t step, int32_t flags, int32_t* dev_status,
                                      void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (zero_status e = check_hparams(hp, step)) return e;
    if (!host_grads || !host_params_out) return ZERO_ERR_NULL;
    if (flags & ~ZERO_FLAG_CHECK_FINITE) return ZERO_ERR_INVALID_ARG;
    if ((flags & ZERO_FLAG_CHECK_FINITE) && !dev_status) return ZERO_ERR_NULL;
    if (plan->N == 0) return ZERO_OK;
    const int RM = plan->R * plan->M;
    for (int q = 0; q < RM; ++q)
        if (!host_grads[q]) return ZERO_ERR_NULL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t gbytes = (size_t)plan->N * 2;

    if (dev_grads) {
        // copy-engine mode: validate the device side before any copy is enqueued
        Range rs[ZERO_MAX_RM + ZERO_MAX_R + 5];
        int nr = 0;
        const uint16_t* const* dg = dev_grads;
        if (zero_status e = check_grads(plan, dg, rs, nr)) return e;
        if (zero_status e = check_replicas(plan, rank_params, rs, nr)) return e;
        if (zero_status e = check_state(plan, master, m, v, rs, nr)) return e;
        if (dev_status) rs[nr++] = rng(dev_status, 4, true);
        if (zero_status e = check_overlap(rs, nr)) return e;
        // the copies write the gradient buffers: they must not overlap each other
        Range gr[ZERO_MAX_RM];
        for (int q = 0; q < RM; ++q) gr[q] = rng(dev_grads[q], 2 * plan->N, true);
        if (zero_status e = check_overlap(gr, RM)) return e;
        for (int q = 0; q < RM; ++q)
            if (cudaMemcpyAsync(dev_grads[q], host_grads[q], gbytes, cudaMemcpyHostToDevice,
                                st) != cudaSuccess)
                return ZERO_ERR_CUDA;
        zero_status e = zero_step(plan, dg, master, m, v, rank_params, hp, step,
                                  ZERO_VARIANT_FUSED, nullptr, 0, flags, dev_status, stream);
        if (e != ZERO_OK) return e;
        if (cudaMemcpyAsync(host_params_out, rank_params[0], gbytes, cudaMemcpyDeviceToHost,
                            st) != cudaSuccess)
            return ZERO_ERR_CUDA;
        return ZERO_OK;
    }

    // zero-copy mode: the fused kernel reads the gradients from host memory and
    // writes replica 0's bits to host_params_out as well as to the R device
    // replicas, so the host-link transfers overlap the HBM work
    int dev = 0, pageable = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZERO_ERR_CUDA;
    cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev);
    FusedArgs a{};
    Range rs[ZERO_MAX_RM + ZERO_MAX_R + 6];
    int nr = 0;
    for (int q = 0; q < RM; ++q) {
        const void* dp = device_view_of_host(host_grads[q], pageable != 0);
        if (!dp) return ZERO_ERR_INVALID_ARG;
        if (!aligned16(dp)) return ZERO_ERR_ALIGN;
        a.g.p[q] = static_cast<const uint16_t*>(dp);
        rs[nr++] = rng(dp, 2 * plan->N, false);
    }
    void* out = const_cast<void*>(device_view_of_host(host_params_out, pageable != 0));
    if (!out) return ZERO_ERR_INVALID_ARG;
    if (!aligned16(out)) return ZERO_ERR_ALIGN;
    rs[nr++] = rng(out, 2 * plan->N, true);
    if (zero_status e = check_replicas(plan, rank_params, rs, nr)) return e;
    if (zero_status e = check_state(plan, master, m, v, rs, nr)) return e;
    if (dev_status) rs[nr++] = rng(dev_status, 4, true);
    if (zero_status e = check_overlap(rs, nr)) return e;
    fill_replica_ptrs(a.P, plan, rank_params);
    a.extra_rep = static_cast<uint16_t*>(out);
    a.W = master;
    a.m = m;
    a.v = v;
    a.n = plan->N;
    a.R = plan->R;
    a.M = plan->M;
    a.s = step_scalars(*hp, step, plan->R, plan->M);
    a.status = dev_status;
    const bool check = (flags & ZERO_FLAG_CHECK_FINITE) != 0;
    return cuda_status(check ? launch_fused<true>(a, st) : launch_fused<false>(a, st));
}

// =========================================== step with global-norm clipping ==
// zero_step_clipped: the averaged gradient of every element is stashed in
// fp32 scratch while its square feeds a fixed pairwise tree (fp32, leaves
// g*g, zero padding to a power of two); the tree is finished level by level,
// one thread turns the squared norm into the clip coefficient (and the
// skip decision for a non-finite norm), and a last pass applies it with the
// AdamW update and the R-way bf16 all-gather.
//
// Tree decomposition: in the streaming pass each warp reduces 256
// consecutive leaves (32 lanes x 8 leaves: a 3-level tree in registers, then
// 5 levels of shuffles) - exactly an aligned subtree of the global tree - and
// writes one partial, with no block-wide barrier; each further level is a
// block reducing 2048 partials (8 leaves per thread, the warp levels, then 3
// levels across the 8 warps), again an aligned subtree.  Adding a zero
// (padding) changes no value, so the result equals the tree over the leaves
// padded to the next power of two for any N and any grid.
namespace {

constexpr int kTreeLeaves = 2048;                 // leaves per tree block (256 x 8)
constexpr int kWarpLeaves = 256;                  // leaves per warp in the streaming pass

struct ClipCtl {
    double sumsq;          // squared norm (the fp32 tree value, widened)
    float coef;            // multiplier when clip != 0
    int32_t clip;          // 1: multiply the averaged gradients by coef
    int32_t skip;          // 1: non-finite norm and skipping requested
    int32_t pad[9];
};

struct ClipLayout {
    int64_t g_off, ctl_off, total;
    int levels;
    int64_t lvl_off[8], lvl_len[8];
};

int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

ClipLayout clip_layout(const zero_plan_t* plan)
{
    ClipLayout L{};
    L.g_off = 0;
    int64_t off = round256(4 * plan->padded);
    int64_t len = (plan->N + kWarpLeaves - 1) / kWarpLeaves;
    if (len < 1) len = 1;
    L.levels = 0;
    while (true) {
        L.lvl_off[L.levels] = off;
        L.lvl_len[L.levels] = len;
        off += round256(4 * len);
        ++L.levels;
        if (len == 1 || L.levels == 8) break;
        len = (len + kTreeLeaves - 1) / kTreeLeaves;
    }
    L.ctl_off = off;
    L.total = off + round256((int64_t)sizeof(ClipCtl));
    return L;
}

// sum of a thread's 8 leaves, then the warp and block levels; returns the
// block's value in thread 0
__device__ __forceinline__ float tree8(const float (&x)[8])
{
    return __fadd_rn(__fadd_rn(__fadd_rn(x[0], x[1]), __fadd_rn(x[2], x[3])),
                     __fadd_rn(__fadd_rn(x[4], x[5]), __fadd_rn(x[6], x[7])));
}

__device__ __forceinline__ float warp_tree(float v)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_down_sync(0xFFFFFFFFu, v, off);
        v = __fadd_rn(v, o);           // meaningful in lanes that are multiples of 2*off
    }
    return v;                          // lane 0 holds the warp's subtree
}

__device__ __forceinline__ float block_tree(float v)
{
    __shared__ float warp_sum[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_down_sync(0xFFFFFFFFu, v, off);
        v = __fadd_rn(v, o);           // meaningful in lanes that are multiples of 2*off
    }
    if (lane == 0) warp_sum[warp] = v;
    __syncthreads();
    float r = 0.0f;
    if (threadIdx.x == 0) {
        const float* w = warp_sum;
        r = __fadd_rn(__fadd_rn(__fadd_rn(w[0], w[1]), __fadd_rn(w[2], w[3])),
                      __fadd_rn(__fadd_rn(w[4], w[5]), __fadd_rn(w[6], w[7])));
    }
    __syncthreads();                   // warp_sum is reused by the next tile
    return r;
}

struct ClipArgs {
    GradPtrs g;
    ReplicaPtrs P;
    float* gs;             // averaged gradients (padded floats; [0, N) used)
    float* lvl0;           // first tree level: one partial per 256 elements (per warp)
    float* W;
    float* m;
    float* v;
    ClipCtl* ctl;
    int64_t n;
    int32_t R, M;
    StepScalars s;
};

// pass 1: averaged gradient of 8 consecutive elements per thread, stashed,
// and the tile's pairwise partial of their squares
template <int RC, int MC>
__global__ void __launch_bounds__(kThreads) k_rs_norm(const __grid_constant__ ClipArgs a)
{
    const int R = RC > 0 ? RC : a.R;
    const int M = MC > 0 ? MC : a.M;
    const int64_t n = a.n;
    const int64_t tiles = (n + kTreeLeaves - 1) / kTreeLeaves;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t e = tile * kTreeLeaves + (int64_t)threadIdx.x * 8;
        float g[8];
        if (e + 8 <= n) {
            float lo[4], hi[4];
            grad_sum4<RC, MC>(a.g, R, M, e, lo);
            grad_sum4<RC, MC>(a.g, R, M, e + 4, hi);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                g[k] = scale_grad(a.s, lo[k]);
                g[4 + k] = scale_grad(a.s, hi[k]);
            }
            st_stream(a.gs + e, make_float4(g[0], g[1], g[2], g[3]));
            st_stream(a.gs + e + 4, make_float4(g[4], g[5], g[6], g[7]));
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                g[k] = 0.0f;
                if (e + k < n) {
                    g[k] = scale_grad(a.s, grad_sum1(a.g, R, M, e + k));
                    a.gs[e + k] = g[k];
                }
            }
        }
        float sq[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sq[k] = __fmul_rn(g[k], g[k]);   // padding leaves are +0
        const float part = warp_tree(tree8(sq));
        const int64_t wpart = tile * (kTreeLeaves / kWarpLeaves) + (threadIdx.x >> 5);
        if ((threadIdx.x & 31) == 0 && wpart * kWarpLeaves < n) a.lvl0[wpart] = part;
    }
}

// one level of the tree: out[b] = pairwise sum of in[2048 b .. 2048 b + 2047]
__global__ void __launch_bounds__(kThreads) k_tree(const float* __restrict__ in, int64_t n_in,
                                                   float* __restrict__ out)
{
    const int64_t blocks = (n_in + kTreeLeaves - 1) / kTreeLeaves;
    for (int64_t b = blockIdx.x; b < blocks; b += gridDim.x) {
        const int64_t e = b * kTreeLeaves + (int64_t)threadIdx.x * 8;
        float x[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = e + k < n_in ? in[e + k] : 0.0f;
        const float part = block_tree(tree8(x));
        if (threadIdx.x == 0) out[b] = part;
    }
}

__global__ void k_clip_coef(const float* __restrict__ root, ClipCtl* ctl, float max_norm,
                            int32_t skip_nonfinite, int32_t* status, double* sumsq_out)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const float ss = *root;
    const double norm = sqrt((double)ss);
    const double coef = (double)max_norm / (norm + 1e-6);
    ClipCtl c{};
    c.sumsq = (double)ss;
    c.clip = coef < 1.0 ? 1 : 0;
    c.coef = c.clip ? (float)coef : 1.0f;
    const bool finite = isfinite(ss);
    c.skip = (!finite && skip_nonfinite) ? 1 : 0;
    *ctl = c;
    if (status) {
        if (!finite) atomicOr(status, ZERO_DEV_NONFINITE);
        if (c.skip) atomicOr(status, ZERO_DEV_SKIPPED);
    }
    if (sumsq_out) *sumsq_out = c.sumsq;
}

// pass 2: g' = g * coef (when clipping), AdamW, bf16 all-gather; tiles of
// 256 threads x 4 elements x 2 units with every load of a tile issued first,
// as in k_fused
template <int RC>
__global__ void __launch_bounds__(kThreads) k_adamw_ag(const __grid_constant__ ClipArgs a)
{
    const ClipCtl c = *a.ctl;
    if (c.skip) return;
    const int R = RC > 0 ? RC : a.R;
    constexpr int U = 4;
    constexpr int T = kUnit * U;
    const int64_t n = a.n;
    const int64_t full_tiles = n / T;
    for (int64_t tile = blockIdx.x; tile < full_tiles; tile += gridDim.x) {
        const int64_t e0 = tile * T + (int64_t)threadIdx.x * kVec;
        float4 g[U], w[U], m[U], v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t e = e0 + (int64_t)u * kUnit;
            g[u] = ld_stream(a.gs + e);
            w[u] = ld_stream(a.W + e);
            m[u] = ld_stream(a.m + e);
            v[u] = ld_stream(a.v + e);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t e = e0 + (int64_t)u * kUnit;
            float* gp = &g[u].x;
            float* wp = &w[u].x;
            float* mp = &m[u].x;
            float* vp = &v[u].x;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float gk = c.clip ? __fmul_rn(gp[k], c.coef) : gp[k];
                adamw(a.s, gk, wp[k], mp[k], vp[k]);
            }
            st_stream(a.W + e, w[u]);
            st_stream(a.m + e, m[u]);
            st_stream(a.v + e, v[u]);
            const uint2 p = make_uint2(pack_bf16x2(w[u].x, w[u].y), pack_bf16x2(w[u].z, w[u].w));
            if constexpr (RC > 0) {
#pragma unroll
                for (int r = 0; r < RC; ++r) st_stream(a.P.p[r] + e, p);
            } else {
                for (int r = 0; r < R; ++r) st_stream(a.P.p[r] + e, p);
            }
        }
    }
    const int64_t tail0 = full_tiles * T;
    if (tail0 < n && blockIdx.x == (unsigned)(full_tiles % gridDim.x)) {
        for (int64_t i = tail0 + threadIdx.x; i < n; i += kThreads) {
            float g = a.gs[i];
            if (c.clip) g = __fmul_rn(g, c.coef);
            float w = a.W[i], m = a.m[i], v = a.v[i];
            adamw(a.s, g, w, m, v);
            a.W[i] = w;
            a.m[i] = m;
            a.v[i] = v;
            const uint16_t p = to_bf16(w);
            for (int r = 0; r < R; ++r) a.P.p[r][i] = p;
        }
    }
}

template <int RC, int MC>
cudaError_t launch_rs_norm_t(const ClipArgs& a, cudaStream_t st)
{
    const void* k = reinterpret_cast<const void*>(&k_rs_norm<RC, MC>);
    const int64_t tiles = (a.n + kTreeLeaves - 1) / kTreeLeaves;
    k_rs_norm<RC, MC><<<grid_for(k, tiles), kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rs_norm(const ClipArgs& a, cudaStream_t st)
{
    const int R = a.R, M = a.M;
#define ZERO_CASE(r_, m_) \
    if (R == r_ && M == m_) return launch_rs_norm_t<r_, m_>(a, st);
    ZERO_CASE(8, 1) ZERO_CASE(4, 1) ZERO_CASE(2, 1) ZERO_CASE(1, 1) ZERO_CASE(4, 2) ZERO_CASE(7, 4)
#undef ZERO_CASE
    return launch_rs_norm_t<0, 0>(a, st);
}

cudaError_t launch_adamw_ag(const ClipArgs& a, cudaStream_t st)
{
    const int64_t work = (a.n + 4 * kUnit - 1) / (4 * kUnit);     // tiles of 4 units
    auto go = [&](const void* k, auto kern) {
        kern<<<grid_for(k, work < 1 ? 1 : work), kThreads, 0, st>>>(a);
        return cudaGetLastError();
    };
    switch (a.R) {
    case 8: return go(reinterpret_cast<const void*>(&k_adamw_ag<8>), k_adamw_ag<8>);
    case 4: return go(reinterpret_cast<const void*>(&k_adamw_ag<4>), k_adamw_ag<4>);
    case 2: return go(reinterpret_cast<const void*>(&k_adamw_ag<2>), k_adamw_ag<2>);
    default: return go(reinterpret_cast<const void*>(&k_adamw_ag<0>), k_adamw_ag<0>);
    }
}

}  // namespace

extern "C" int64_t zero_clip_scratch_bytes(const zero_plan_t* plan)
{
    if (check_plan(plan) != ZERO_OK) return -1;
    return clip_layout(plan).total;
}

extern "C" zero_status zero_step_clipped(const zero_plan_t* plan,
                                         const uint16_t* const* rank_grads, float* master,
                                         float* m, float* v, uint16_t* const* rank_params,
                                         const zero_adamw_hparams* hp, int64_t step,
                                         float max_norm, void* scratch, int64_t scratch_bytes,
                                         int32_t flags, int32_t* dev_status, double* dev_sumsq,
                                         void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (zero_status e = check_hparams(hp, step)) return e;
    if (!(max_norm > 0.0f) || !std::isfinite(max_norm)) return ZERO_ERR_INVALID_ARG;
    if (flags & ~(ZERO_FLAG_CHECK_FINITE | ZERO_FLAG_SKIP_NONFINITE)) return ZERO_ERR_INVALID_ARG;
    if ((flags & ZERO_FLAG_CHECK_FINITE) && !dev_status) return ZERO_ERR_NULL;
    if (plan->N == 0) return ZERO_OK;
    const ClipLayout L = clip_layout(plan);
    Range rs[ZERO_MAX_RM + ZERO_MAX_R + 6];
    int nr = 0;
    if (zero_status e = check_grads(plan, rank_grads, rs, nr)) return e;
    if (zero_status e = check_replicas(plan, rank_params, rs, nr)) return e;
    if (zero_status e = check_state(plan, master, m, v, rs, nr)) return e;
    if (zero_status e = check_ptr(scratch)) return e;
    if (scratch_bytes < L.total) return ZERO_ERR_SIZE;
    rs[nr++] = rng(scratch, L.total, true);
    if (dev_status) rs[nr++] = rng(dev_status, 4, true);
    if (dev_sumsq) {
        if ((uintptr_t)dev_sumsq & 7u) return ZERO_ERR_ALIGN;
        rs[nr++] = rng(dev_sumsq, 8, true);
    }
    if (zero_status e = check_overlap(rs, nr)) return e;

    char* base = static_cast<char*>(scratch);
    ClipArgs a{};
    fill_grad_ptrs(a.g, plan, rank_grads);
    fill_replica_ptrs(a.P, plan, rank_params);
    a.gs = reinterpret_cast<float*>(base + L.g_off);
    a.lvl0 = reinterpret_cast<float*>(base + L.lvl_off[0]);
    a.W = master;
    a.m = m;
    a.v = v;
    a.ctl = reinterpret_cast<ClipCtl*>(base + L.ctl_off);
    a.n = plan->N;
    a.R = plan->R;
    a.M = plan->M;
    a.s = step_scalars(*hp, step, plan->R, plan->M);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    cudaError_t err = launch_rs_norm(a, st);
    for (int l = 1; l < L.levels && err == cudaSuccess; ++l) {
        const float* in = reinterpret_cast<const float*>(base + L.lvl_off[l - 1]);
        float* out = reinterpret_cast<float*>(base + L.lvl_off[l]);
        const void* k = reinterpret_cast<const void*>(&k_tree);
        k_tree<<<grid_for(k, L.lvl_len[l]), kThreads, 0, st>>>(in, L.lvl_len[l - 1], out);
        err = cudaGetLastError();
    }
    if (err == cudaSuccess) {
        const float* root = reinterpret_cast<const float*>(base + L.lvl_off[L.levels - 1]);
        k_clip_coef<<<1, 32, 0, st>>>(root, a.ctl, max_norm,
                                      (flags & ZERO_FLAG_SKIP_NONFINITE) ? 1 : 0, dev_status,
                                      dev_sumsq);
        err = cudaGetLastError();
    }
    if (err == cudaSuccess) err = launch_adamw_ag(a, st);
    return cuda_status(err);
}

// ================================================ compressed reduce-scatter ==
// zero_step_compressed: every rank compresses its locally accumulated
// gradient (plus its error-feedback residual) over aligned blocks of 128
// elements of the flat vector before the emulated reduce-scatter, and the
// owner sums the decompressed values in rank order (the header gives the
// three codecs).  One warp owns one block: lane l holds elements 4l..4l+3,
// so the block max is a warp max of |x| and the block's |x| sum is a pairwise
// tree - the 4 leaves of a lane, then 5 shuffle levels - in element order.
// The compressed message is never written to memory: on one GPU the wire
// is a register, and only its decompressed value matters to the owner.
namespace {

constexpr int kCompBlock = 128;

struct CompArgs {
    GradPtrs g;
    ReplicaPtrs P;
    float* E[ZERO_MAX_R];  // error-feedback residuals (N floats per rank) or unused
    float* W;
    float* m;
    float* v;
    int64_t n;
    int32_t R, M;
    StepScalars s;
};

// x / b rounded to nearest even from r = RN(1/b): a first FMA correction
// makes the product x*r a faithful quotient, and a second one with the
// correctly rounded reciprocal gives the correctly rounded quotient
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990: the residual of a
// faithful quotient is exact under FMA, and one more correction rounds it
// correctly).  The argument needs the residuals to stay normal: it is used
// for 2^-100 <= b <= 2^100 and |x / b| <= 128, where any quotient below 0.5 in
// magnitude may come out a few ulps off but still rounds to the same
// integer (a signed zero), which is all the int8 codec takes from it.
__device__ __forceinline__ float quot_by_recip(float x, float b, float r)
{
    const float y0 = __fmul_rn(x, r);
    const float y1 = __fmaf_rn(__fmaf_rn(-y0, b, x), r, y0);
    return __fmaf_rn(__fmaf_rn(-y1, b, x), r, y1);
}

// Two ways to the same bits, chosen per kernel by measurement (the codec's
// arithmetic cost is hidden or not depending on what else the kernel moves):
//   RECIP  int8 quotients through quot_by_recip instead of one IEEE division
//          each (taken without error feedback, where the kernel is bound by
//          instruction issue);
//   POW2   a full sign block's |x| sum scaled by the exact 2^-7 instead of
//          divided by 128 (taken with error feedback).
// Without error feedback the full blocks of the compile-time (R, M) cases go
// through int8_transposed and sign_transposed below, which give these bits
// too with fewer instructions.
template <int KIND, bool RECIP = false, bool POW2 = false>
__device__ __forceinline__ void codec(float (&x)[4], const bool (&valid)[4], int64_t block_count,
                                      float (&d)[4])
{
    if constexpr (KIND == ZERO_COMP_FP16) {
#pragma unroll
        for (int k = 0; k < 4; ++k) d[k] = __half2float(__float2half_rn(x[k]));
    } else if constexpr (KIND == ZERO_COMP_INT8) {
        uint32_t amax = 0;                        // |x| bits order like the values
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (valid[k]) amax = max(amax, __float_as_uint(x[k]) & 0x7FFFFFFFu);
        amax = __reduce_max_sync(0xFFFFFFFFu, amax);
        const float sc = __fdiv_rn(__uint_as_float(amax), 127.0f);
        if constexpr (RECIP) {
            // x / sc correctly rounded: the block shares sc, so while sc is
            // a normal number well inside the exponent range (warp-uniform
            // test) every quotient comes from one reciprocal and FMA
            // corrections (quot_by_recip); otherwise the IEEE division
            const bool fast = sc >= 0x1p-100f && sc <= 0x1p100f;
            float t[4];
            if (fast) {
                const float rc = __frcp_rn(sc);
#pragma unroll
                for (int k = 0; k < 4; ++k) t[k] = quot_by_recip(x[k], sc, rc);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) t[k] = __fdiv_rn(x[k], sc);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (sc == 0.0f) {
                    d[k] = 0.0f;
                } else {
                    float q = rintf(t[k]);
                    q = fminf(fmaxf(q, -127.0f), 127.0f);
                    d[k] = __fmul_rn(q, sc);
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (sc == 0.0f) {
                    d[k] = 0.0f;
                } else {
                    float q = rintf(__fdiv_rn(x[k], sc));
                    q = fminf(fmaxf(q, -127.0f), 127.0f);
                    d[k] = __fmul_rn(q, sc);
                }
            }
        }
    } else {                                      // ZERO_COMP_SIGN
        float a[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) a[k] = valid[k] ? fabsf(x[k]) : 0.0f;
        float t = __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3]));
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) t = __fadd_rn(t, __shfl_down_sync(0xFFFFFFFFu, t, off));
        t = __shfl_sync(0xFFFFFFFFu, t, 0);
        // a full block divides by 128: scaling by the exact 2^-7 rounds the
        // same quotient
        const float sc = POW2 && block_count == kCompBlock ? __fmul_rn(t, 1.0f / kCompBlock)
                                                           : __fdiv_rn(t, (float)block_count);
#pragma unroll
        for (int k = 0; k < 4; ++k) d[k] = x[k] < 0.0f ? -sc : sc;
    }
}

// int8 codec of every rank's full block without error feedback, with the
// block scales computed across lanes: lane l derives the scale and its
// reciprocal of rank l % RC once, instead of every lane for every rank, and
// rank r's pair is then broadcast from lane r.  Inside the fast range of
// quot_by_recip the clamp to [-127, 127] and the zero-scale test are no-ops:
// |x| <= amax and sc = RN(amax / 127) >= (amax / 127)(1 - 2^-24) give
// |x / sc| < 127 (1 + 2^-23) < 127.5, so the rounded quotient is at most 127
// in magnitude.  Outside that range the codec's IEEE path runs unchanged.
template <int RC, int MC>
__device__ __forceinline__ void int8_transposed(const uint2 (&gx)[RC * MC], int lane,
                                                float (&acc)[4])
{
    float x[RC][4];
    uint32_t amax[RC];
#pragma unroll
    for (int r = 0; r < RC; ++r) {
#pragma unroll
        for (int j = 0; j < MC; ++j) {
            const uint2 u = gx[r * MC + j];
            const float y[4] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y)};
#pragma unroll
            for (int k = 0; k < 4; ++k) x[r][k] = j == 0 ? y[k] : __fadd_rn(x[r][k], y[k]);
        }
        uint32_t mx = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) mx = max(mx, __float_as_uint(x[r][k]) & 0x7FFFFFFFu);
        amax[r] = __reduce_max_sync(0xFFFFFFFFu, mx);
    }
    const int mine = lane % RC;
    uint32_t am = amax[0];
#pragma unroll
    for (int r = 1; r < RC; ++r) am = mine == r ? amax[r] : am;
    const float sc_l = __fdiv_rn(__uint_as_float(am), 127.0f);
    const float rc_l = __frcp_rn(sc_l);
#pragma unroll
    for (int r = 0; r < RC; ++r) {
        const float sc = __shfl_sync(0xFFFFFFFFu, sc_l, r);
        const float rc = __shfl_sync(0xFFFFFFFFu, rc_l, r);
        float d[4];
        if (sc >= 0x1p-100f && sc <= 0x1p100f) {
#pragma unroll
            for (int k = 0; k < 4; ++k) d[k] = __fmul_rn(rintf(quot_by_recip(x[r][k], sc, rc)), sc);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (sc == 0.0f) {
                    d[k] = 0.0f;
                } else {
                    float q = rintf(__fdiv_rn(x[r][k], sc));
                    q = fminf(fmaxf(q, -127.0f), 127.0f);
                    d[k] = __fmul_rn(q, sc);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = r == 0 ? d[k] : __fadd_rn(acc[k], d[k]);
    }
}

// Magnitudes of the sign codec for RC full blocks at once (x[r] holds a
// lane's 4 elements of rank r's block): sc[r] = (pairwise sum of |x| over
// the block) / 128, the RC sums reduced together.  At each of the first
// log2(RC) levels of the lane tree a lane keeps half of its remaining ranks
// and receives its partner's values of them (one shuffle per kept rank
// instead of one per rank), so lane l ends with one rank; the last levels and
// the scaling run once per lane, and each rank's magnitude is then broadcast
// from a lane that holds it.  The additions pair the same lanes as the
// shuffle-down tree of the codec (lanes 2i and 2i+1, then pairs of pairs,
// ...), and a + b == b + a in IEEE arithmetic, so every sum has the same bits;
// scaling by the exact 2^-7 rounds the same quotient as dividing by 128.
template <int RC>
__device__ __forceinline__ void sign_scales_joint(const float (&x)[RC][4], int lane,
                                                  float (&sc)[RC])
{
    static_assert((RC & (RC - 1)) == 0 && RC <= 32, "RC must be a power of two");
    constexpr int P = RC == 1 ? 0 : RC == 2 ? 1 : RC == 4 ? 2 : RC == 8 ? 3 : RC == 16 ? 4 : 5;
    float cur[RC];
#pragma unroll
    for (int r = 0; r < RC; ++r)
        cur[r] = __fadd_rn(__fadd_rn(fabsf(x[r][0]), fabsf(x[r][1])),
                           __fadd_rn(fabsf(x[r][2]), fabsf(x[r][3])));
#pragma unroll
    for (int lvl = 0; lvl < P; ++lvl) {
        const int half = RC >> (lvl + 1);
        const bool up = (lane >> lvl) & 1;
#pragma unroll
        for (int k = 0; k < half; ++k) {
            const float send = up ? cur[k] : cur[k + half];
            const float keep = up ? cur[k + half] : cur[k];
            cur[k] = __fadd_rn(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 1 << lvl));
        }
    }
#pragma unroll
    for (int lvl = P; lvl < 5; ++lvl)
        cur[0] = __fadd_rn(cur[0], __shfl_xor_sync(0xFFFFFFFFu, cur[0], 1 << lvl));
    const float sc_l = __fmul_rn(cur[0], 1.0f / kCompBlock);
#pragma unroll
    for (int r = 0; r < RC; ++r) {
        int src = 0;                          // a lane whose kept rank is r
#pragma unroll
        for (int lvl = 0; lvl < P; ++lvl) src |= ((r >> (P - 1 - lvl)) & 1) << lvl;
        sc[r] = __shfl_sync(0xFFFFFFFFu, sc_l, src);
    }
}

// sign codec of every rank's full block without error feedback, through
// sign_scales_joint, and the decoded values summed in rank order
template <int RC, int MC>
__device__ __forceinline__ void sign_transposed(const uint2 (&gx)[RC * MC], int lane,
                                                float (&acc)[4])
{
    float x[RC][4];
#pragma unroll
    for (int r = 0; r < RC; ++r) {
#pragma unroll
        for (int j = 0; j < MC; ++j) {
            const uint2 u = gx[r * MC + j];
            const float y[4] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y)};
#pragma unroll
            for (int k = 0; k < 4; ++k) x[r][k] = j == 0 ? y[k] : __fadd_rn(x[r][k], y[k]);
        }
    }
    float sc[RC];
    sign_scales_joint<RC>(x, lane, sc);
#pragma unroll
    for (int r = 0; r < RC; ++r) {
        float d[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) d[k] = x[r][k] < 0.0f ? -sc[r] : sc[r];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = r == 0 ? d[k] : __fadd_rn(acc[k], d[k]);
    }
}

template <int KIND, bool EF>
__device__ __forceinline__ void comp_ranks_generic(const CompArgs& a, int R, int M, int64_t e,
                                                   bool full, const bool (&valid)[4],
                                                   int64_t block_count, float (&acc)[4])
{
    for (int r = 0; r < R; ++r) {
        float x[4];
        // rank r's local accumulation of its micro-batches
        for (int j = 0; j < M; ++j) {
            float y[4];
            if (full) {
                const uint2 u = ld_stream(a.g.p[r * M + j] + e);
                y[0] = bf16_lo(u.x); y[1] = bf16_hi(u.x); y[2] = bf16_lo(u.y); y[3] = bf16_hi(u.y);
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) y[k] = valid[k] ? bf16_bits(a.g.p[r * M + j][e + k]) : 0.0f;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] = j == 0 ? y[k] : __fadd_rn(x[k], y[k]);
        }
        float res[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if constexpr (EF) {
            if (full) {
                const float4 q = ld_stream(a.E[r] + e);
                res[0] = q.x; res[1] = q.y; res[2] = q.z; res[3] = q.w;
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) res[k] = valid[k] ? a.E[r][e + k] : 0.0f;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] = __fadd_rn(x[k], res[k]);
        }
        float d[4];
        codec<KIND, !EF, EF>(x, valid, block_count, d);
        if constexpr (EF) {
            float o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) o[k] = __fsub_rn(x[k], d[k]);
            if (full) {
                st_stream(a.E[r] + e, make_float4(o[0], o[1], o[2], o[3]));
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) if (valid[k]) a.E[r][e + k] = o[k];
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = r == 0 ? d[k] : __fadd_rn(acc[k], d[k]);
    }
}

template <int RC, int MC, int KIND, bool EF>
__global__ void __launch_bounds__(kThreads) k_comp(const __grid_constant__ CompArgs a)
{
    const int R = RC > 0 ? RC : a.R;
    const int M = MC > 0 ? MC : a.M;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
    const int64_t n = a.n;
    const int64_t nblk = (n + kCompBlock - 1) / kCompBlock;
    for (int64_t b = warp; b < nblk; b += nwarps) {       // warp-uniform loop
        const int64_t e = b * kCompBlock + 4 * lane;
        const bool full = b * kCompBlock + kCompBlock <= n;
        const int64_t block_count = full ? kCompBlock : n - b * kCompBlock;
        bool valid[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) valid[k] = e + k < n;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float4 w4, m4, v4;                        // the owner's state of a full block
        bool have_state = false;
        // every rank's loads first, then the codecs and their warp reductions,
        // so the loads are all in flight before the first sync.  Whether the
        // owner's state joins them was measured per codec: it does for int8
        // without error feedback (0.86 -> 0.96 of peak), and slows the others.
        // fp16 without error feedback has no sync and runs faster in the
        // rank-by-rank form (fewer registers, more blocks per SM).
        if constexpr (RC > 0 && MC > 0 && (KIND != ZERO_COMP_FP16 || EF)) {
            if (full) {
                uint2 gx[RC * MC];
                float4 ex[EF ? RC : 1];
#pragma unroll
                for (int q = 0; q < RC * MC; ++q) gx[q] = ld_stream(a.g.p[q] + e);
                if constexpr (EF) {
#pragma unroll
                    for (int r = 0; r < RC; ++r) ex[r] = ld_stream(a.E[r] + e);
                }
                if constexpr (KIND == ZERO_COMP_INT8 && !EF) {
                    w4 = ld_stream(a.W + e);
                    m4 = ld_stream(a.m + e);
                    v4 = ld_stream(a.v + e);
                    have_state = true;
                    int8_transposed<RC, MC>(gx, lane, acc);
                } else if constexpr (KIND == ZERO_COMP_SIGN && !EF && (RC & (RC - 1)) == 0) {
                    sign_transposed<RC, MC>(gx, lane, acc);
                } else {
#pragma unroll
                    for (int r = 0; r < RC; ++r) {
                        float x[4];
#pragma unroll
                        for (int j = 0; j < MC; ++j) {
                            const uint2 u = gx[r * MC + j];
                            const float y[4] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y),
                                                bf16_hi(u.y)};
#pragma unroll
                            for (int k = 0; k < 4; ++k) x[k] = j == 0 ? y[k] : __fadd_rn(x[k], y[k]);
                        }
                        if constexpr (EF) {
                            x[0] = __fadd_rn(x[0], ex[r].x);
                            x[1] = __fadd_rn(x[1], ex[r].y);
                            x[2] = __fadd_rn(x[2], ex[r].z);
                            x[3] = __fadd_rn(x[3], ex[r].w);
                        }
                        float d[4];
                        codec<KIND, !EF, EF>(x, valid, block_count, d);
                        if constexpr (EF)
                            st_stream(a.E[r] + e,
                                      make_float4(__fsub_rn(x[0], d[0]), __fsub_rn(x[1], d[1]),
                                                  __fsub_rn(x[2], d[2]), __fsub_rn(x[3], d[3])));
#pragma unroll
                        for (int k = 0; k < 4; ++k) acc[k] = r == 0 ? d[k] : __fadd_rn(acc[k], d[k]);
                    }
                }
            } else {
                comp_ranks_generic<KIND, EF>(a, R, M, e, full, valid, block_count, acc);
            }
        } else {
            comp_ranks_generic<KIND, EF>(a, R, M, e, full, valid, block_count, acc);
        }
        // the owner: average, AdamW, all-gather
        if (full) {
            if (!have_state) {
                w4 = ld_stream(a.W + e);
                m4 = ld_stream(a.m + e);
                v4 = ld_stream(a.v + e);
            }
            float4 w = w4, m = m4, v = v4;
            float* wp = &w.x;
            float* mp = &m.x;
            float* vp = &v.x;
#pragma unroll
            for (int k = 0; k < 4; ++k) adamw(a.s, scale_grad(a.s, acc[k]), wp[k], mp[k], vp[k]);
            st_stream(a.W + e, w);
            st_stream(a.m + e, m);
            st_stream(a.v + e, v);
            const uint2 p = make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w));
            for (int r = 0; r < R; ++r) st_stream(a.P.p[r] + e, p);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (!valid[k]) continue;
                const int64_t i = e + k;
                float w = a.W[i], m = a.m[i], v = a.v[i];
                adamw(a.s, scale_grad(a.s, acc[k]), w, m, v);
                a.W[i] = w;
                a.m[i] = m;
                a.v[i] = v;
                const uint16_t p = to_bf16(w);
                for (int r = 0; r < R; ++r) a.P.p[r][i] = p;
            }
        }
    }
}

template <int RC, int MC, int KIND, bool EF>
cudaError_t launch_comp_t(const CompArgs& a, cudaStream_t st)
{
    const void* k = reinterpret_cast<const void*>(&k_comp<RC, MC, KIND, EF>);
    const int64_t blocks = (a.n + kCompBlock - 1) / kCompBlock;   // one warp each
    const int64_t work = (blocks + kThreads / 32 - 1) / (kThreads / 32);
    // the sign codec without error feedback: 3.5 blocks per SM of the 4 that
    // fit, 0.962 -> 0.974 of the copy peak on the 1B-shaped workload and
    // 0.98 -> 1.0 on the GPT-2-shaped one (grid-size sweep); every other
    // codec measured fastest with all resident blocks
    constexpr int quarters = (KIND == ZERO_COMP_SIGN && !EF) ? 14 : 0;
    k_comp<RC, MC, KIND, EF><<<grid_for(k, work < 1 ? 1 : work, quarters), kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <int KIND, bool EF>
cudaError_t launch_comp_rm(const CompArgs& a, cudaStream_t st)
{
    if (a.R == 8 && a.M == 1) return launch_comp_t<8, 1, KIND, EF>(a, st);
    if (a.R == 4 && a.M == 1) return launch_comp_t<4, 1, KIND, EF>(a, st);
    if (a.R == 7 && a.M == 4) return launch_comp_t<7, 4, KIND, EF>(a, st);
    return launch_comp_t<0, 0, KIND, EF>(a, st);
}

cudaError_t launch_comp(const CompArgs& a, int kind, bool ef, cudaStream_t st)
{
    switch (kind) {
    case ZERO_COMP_FP16:
        return ef ? launch_comp_rm<ZERO_COMP_FP16, true>(a, st) : launch_comp_rm<ZERO_COMP_FP16, false>(a, st);
    case ZERO_COMP_INT8:
        return ef ? launch_comp_rm<ZERO_COMP_INT8, true>(a, st) : launch_comp_rm<ZERO_COMP_INT8, false>(a, st);
    default:
        return ef ? launch_comp_rm<ZERO_COMP_SIGN, true>(a, st) : launch_comp_rm<ZERO_COMP_SIGN, false>(a, st);
    }
}

}  // namespace

extern "C" zero_status zero_step_compressed(const zero_plan_t* plan,
                                            const uint16_t* const* rank_grads, float* master,
                                            float* m, float* v, uint16_t* const* rank_params,
                                            const zero_adamw_hparams* hp, int64_t step,
                                            int32_t kind, float* const* residuals, void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (zero_status e = check_hparams(hp, step)) return e;
    if (kind != ZERO_COMP_FP16 && kind != ZERO_COMP_INT8 && kind != ZERO_COMP_SIGN)
        return ZERO_ERR_INVALID_ARG;
    if (plan->N == 0) return ZERO_OK;
    Range rs[ZERO_MAX_RM + 2 * ZERO_MAX_R + 4];
    int nr = 0;
    if (zero_status e = check_grads(plan, rank_grads, rs, nr)) return e;
    if (zero_status e = check_replicas(plan, rank_params, rs, nr)) return e;
    if (zero_status e = check_state(plan, master, m, v, rs, nr)) return e;
    CompArgs a{};
    if (residuals) {
        for (int r = 0; r < plan->R; ++r) {
            if (zero_status e = check_ptr(residuals[r])) return e;
            rs[nr++] = rng(residuals[r], 4 * plan->N, true);
            a.E[r] = residuals[r];
        }
    }
    if (zero_status e = check_overlap(rs, nr)) return e;
    fill_grad_ptrs(a.g, plan, rank_grads);
    fill_replica_ptrs(a.P, plan, rank_params);
    a.W = master;
    a.m = m;
    a.v = v;
    a.n = plan->N;
    a.R = plan->R;
    a.M = plan->M;
    a.s = step_scalars(*hp, step, plan->R, plan->M);
    return cuda_status(launch_comp(a, kind, residuals != nullptr, static_cast<cudaStream_t>(stream)));
}

// ============================================================ 1-bit Adam ==
// zero_step_onebit after its warm-up: each rank's local momentum (plus its
// residual) goes through the sign codec, the owner averages the decoded
// momenta, adds its own residual and applies the codec again, and the update
// divides by the frozen preconditioner.  The plan's shard length is a
// multiple of the 128-element block, so a block of the flat vector never
// straddles two owners: one warp owns one block for the worker codecs, the
// owner's codec and the update alike, and the whole step is one pass.
namespace {

struct OneBitScalars {
    float b1, omb1;
    float decay;           // 1 - lr * wd
    float step_size;       // lr / (1 - beta1^t)
    float bc2f_sqrt;       // sqrt(1 - beta2^T_w), frozen at the end of the warm-up
    float eps;
    float denom_m, inv_m;  // M, and 1/M when M is a power of two
    float denom_r, inv_r;  // R, and 1/R when R is a power of two
    int32_t m_pow2, r_pow2;
};

struct OneBitArgs {
    GradPtrs g;
    ReplicaPtrs P;
    float* E[ZERO_MAX_R];  // worker residuals, N floats each
    float* Es;             // owner residuals, element i at index i
    float* W;
    float* m;
    const float* v;
    int64_t n;
    int32_t R, M;
    OneBitScalars s;
};

OneBitScalars onebit_scalars(const zero_adamw_hparams& hp, int64_t step, int64_t freeze_step,
                             int R, int M)
{
    const StepScalars now = step_scalars(hp, step, R, M);
    const StepScalars frozen = step_scalars(hp, freeze_step, R, M);
    OneBitScalars s;
    s.b1 = now.b1;
    s.omb1 = now.omb1;
    s.decay = now.decay;
    s.step_size = now.step_size;
    s.bc2f_sqrt = frozen.bc2_sqrt;
    s.eps = now.eps;
    s.denom_m = (float)M;
    s.m_pow2 = (M & (M - 1)) == 0;
    s.inv_m = s.m_pow2 ? 1.0f / (float)M : 0.0f;
    s.denom_r = (float)R;
    s.r_pow2 = (R & (R - 1)) == 0;
    s.inv_r = s.r_pow2 ? 1.0f / (float)R : 0.0f;
    return s;
}

// x / d, as a multiplication when d is a power of two (the same rounding)
__device__ __forceinline__ float div_by(float x, float d, float inv, int32_t pow2)
{
    return pow2 ? __fmul_rn(x, inv) : __fdiv_rn(x, d);
}

// one rank's worker stage on the 4 elements of a lane: local momentum from
// the micro-batch sum, residual added, sign codec, new residual returned in x
__device__ __forceinline__ void onebit_worker(const OneBitScalars& s, const float (&loc)[4],
                                              const float (&mo)[4], const float (&res)[4],
                                              const bool (&valid)[4], int64_t block_count,
                                              float (&x)[4], float (&d)[4])
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float gl = div_by(loc[k], s.denom_m, s.inv_m, s.m_pow2);
        const float ml = __fadd_rn(__fmul_rn(s.b1, mo[k]), __fmul_rn(s.omb1, gl));
        x[k] = __fadd_rn(ml, res[k]);
    }
    codec<ZERO_COMP_SIGN>(x, valid, block_count, d);
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = __fsub_rn(x[k], d[k]);
}

__device__ __forceinline__ float onebit_update(const OneBitScalars& s, float w, float ds, float v)
{
    const float wd = __fmul_rn(w, s.decay);
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.bc2f_sqrt), s.eps);
    return __fsub_rn(wd, __fmul_rn(s.step_size, __fdiv_rn(ds, den)));
}

template <int RC, int MC>
__global__ void __launch_bounds__(kThreads) k_onebit(const __grid_constant__ OneBitArgs a)
{
    const int R = RC > 0 ? RC : a.R;
    const int M = MC > 0 ? MC : a.M;
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
    const int64_t n = a.n;
    const int64_t nblk = (n + kCompBlock - 1) / kCompBlock;
    for (int64_t b = warp; b < nblk; b += nwarps) {       // warp-uniform loop
        const int64_t e = b * kCompBlock + 4 * lane;
        const bool full = b * kCompBlock + kCompBlock <= n;
        const int64_t block_count = full ? kCompBlock : n - b * kCompBlock;
        bool valid[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) valid[k] = e + k < n;
        float mo[4], es[4], w[4], vv[4], dsum[4];
        float4 q_es, q_w, q_v;                    // the owner's state of a full block
        bool have_owner = false;
        if (full) {
            const float4 q = ld_stream(a.m + e);
            mo[0] = q.x; mo[1] = q.y; mo[2] = q.z; mo[3] = q.w;
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) mo[k] = valid[k] ? a.m[e + k] : 0.0f;
        }
        if constexpr (RC > 0 && MC > 0) {
            if (full) {
                // every rank's loads first, then the codecs and their warp
                // reductions
                uint2 gx[RC * MC];
                float4 ex[RC];
#pragma unroll
                for (int q = 0; q < RC * MC; ++q) gx[q] = ld_stream(a.g.p[q] + e);
#pragma unroll
                for (int r = 0; r < RC; ++r) ex[r] = ld_stream(a.E[r] + e);
                q_es = ld_stream(a.Es + e);
                q_w = ld_stream(a.W + e);
                q_v = ld_stream(a.v + e);
                have_owner = true;
                if constexpr ((RC & (RC - 1)) == 0) {
                    // the worker codecs of all ranks, their block sums
                    // reduced together (sign_scales_joint)
                    float x[RC][4];
#pragma unroll
                    for (int r = 0; r < RC; ++r) {
                        float loc[4];
#pragma unroll
                        for (int j = 0; j < MC; ++j) {
                            const uint2 u = gx[r * MC + j];
                            const float y[4] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y),
                                                bf16_hi(u.y)};
#pragma unroll
                            for (int k = 0; k < 4; ++k) loc[k] = j == 0 ? y[k] : __fadd_rn(loc[k], y[k]);
                        }
                        const float res[4] = {ex[r].x, ex[r].y, ex[r].z, ex[r].w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float gl = div_by(loc[k], a.s.denom_m, a.s.inv_m, a.s.m_pow2);
                            const float ml = __fadd_rn(__fmul_rn(a.s.b1, mo[k]), __fmul_rn(a.s.omb1, gl));
                            x[r][k] = __fadd_rn(ml, res[k]);
                        }
                    }
                    float sc[RC];
                    sign_scales_joint<RC>(x, lane, sc);
#pragma unroll
                    for (int r = 0; r < RC; ++r) {
                        float d[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) d[k] = x[r][k] < 0.0f ? -sc[r] : sc[r];
                        st_stream(a.E[r] + e, make_float4(__fsub_rn(x[r][0], d[0]), __fsub_rn(x[r][1], d[1]),
                                                          __fsub_rn(x[r][2], d[2]), __fsub_rn(x[r][3], d[3])));
#pragma unroll
                        for (int k = 0; k < 4; ++k) dsum[k] = r == 0 ? d[k] : __fadd_rn(dsum[k], d[k]);
                    }
                } else {
#pragma unroll
                for (int r = 0; r < RC; ++r) {
                    float loc[4];
#pragma unroll
                    for (int j = 0; j < MC; ++j) {
                        const uint2 u = gx[r * MC + j];
                        const float y[4] = {bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y)};
#pragma unroll
                        for (int k = 0; k < 4; ++k) loc[k] = j == 0 ? y[k] : __fadd_rn(loc[k], y[k]);
                    }
                    const float res[4] = {ex[r].x, ex[r].y, ex[r].z, ex[r].w};
                    float x[4], d[4];
                    onebit_worker(a.s, loc, mo, res, valid, block_count, x, d);
                    st_stream(a.E[r] + e, make_float4(x[0], x[1], x[2], x[3]));
#pragma unroll
                    for (int k = 0; k < 4; ++k) dsum[k] = r == 0 ? d[k] : __fadd_rn(dsum[k], d[k]);
                }
                }
            }
        }
        if (!(RC > 0 && MC > 0) || !full) {
            for (int r = 0; r < R; ++r) {
                float loc[4], res[4];
                for (int j = 0; j < M; ++j) {
                    float y[4];
                    if (full) {
                        const uint2 u = ld_stream(a.g.p[r * M + j] + e);
                        y[0] = bf16_lo(u.x); y[1] = bf16_hi(u.x); y[2] = bf16_lo(u.y); y[3] = bf16_hi(u.y);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k) y[k] = valid[k] ? bf16_bits(a.g.p[r * M + j][e + k]) : 0.0f;
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) loc[k] = j == 0 ? y[k] : __fadd_rn(loc[k], y[k]);
                }
                if (full) {
                    const float4 q = ld_stream(a.E[r] + e);
                    res[0] = q.x; res[1] = q.y; res[2] = q.z; res[3] = q.w;
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) res[k] = valid[k] ? a.E[r][e + k] : 0.0f;
                }
                float x[4], d[4];
                onebit_worker(a.s, loc, mo, res, valid, block_count, x, d);
                if (full) {
                    st_stream(a.E[r] + e, make_float4(x[0], x[1], x[2], x[3]));
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) if (valid[k]) a.E[r][e + k] = x[k];
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) dsum[k] = r == 0 ? d[k] : __fadd_rn(dsum[k], d[k]);
            }
        }
        // the owner: average, its residual, the codec again, the update
        if (full) {
            if (!have_owner) {
                q_es = ld_stream(a.Es + e);
                q_w = ld_stream(a.W + e);
                q_v = ld_stream(a.v + e);
            }
            const float4 q = q_es, wq = q_w, vq = q_v;
            es[0] = q.x; es[1] = q.y; es[2] = q.z; es[3] = q.w;
            w[0] = wq.x; w[1] = wq.y; w[2] = wq.z; w[3] = wq.w;
            vv[0] = vq.x; vv[1] = vq.y; vv[2] = vq.z; vv[3] = vq.w;
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                es[k] = valid[k] ? a.Es[e + k] : 0.0f;
                w[k] = valid[k] ? a.W[e + k] : 0.0f;
                vv[k] = valid[k] ? a.v[e + k] : 0.0f;
            }
        }
        float y[4], ds[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            y[k] = __fadd_rn(div_by(dsum[k], a.s.denom_r, a.s.inv_r, a.s.r_pow2), es[k]);
        codec<ZERO_COMP_SIGN>(y, valid, block_count, ds);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            es[k] = __fsub_rn(y[k], ds[k]);
            w[k] = onebit_update(a.s, w[k], ds[k], vv[k]);
        }
        if (full) {
            st_stream(a.Es + e, make_float4(es[0], es[1], es[2], es[3]));
            st_stream(a.m + e, make_float4(ds[0], ds[1], ds[2], ds[3]));
            st_stream(a.W + e, make_float4(w[0], w[1], w[2], w[3]));
            const uint2 p = make_uint2(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]));
            for (int r = 0; r < R; ++r) st_stream(a.P.p[r] + e, p);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (!valid[k]) continue;
                const int64_t i = e + k;
                a.Es[i] = es[k];
                a.m[i] = ds[k];
                a.W[i] = w[k];
                const uint16_t p = to_bf16(w[k]);
                for (int r = 0; r < R; ++r) a.P.p[r][i] = p;
            }
        }
    }
}

template <int RC, int MC>
cudaError_t launch_onebit_t(const OneBitArgs& a, cudaStream_t st)
{
    const void* k = reinterpret_cast<const void*>(&k_onebit<RC, MC>);
    const int64_t blocks = (a.n + kCompBlock - 1) / kCompBlock;   // one warp each
    const int64_t work = (blocks + kThreads / 32 - 1) / (kThreads / 32);
    k_onebit<RC, MC><<<grid_for(k, work < 1 ? 1 : work), kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_onebit(const OneBitArgs& a, cudaStream_t st)
{
    if (a.R == 8 && a.M == 1) return launch_onebit_t<8, 1>(a, st);
    if (a.R == 4 && a.M == 1) return launch_onebit_t<4, 1>(a, st);
    if (a.R == 7 && a.M == 4) return launch_onebit_t<7, 4>(a, st);
    return launch_onebit_t<0, 0>(a, st);
}

}  // namespace

extern "C" zero_status zero_step_onebit(const zero_plan_t* plan,
                                        const uint16_t* const* rank_grads, float* master,
                                        float* m, float* v, uint16_t* const* rank_params,
                                        const zero_adamw_hparams* hp, int64_t step,
                                        int64_t freeze_step, float* const* worker_residuals,
                                        float* server_residual, void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (zero_status e = check_hparams(hp, step)) return e;
    if (freeze_step < 1 || plan->S % kCompBlock != 0) return ZERO_ERR_INVALID_ARG;
    if (!worker_residuals) return ZERO_ERR_NULL;
    if (zero_status e = check_ptr(server_residual)) return e;
    for (int r = 0; r < plan->R; ++r)
        if (zero_status e = check_ptr(worker_residuals[r])) return e;
    if (step <= freeze_step)     // the warm-up: the plain fused step
        return zero_step(plan, rank_grads, master, m, v, rank_params, hp, step,
                         ZERO_VARIANT_FUSED, nullptr, 0, 0, nullptr, stream);
    if (plan->N == 0) return ZERO_OK;
    Range rs[ZERO_MAX_RM + 3 * ZERO_MAX_R + 5];
    int nr = 0;
    if (zero_status e = check_grads(plan, rank_grads, rs, nr)) return e;
    if (zero_status e = check_replicas(plan, rank_params, rs, nr)) return e;
    if (zero_status e = check_state(plan, master, m, v, rs, nr)) return e;
    rs[nr++] = rng(server_residual, 4 * plan->padded, true);
    OneBitArgs a{};
    for (int r = 0; r < plan->R; ++r) {
        rs[nr++] = rng(worker_residuals[r], 4 * plan->N, true);
        a.E[r] = worker_residuals[r];
    }
    if (zero_status e = check_overlap(rs, nr)) return e;
    fill_grad_ptrs(a.g, plan, rank_grads);
    fill_replica_ptrs(a.P, plan, rank_params);
    a.Es = server_residual;
    a.W = master;
    a.m = m;
    a.v = v;
    a.n = plan->N;
    a.R = plan->R;
    a.M = plan->M;
    a.s = onebit_scalars(*hp, step, freeze_step, plan->R, plan->M);
    return cuda_status(launch_onebit(a, static_cast<cudaStream_t>(stream)));
}

// ============================================== fused step, TMA bulk staging ==
// k_fused_tma: the fused step with the R*M gradient tiles and the three
// state tiles of each 1024-element tile brought into shared memory by
// cp.async.bulk (one elected thread, completion on an mbarrier, 3 stages
// in flight per block) and the replica tile written back by R bulk stores
// from a double-buffered shared tile.  Same arithmetic as k_fused, same bits.
// On this access pattern it measures a few percent below the register-
// direct k_fused, which stays the default; it is the selectable variant
// ZERO_VARIANT_FUSED_TMA.
//
// Every mbarrier wait is bounded.  When a wait runs out, the whole block
// (the decision is block-uniform) stops, thread 0 waits - again bounded -
// for the stage loads it has issued and not consumed, and for its bulk
// stores, sets ZERO_DEV_TIMEOUT in the status word and the block returns, so
// no copy can land in shared memory after the block has left.
namespace {

constexpr int kTmaTile = 1024;                   // 256 threads x 4 elements
constexpr int kTmaStages = 3;
constexpr uint32_t kWaitLimit = 1u << 22;        // tries of mbarrier.try_wait
constexpr uint32_t kDrainLimit = 1u << 24;

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, uint32_t limit)
{
    for (uint32_t it = 0; it < limit; ++it)
        if (mbar_try(b, parity)) return true;
    return false;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* b)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(b))
        : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_addr(src)), "r"(bytes)
                 : "memory");
}

struct TmaLayout {
    uint32_t stage_bytes, smem_bytes;
};

TmaLayout tma_layout(int RM)
{
    TmaLayout L;
    L.stage_bytes = (uint32_t)(RM * kTmaTile * 2 + 3 * kTmaTile * 4);
    L.smem_bytes = 128 + kTmaStages * L.stage_bytes + 2 * kTmaTile * 2;
    return L;
}

__global__ void __launch_bounds__(kThreads) k_fused_tma(const __grid_constant__ FusedArgs a,
                                                        uint32_t wait_limit, int32_t check)
{
    const int R = a.R, M = a.M, RM = R * M;
    constexpr uint32_t GB = kTmaTile * 2, SB = kTmaTile * 4;
    const uint32_t stage_bytes = (uint32_t)RM * GB + 3 * SB;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint8_t* stages = smem + 128;
    uint16_t* outbuf = reinterpret_cast<uint16_t*>(stages + kTmaStages * stage_bytes);
    const int64_t ntiles = a.n / kTmaTile;
    const int64_t my = ntiles > blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int tid = threadIdx.x;

    if (tid == 0) {
        for (int s = 0; s < kTmaStages; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    auto issue = [&](int64_t k) {
        const int s = (int)(k % kTmaStages);
        const int64_t e = (blockIdx.x + k * gridDim.x) * (int64_t)kTmaTile;
        uint8_t* st = stages + s * stage_bytes;
        mbar_expect_tx(&full[s], stage_bytes);
        for (int q = 0; q < RM; ++q) bulk_load(st + q * GB, a.g.p[q] + e, GB, &full[s]);
        bulk_load(st + RM * GB, a.W + e, SB, &full[s]);
        bulk_load(st + RM * GB + SB, a.m + e, SB, &full[s]);
        bulk_load(st + RM * GB + 2 * SB, a.v + e, SB, &full[s]);
    };
    if (tid == 0)
        for (int64_t k = 0; k < kTmaStages && k < my; ++k) issue(k);

    bool timed_out = false, bad = false;
    int64_t k_fail = 0;
    for (int64_t k = 0; k < my; ++k) {
        const int s = (int)(k % kTmaStages);
        const uint32_t ph = (uint32_t)((k / kTmaStages) & 1);
        const bool ok = mbar_wait(&full[s], ph, wait_limit);
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            k_fail = k;
            break;
        }
        const uint8_t* st = stages + s * stage_bytes;
        const int64_t tile0 = (blockIdx.x + k * gridDim.x) * (int64_t)kTmaTile;
        const int64_t e = tile0 + tid * 4;
        float loc[4], tot[4];
        int r = 0, j = 0;
        for (int q = 0; q < RM; ++q) {
            const uint2 x = *reinterpret_cast<const uint2*>(st + q * GB + tid * 8);
            fold4(loc, tot, x, r, j, M);
            if (++j == M) { j = 0; ++r; }
        }
        float4 w = *reinterpret_cast<const float4*>(st + RM * GB + tid * 16);
        float4 m = *reinterpret_cast<const float4*>(st + RM * GB + SB + tid * 16);
        float4 v = *reinterpret_cast<const float4*>(st + RM * GB + 2 * SB + tid * 16);
        float* wp = &w.x;
        float* mp = &m.x;
        float* vp = &v.x;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float g = scale_grad(a.s, tot[q]);
            if (check) bad |= !isfinite(g);
            adamw(a.s, g, wp[q], mp[q], vp[q]);
        }
        st_stream(a.W + e, w);
        st_stream(a.m + e, m);
        st_stream(a.v + e, v);
        uint16_t* ob = outbuf + (k & 1) * kTmaTile;
        *reinterpret_cast<uint2*>(ob + tid * 4) =
            make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w));
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();                       // stage s consumed, replica tile written
        if (tid == 0) {
            for (int q = 0; q < R; ++q) bulk_store(a.P.p[q] + tile0, ob, GB);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            if (k + kTmaStages < my) issue(k + kTmaStages);
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");   // tile k-1's stores
        }
        __syncthreads();                       // out tile (k+1)&1 free again
    }

    if (timed_out) {
        if (tid == 0) {
            if (a.status) atomicOr(a.status, ZERO_DEV_TIMEOUT);
            // the loads issued for tiles k_fail .. k_fail+stages-1 must land
            // before this block's shared memory can be given to another block
            for (int64_t kk = k_fail; kk < k_fail + kTmaStages && kk < my; ++kk)
                mbar_wait(&full[kk % kTmaStages], (uint32_t)((kk / kTmaStages) & 1), kDrainLimit);
        }
        __syncthreads();
    }
    if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");

    // the last partial tile, element by element, by the block that owns it
    const int64_t tail0 = ntiles * kTmaTile;
    if (!timed_out && tail0 < a.n && blockIdx.x == (unsigned)(ntiles % gridDim.x)) {
        for (int64_t i = tail0 + tid; i < a.n; i += kThreads) {
            const float g = scale_grad(a.s, grad_sum1(a.g, R, M, i));
            if (check) bad |= !isfinite(g);
            float w = a.W[i], m = a.m[i], v = a.v[i];
            adamw(a.s, g, w, m, v);
            a.W[i] = w;
            a.m[i] = m;
            a.v[i] = v;
            const uint16_t p = to_bf16(w);
            for (int q = 0; q < R; ++q) a.P.p[q][i] = p;
        }
    }
    if (check && __any_sync(0xFFFFFFFFu, bad) && (tid & 31) == 0 && a.status)
        atomicOr(a.status, ZERO_DEV_NONFINITE);
}

cudaError_t launch_fused_tma(const FusedArgs& a, bool expire_waits, bool check, cudaStream_t st)
{
    const TmaLayout L = tma_layout(a.R * a.M);
    int dev = 0;
    cudaGetDevice(&dev);
    static std::mutex mu;
    static uint32_t configured[64] = {};         // largest dynamic smem set per device
    {
        std::lock_guard<std::mutex> lk(mu);
        if (configured[dev & 63] < L.smem_bytes) {
            cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&k_fused_tma),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)L.smem_bytes);
            if (e != cudaSuccess) return e;
            configured[dev & 63] = L.smem_bytes;
        }
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void*>(&k_fused_tma),
                                                      kThreads, L.smem_bytes) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t tiles = a.n / kTmaTile;
    int64_t grid = (int64_t)device_sms(dev) * per_sm;
    if (grid > tiles) grid = tiles;
    if (grid < 1) grid = 1;
    k_fused_tma<<<(unsigned)grid, kThreads, L.smem_bytes, st>>>(a, expire_waits ? 0u : kWaitLimit,
                                                               check ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace

// ====================================================== replica consistency ==
// zero_check_replicas: count the elements where any rank's replica differs
// from rank 0's, and the first such index - a silent-data-corruption check
// (every replica must hold the same bits after the all-gather).
namespace {

struct CheckArgs {
    ReplicaPtrs P;
    int64_t n;
    int32_t R;
    unsigned long long* count;
    long long* first;
};

__global__ void __launch_bounds__(kThreads) k_check(const __grid_constant__ CheckArgs a)
{
    const int64_t nvec = a.n / 8;
    unsigned long long bad = 0;
    long long first = LLONG_MAX;
    for (int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x; q < nvec;
         q += (int64_t)gridDim.x * kThreads) {
        const int64_t e = q * 8;
        const uint4 r0 = __ldcs(reinterpret_cast<const uint4*>(a.P.p[0] + e));
        uint32_t diff[4] = {0, 0, 0, 0};
        for (int r = 1; r < a.R; ++r) {
            const uint4 x = __ldcs(reinterpret_cast<const uint4*>(a.P.p[r] + e));
            diff[0] |= x.x ^ r0.x;
            diff[1] |= x.y ^ r0.y;
            diff[2] |= x.z ^ r0.z;
            diff[3] |= x.w ^ r0.w;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (diff[k] & 0xFFFFu) { ++bad; first = min(first, (long long)(e + 2 * k)); }
            if (diff[k] >> 16) { ++bad; first = min(first, (long long)(e + 2 * k + 1)); }
        }
    }
    if (blockIdx.x == 0) {
        for (int64_t i = nvec * 8 + threadIdx.x; i < a.n; i += kThreads) {
            bool d = false;
            for (int r = 1; r < a.R; ++r) d |= a.P.p[r][i] != a.P.p[0][i];
            if (d) { ++bad; first = min(first, (long long)i); }
        }
    }
    // warp-aggregated: one atomic per warp that saw a mismatch
    for (int off = 16; off > 0; off >>= 1) {
        bad += __shfl_down_sync(0xFFFFFFFFu, bad, off);
        first = min(first, __shfl_down_sync(0xFFFFFFFFu, first, off));
    }
    if ((threadIdx.x & 31) == 0 && bad) {
        atomicAdd(a.count, bad);
        if (a.first) atomicMin(a.first, first);
    }
}

}  // namespace

extern "C" zero_status zero_check_replicas(const zero_plan_t* plan, uint16_t* const* rank_params,
                                           int64_t* dev_count, int64_t* dev_first, void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (!dev_count) return ZERO_ERR_NULL;
    if (((uintptr_t)dev_count & 7u) || ((uintptr_t)dev_first & 7u)) return ZERO_ERR_ALIGN;
    Range rs[ZERO_MAX_R + 2];
    int nr = 0;
    if (plan->N > 0)
        if (zero_status e = check_replicas(plan, rank_params, rs, nr)) return e;
    for (int k = 0; k < nr; ++k) rs[k].out = false;             // read only here
    rs[nr++] = rng(dev_count, 8, true);
    if (dev_first) rs[nr++] = rng(dev_first, 8, true);
    if (zero_status e = check_overlap(rs, nr)) return e;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const long long none = LLONG_MAX;
    if (cudaMemsetAsync(dev_count, 0, 8, st) != cudaSuccess) return ZERO_ERR_CUDA;
    if (dev_first && cudaMemcpyAsync(dev_first, &none, 8, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return ZERO_ERR_CUDA;
    if (plan->N == 0 || plan->R == 1) return ZERO_OK;
    CheckArgs a{};
    fill_replica_ptrs(a.P, plan, rank_params);
    a.n = plan->N;
    a.R = plan->R;
    a.count = reinterpret_cast<unsigned long long*>(dev_count);
    a.first = reinterpret_cast<long long*>(dev_first);
    const void* k = reinterpret_cast<const void*>(&k_check);
    const int64_t work = (a.n / 8 + kThreads - 1) / kThreads;
    k_check<<<grid_for(k, work < 1 ? 1 : work), kThreads, 0, st>>>(a);
    return cuda_status(cudaGetLastError());
}

// ================================================================ ZeRO-3 ==
// zero3_step: the fused reduce-scatter + AdamW with the bf16 result cast
// into each rank's own parameter shard (one buffer in the padded layout of
// the state); no all-gather.  zero3_gather: the all-gather of one unit
// [lo, hi) of the flat vector from the shards into n_out transient buffers
// (the ranks that need the unit), on demand before its use.
//
// k_gather copies 8 elements (16 bytes) per thread to every destination.
// A unit can start at any element, so the source window of a destination
// vector is shifted by SHIFT = lo mod 8 elements: the thread loads the two
// aligned 16-byte source vectors that cover it and funnel-shifts them into
// place (SHIFT is a template parameter: 8 instantiations).  Vectors whose
// source window would cross the end of the shard buffer, and the last
// partial vector, are copied element by element.
namespace {

struct GatherArgs {
    ReplicaPtrs out;
    const uint16_t* src;
    int64_t src_len;       // elements in the shard buffer (plan->padded)
    int64_t lo, len;
    int32_t n_out;
};

template <int SHIFT>
__device__ __forceinline__ uint4 realign8(uint4 A, uint4 B)
{
    const uint32_t w[8] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w};
    constexpr int h = SHIFT / 2;
    uint4 r;
    if constexpr (SHIFT % 2 == 0) {
        r.x = w[h];
        r.y = w[h + 1];
        r.z = w[h + 2];
        r.w = w[h + 3];
    } else {
        r.x = __funnelshift_r(w[h], w[h + 1], 16);
        r.y = __funnelshift_r(w[h + 1], w[h + 2], 16);
        r.z = __funnelshift_r(w[h + 2], w[h + 3], 16);
        r.w = __funnelshift_r(w[h + 3], w[h + 4], 16);
    }
    return r;
}

template <int SHIFT>
__global__ void __launch_bounds__(kThreads) k_gather(const __grid_constant__ GatherArgs a)
{
    const int64_t base = a.lo - SHIFT;            // 8-element (16-byte) aligned
    const int64_t nvec = a.len / 8;
    constexpr int64_t window = SHIFT ? 16 : 8;
    for (int64_t k = (int64_t)blockIdx.x * kThreads + threadIdx.x; k < nvec;
         k += (int64_t)gridDim.x * kThreads) {
        const int64_t sb = base + 8 * k;
        uint4 v;
        if (sb + window <= a.src_len) {
            const uint4 A = __ldcs(reinterpret_cast<const uint4*>(a.src + sb));
            if constexpr (SHIFT == 0) {
                v = A;
            } else {
                const uint4 B = __ldcs(reinterpret_cast<const uint4*>(a.src + sb + 8));
                v = realign8<SHIFT>(A, B);
            }
        } else {
            uint16_t t[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) t[j] = a.src[a.lo + 8 * k + j];
            v.x = (uint32_t)t[0] | ((uint32_t)t[1] << 16);
            v.y = (uint32_t)t[2] | ((uint32_t)t[3] << 16);
            v.z = (uint32_t)t[4] | ((uint32_t)t[5] << 16);
            v.w = (uint32_t)t[6] | ((uint32_t)t[7] << 16);
        }
        for (int o = 0; o < a.n_out; ++o) __stcs(reinterpret_cast<uint4*>(a.out.p[o] + 8 * k), v);
    }
    if (blockIdx.x == 0) {
        for (int64_t d = nvec * 8 + threadIdx.x; d < a.len; d += kThreads) {
            const uint16_t x = a.src[a.lo + d];
            for (int o = 0; o < a.n_out; ++o) a.out.p[o][d] = x;
        }
    }
}

cudaError_t launch_gather(const GatherArgs& a, cudaStream_t st)
{
    const int64_t work = (a.len / 8 + kThreads - 1) / kThreads;
    auto go = [&](const void* k, auto kern) {
        kern<<<grid_for(k, work < 1 ? 1 : work), kThreads, 0, st>>>(a);
        return cudaGetLastError();
    };
    switch ((int)(a.lo & 7)) {
    case 0: return go(reinterpret_cast<const void*>(&k_gather<0>), k_gather<0>);
    case 1: return go(reinterpret_cast<const void*>(&k_gather<1>), k_gather<1>);
    case 2: return go(reinterpret_cast<const void*>(&k_gather<2>), k_gather<2>);
    case 3: return go(reinterpret_cast<const void*>(&k_gather<3>), k_gather<3>);
    case 4: return go(reinterpret_cast<const void*>(&k_gather<4>), k_gather<4>);
    case 5: return go(reinterpret_cast<const void*>(&k_gather<5>), k_gather<5>);
    case 6: return go(reinterpret_cast<const void*>(&k_gather<6>), k_gather<6>);
    default: return go(reinterpret_cast<const void*>(&k_gather<7>), k_gather<7>);
    }
}

}  // namespace

extern "C" zero_status zero3_step(const zero_plan_t* plan, const uint16_t* const* rank_grads,
                                  float* master, float* m, float* v, uint16_t* param_shards,
                                  const zero_adamw_hparams* hp, int64_t step, int32_t flags,
                                  int32_t* dev_status, void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (zero_status e = check_hparams(hp, step)) return e;
    if (flags & ~ZERO_FLAG_CHECK_FINITE) return ZERO_ERR_INVALID_ARG;
    if ((flags & ZERO_FLAG_CHECK_FINITE) && !dev_status) return ZERO_ERR_NULL;
    if (plan->N == 0) return ZERO_OK;
    Range rs[ZERO_MAX_RM + 6];
    int nr = 0;
    if (zero_status e = check_grads(plan, rank_grads, rs, nr)) return e;
    if (zero_status e = check_state(plan, master, m, v, rs, nr)) return e;
    if (zero_status e = check_ptr(param_shards)) return e;
    rs[nr++] = rng(param_shards, 2 * plan->padded, true);
    if (dev_status) rs[nr++] = rng(dev_status, 4, true);
    if (zero_status e = check_overlap(rs, nr)) return e;
    FusedArgs a{};
    fill_grad_ptrs(a.g, plan, rank_grads);
    a.P.p[0] = param_shards;
    a.zero3 = 1;
    a.W = master;
    a.m = m;
    a.v = v;
    a.n = plan->N;
    a.R = plan->R;
    a.M = plan->M;
    a.s = step_scalars(*hp, step, plan->R, plan->M);
    a.status = dev_status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool check = (flags & ZERO_FLAG_CHECK_FINITE) != 0;
    return cuda_status(check ? launch_fused<true>(a, st) : launch_fused<false>(a, st));
}

extern "C" zero_status zero3_gather(const zero_plan_t* plan, const uint16_t* param_shards,
                                    int64_t lo, int64_t hi, uint16_t* const* outs, int32_t n_out,
                                    void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (lo < 0 || hi < lo || hi > plan->N) return ZERO_ERR_INVALID_ARG;
    if (n_out < 1 || n_out > plan->R) return ZERO_ERR_INVALID_ARG;
    if (hi == lo) return ZERO_OK;
    if (!outs) return ZERO_ERR_NULL;
    Range rs[ZERO_MAX_R + 1];
    int nr = 0;
    if (zero_status e = check_ptr(param_shards)) return e;
    rs[nr++] = rng(param_shards, 2 * plan->padded, false);
    for (int o = 0; o < n_out; ++o) {
        if (zero_status e = check_ptr(outs[o])) return e;
        rs[nr++] = rng(outs[o], 2 * (hi - lo), true);
    }
    if (zero_status e = check_overlap(rs, nr)) return e;
    GatherArgs a{};
    for (int o = 0; o < n_out; ++o) a.out.p[o] = outs[o];
    a.src = param_shards;
    a.src_len = plan->padded;
    a.lo = lo;
    a.len = hi - lo;
    a.n_out = n_out;
    return cuda_status(launch_gather(a, static_cast<cudaStream_t>(stream)));
}

// ============================================= ZeRO-3, unit by unit (FSDP) ==
// zero3_rs_unit: right after a unit's backward, the ordered fp32 average of
// the unit's R*M gradient buffers goes into the owners' fp32 gradient shards
// (element i at index i); zero3_update then updates every owned element from
// its shard and casts it into the rank's own bf16 parameter shard.  Over a
// set of units that covers the vector once the result is zero3_step's, bit
// for bit: the same ordered sums, the same division, the same update.
// A unit may start at any element: its buffers are read as 4-vectors from
// their own start, and the fp32 shard stores are 16-byte vectors only when
// the unit starts on a multiple of 4 (a warp-uniform choice), else scalars.
namespace {

struct UnitArgs {
    GradPtrs g;            // the unit's buffers, element i at index i - lo
    float* gs;             // fp32 gradient shards, element i at index i
    int64_t lo, len;
    int32_t R, M;
    StepScalars s;
    int32_t* status;
};

// the divisor R*M of scale_grad, the only scalars the reduce-scatter uses
StepScalars divisor_scalars(int R, int M)
{
    StepScalars s{};
    const int rm = R * M;
    s.denom_rm = (float)rm;
    s.rm_pow2 = (rm & (rm - 1)) == 0;
    s.inv_rm = s.rm_pow2 ? 1.0f / (float)rm : 0.0f;
    return s;
}

template <int RC, int MC, bool CHECK>
__global__ void __launch_bounds__(kThreads) k_rs_unit(const __grid_constant__ UnitArgs a)
{
    const int R = RC > 0 ? RC : a.R;
    const int M = MC > 0 ? MC : a.M;
    const int64_t nvec = a.len / kVec;
    const bool vec_store = (a.lo & 3) == 0;
    float* out = a.gs + a.lo;
    bool bad = false;
    for (int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x; q < nvec;
         q += (int64_t)gridDim.x * kThreads) {
        const int64_t k = q * kVec;
        float acc[4];
        grad_sum4<RC, MC>(a.g, R, M, k, acc);
        float o[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            o[c] = scale_grad(a.s, acc[c]);
            if (CHECK) bad |= !isfinite(o[c]);
        }
        if (vec_store) {
            st_stream(out + k, make_float4(o[0], o[1], o[2], o[3]));
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) out[k + c] = o[c];
        }
    }
    if (blockIdx.x == 0) {
        for (int64_t k = nvec * kVec + threadIdx.x; k < a.len; k += kThreads) {
            const float g = scale_grad(a.s, grad_sum1(a.g, R, M, k));
            if (CHECK) bad |= !isfinite(g);
            out[k] = g;
        }
    }
    report_nonfinite<CHECK>(bad, a.status);
}

template <bool CHECK>
cudaError_t launch_rs_unit(const UnitArgs& a, cudaStream_t st)
{
    const int64_t work = (a.len / kVec + kThreads - 1) / kThreads;
    auto go = [&](const void* k, auto kern) {
        kern<<<grid_for(k, work < 1 ? 1 : work), kThreads, 0, st>>>(a);
        return cudaGetLastError();
    };
#define ZERO_CASE(r_, m_)                                                      \
    if (a.R == r_ && a.M == m_)                                                \
        return go(reinterpret_cast<const void*>(&k_rs_unit<r_, m_, CHECK>),    \
                  k_rs_unit<r_, m_, CHECK>);
    ZERO_CASE(8, 1) ZERO_CASE(4, 1) ZERO_CASE(2, 1) ZERO_CASE(1, 1) ZERO_CASE(16, 1)
    ZERO_CASE(4, 2) ZERO_CASE(7, 4) ZERO_CASE(8, 2) ZERO_CASE(4, 4) ZERO_CASE(2, 2)
#undef ZERO_CASE
    return go(reinterpret_cast<const void*>(&k_rs_unit<0, 0, CHECK>), k_rs_unit<0, 0, CHECK>);
}

struct Z3UpdateArgs {
    const float* gs;
    float* W;
    float* m;
    float* v;
    uint16_t* Ps;          // bf16 parameter shards, element i at index i
    int64_t n;
    StepScalars s;
};

__global__ void __launch_bounds__(kThreads) k_z3_update(const __grid_constant__ Z3UpdateArgs a)
{
    const int64_t nvec = a.n / kVec;
    for (int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x; q < nvec;
         q += (int64_t)gridDim.x * kThreads) {
        const int64_t e = q * kVec;
        const float4 g = ld_stream(a.gs + e);
        float4 w = ld_stream(a.W + e), m = ld_stream(a.m + e), v = ld_stream(a.v + e);
        adamw(a.s, g.x, w.x, m.x, v.x);
        adamw(a.s, g.y, w.y, m.y, v.y);
        adamw(a.s, g.z, w.z, m.z, v.z);
        adamw(a.s, g.w, w.w, m.w, v.w);
        st_stream(a.W + e, w);
        st_stream(a.m + e, m);
        st_stream(a.v + e, v);
        st_stream(a.Ps + e, make_uint2(pack_bf16x2(w.x, w.y), pack_bf16x2(w.z, w.w)));
    }
    if (blockIdx.x == 0) {
        for (int64_t i = nvec * kVec + threadIdx.x; i < a.n; i += kThreads) {
            float w = a.W[i], m = a.m[i], v = a.v[i];
            adamw(a.s, a.gs[i], w, m, v);
            a.W[i] = w;
            a.m[i] = m;
            a.v[i] = v;
            a.Ps[i] = to_bf16(w);
        }
    }
}

}  // namespace

extern "C" zero_status zero3_rs_unit(const zero_plan_t* plan, const uint16_t* const* unit_grads,
                                     int64_t lo, int64_t hi, float* grad_shards, int32_t flags,
                                     int32_t* dev_status, void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (lo < 0 || hi < lo || hi > plan->N) return ZERO_ERR_INVALID_ARG;
    if (flags & ~ZERO_FLAG_CHECK_FINITE) return ZERO_ERR_INVALID_ARG;
    if ((flags & ZERO_FLAG_CHECK_FINITE) && !dev_status) return ZERO_ERR_NULL;
    if (hi == lo) return ZERO_OK;
    if (!unit_grads) return ZERO_ERR_NULL;
    Range rs[ZERO_MAX_RM + 2];
    int nr = 0;
    const int RM = plan->R * plan->M;
    for (int q = 0; q < RM; ++q) {
        if (zero_status e = check_ptr(unit_grads[q])) return e;
        rs[nr++] = rng(unit_grads[q], 2 * (hi - lo), false);
    }
    if (zero_status e = check_ptr(grad_shards)) return e;
    rs[nr++] = rng(grad_shards, 4 * plan->padded, true);
    if (dev_status) rs[nr++] = rng(dev_status, 4, true);
    if (zero_status e = check_overlap(rs, nr)) return e;
    UnitArgs a{};
    for (int q = 0; q < RM; ++q) a.g.p[q] = unit_grads[q];
    a.gs = grad_shards;
    a.lo = lo;
    a.len = hi - lo;
    a.R = plan->R;
    a.M = plan->M;
    a.s = divisor_scalars(plan->R, plan->M);
    a.status = dev_status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool check = (flags & ZERO_FLAG_CHECK_FINITE) != 0;
    return cuda_status(check ? launch_rs_unit<true>(a, st) : launch_rs_unit<false>(a, st));
}

extern "C" zero_status zero3_update(const zero_plan_t* plan, const float* grad_shards,
                                    float* master, float* m, float* v, uint16_t* param_shards,
                                    const zero_adamw_hparams* hp, int64_t step, void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (zero_status e = check_hparams(hp, step)) return e;
    if (plan->N == 0) return ZERO_OK;
    Range rs[6];
    int nr = 0;
    if (zero_status e = check_ptr(grad_shards)) return e;
    rs[nr++] = rng(grad_shards, 4 * plan->padded, false);
    if (zero_status e = check_state(plan, master, m, v, rs, nr)) return e;
    if (zero_status e = check_ptr(param_shards)) return e;
    rs[nr++] = rng(param_shards, 2 * plan->padded, true);
    if (zero_status e = check_overlap(rs, nr)) return e;
    Z3UpdateArgs a{};
    a.gs = grad_shards;
    a.W = master;
    a.m = m;
    a.v = v;
    a.Ps = param_shards;
    a.n = plan->N;
    a.s = step_scalars(*hp, step, plan->R, plan->M);
    const void* k = reinterpret_cast<const void*>(&k_z3_update);
    const int64_t work = (a.n / kVec + kThreads - 1) / kThreads;
    // 3 blocks per SM of the 5 that fit: 0.955 -> 0.98 of the copy peak on
    // the 1B-shaped workload (grid-size sweep)
    const unsigned grid = grid_for(k, work < 1 ? 1 : work, 12);
    k_z3_update<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cuda_status(cudaGetLastError());
}

// ================================================ staged step, no allocation ==
// zero_step_staged_noalloc: the staged trio with its fp32 reduced-gradient
// scratch in a fixed device array of this file instead of a caller buffer,
// for callers that cannot allocate device memory.  The array's address is a
// device address only on the device side; host code looks it up once per
// device with cudaGetSymbolAddress (with that device current) and passes it
// to the kernels like any other scratch pointer.
namespace {

static __device__ __align__(256) float g_noalloc_scratch[ZERO_NOALLOC_MAX_ELEMS];

std::mutex g_noalloc_mu;
float* g_noalloc_addr[64] = {};            // per device ordinal, looked up once

zero_status noalloc_scratch(float** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ZERO_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();            // clear it so later launch checks do not see it
            return ZERO_ERR_CUDA;
        }
        g_noalloc_addr[dev] = static_cast<float*>(p);
    }
    *out = g_noalloc_addr[dev];
    return ZERO_OK;
}

}  // namespace

extern "C" zero_status zero_step_staged_noalloc(const zero_plan_t* plan,
                                                const uint16_t* const* rank_grads, float* master,
                                                float* m, float* v,
                                                uint16_t* const* rank_params,
                                                const zero_adamw_hparams* hp, int64_t step,
                                                int32_t flags, int32_t* dev_status, void* stream)
{
    if (zero_status e = check_plan(plan)) return e;
    if (plan->padded > (int64_t)ZERO_NOALLOC_MAX_ELEMS) return ZERO_ERR_SIZE;
    if (zero_status e = check_hparams(hp, step)) return e;
    if (flags & ~ZERO_FLAG_CHECK_FINITE) return ZERO_ERR_INVALID_ARG;
    if ((flags & ZERO_FLAG_CHECK_FINITE) && !dev_status) return ZERO_ERR_NULL;
    if (plan->N == 0) return ZERO_OK;

    Range rs[ZERO_MAX_RM + ZERO_MAX_R + 4];
    int nr = 0;
    if (zero_status e = check_grads(plan, rank_grads, rs, nr)) return e;
    if (zero_status e = check_replicas(plan, rank_params, rs, nr)) return e;
    if (zero_status e = check_state(plan, master, m, v, rs, nr)) return e;
    if (dev_status) rs[nr++] = rng(dev_status, 4, true);
    if (zero_status e = check_overlap(rs, nr)) return e;

    float* scratch = nullptr;
    if (zero_status e = noalloc_scratch(&scratch)) return e;

    StagedArgs a{};
    fill_grad_ptrs(a.g, plan, rank_grads);
    fill_replica_ptrs(a.P, plan, rank_params);
    a.gs = scratch;
    a.gs_out = scratch;
    a.W = master;
    a.m = m;
    a.v = v;
    a.n = plan->N;
    a.S = plan->S;
    a.R = plan->R;
    a.M = plan->M;
    a.s = step_scalars(*hp, step, plan->R, plan->M);
    a.status = dev_status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool check = (flags & ZERO_FLAG_CHECK_FINITE) != 0;
    cudaError_t err = check ? launch_rs<true>(a, st) : launch_rs<false>(a, st);
    if (err == cudaSuccess) err = launch_adamw(a, st);
    if (err == cudaSuccess) err = launch_ag(a, st);
    return cuda_status(err);
}
