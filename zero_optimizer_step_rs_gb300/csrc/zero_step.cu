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

#include <algorithm>
#include <climits>
#include <utility>
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
    uint16_t* g_lo;       // or, when set, the gradient kept in two gradient buffers:
    uint16_t* g_hi;       // the low and high 16 bits of each element's fp32 value
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

// Programmatic dependent launch.  The kernels of a step are launched with
// programmatic stream serialization: the next such launch on the stream may
// be scheduled while the kernel before it still runs, which hides the launch
// gap between back-to-back steps (and between the kernels of a step).  Every
// kernel launched this way first allows its own dependent to launch, then
// waits until the grid before it has completed and its writes are visible,
// before touching memory.  A launch that follows anything other than such a
// kernel (a copy, an event, another library's kernel) waits as usual.
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------ launch helpers --

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, int threads, cudaStream_t st,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

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

int blocks_per_sm(int dev, const void* kernel, int threads = kThreads)
{
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo& d = g_dev[dev & 63];
    auto it = d.occ.find(kernel);
    if (it != d.occ.end()) return it->second;
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, 0) != cudaSuccess ||
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
unsigned grid_for(const void* kernel, int64_t work_blocks, int quarter_blocks = 0,
                  int threads = kThreads)
{
    int dev = 0;
    cudaGetDevice(&dev);
    int64_t cap = (int64_t)device_sms(dev) * blocks_per_sm(dev, kernel, threads);
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
template <int RC, int MC, int U, bool CHECK, int OUT, int TPB = kThreads>
__global__ void __launch_bounds__(TPB) k_fused(const __grid_constant__ FusedArgs a)
{
    pdl_enter();
    const int R = RC > 0 ? RC : a.R;
    const int M = MC > 0 ? MC : a.M;
    constexpr int kU = TPB * kVec;             // elements per block per unit
    constexpr int T = kU * U;
    const int64_t n = a.n;
    const int64_t full_tiles = n / T;
    bool bad = false;

    for (int64_t tile = blockIdx.x; tile < full_tiles; tile += gridDim.x) {
        const int64_t e0 = tile * T + (int64_t)threadIdx.x * kVec;
        float acc[U][4];
        float4 w[U], mm[U], vv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t e = e0 + (int64_t)u * kU;
            w[u] = ld_stream(a.W + e);
            mm[u] = ld_stream(a.m + e);
            vv[u] = ld_stream(a.v + e);
            grad_sum4<RC, MC>(a.g, R, M, e, acc[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t e = e0 + (int64_t)u * kU;
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
        for (int64_t i = tail0 + threadIdx.x; i < n; i += TPB) {
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

// A vector too short to give every resident block of the full-size tiling a
// tile (fewer than one wave) leaves SMs idle, and its step is bound by
// latency, not bandwidth: it takes tiles of one unit instead, spread over
// twice the blocks.  On GB300 the tiny 65,536-element workload then runs
// 4.1 us a step back to back (6.2 with two-unit tiles); 64- and 128-thread
// blocks measured the same.
constexpr int kSmallThreads = 256;
constexpr int kSmallUnits = 1;

template <int RC, int MC, bool CHECK, int OUT = 0>
cudaError_t launch_fused_t(const FusedArgs& a, cudaStream_t st)
{
    constexpr int U = 2;
    const void* k = reinterpret_cast<const void*>(&k_fused<RC, MC, U, CHECK, OUT>);
    const int64_t tiles = (a.n + kUnit * U - 1) / (kUnit * U);
    int dev = 0;
    cudaGetDevice(&dev);
    if (tiles < (int64_t)device_sms(dev) * blocks_per_sm(dev, k)) {
        constexpr int TS = kSmallThreads, US = kSmallUnits;
        const void* ks = reinterpret_cast<const void*>(&k_fused<RC, MC, US, CHECK, OUT, TS>);
        const int64_t small_tiles = (a.n + TS * kVec * US - 1) / (TS * kVec * US);
        const unsigned grid = grid_for(ks, small_tiles, 0, TS);
        return launch_pdl(k_fused<RC, MC, US, CHECK, OUT, TS>, dim3(grid), TS, st, a);
    }
    const unsigned grid = grid_for(k, tiles, fused_quarter_blocks<RC, MC, OUT>());
    return launch_pdl(k_fused<RC, MC, U, CHECK, OUT>, dim3(grid), kThreads, st, a);
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
    pdl_enter();
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
            const int64_t e = e0 + (int64_t)u * kUnit;
            if (a.g_lo) {
                // every gradient of these elements has been read above: their
                // slots in buffers 0 and 1 are free to hold the result
                const uint32_t b0 = __float_as_uint(o.x), b1 = __float_as_uint(o.y);
                const uint32_t b2 = __float_as_uint(o.z), b3 = __float_as_uint(o.w);
                st_stream(a.g_lo + e, make_uint2(__byte_perm(b0, b1, 0x5410),
                                                 __byte_perm(b2, b3, 0x5410)));
                st_stream(a.g_hi + e, make_uint2(__byte_perm(b0, b1, 0x7632),
                                                 __byte_perm(b2, b3, 0x7632)));
            } else {
                st_stream(a.gs_out + e, o);
            }
        }
    }
    // the shard's last partial tile, element by element, by the block that owns it
    const int64_t tail0 = lo + full_tiles * T;
    if (tail0 < lo + len && blockIdx.x == (unsigned)(full_tiles % gridDim.x)) {
        for (int64_t i = tail0 + threadIdx.x; i < lo + len; i += kThreads) {
            const float g = scale_grad(a.s, grad_sum1(a.g, R, M, i));
            if (CHECK) bad |= !isfinite(g);
            if (a.g_lo) {
                a.g_lo[i] = (uint16_t)(__float_as_uint(g) & 0xFFFFu);
                a.g_hi[i] = (uint16_t)(__float_as_uint(g) >> 16);
            } else {
                a.gs_out[i] = g;
            }
        }
    }
    report_nonfinite<CHECK>(bad, a.status);
}

// SPLIT: the gradient comes as low and high halves from gradient buffers 0
// and 1 (ZeRO-2 without scratch) instead of from the fp32 scratch
template <bool SPLIT>
__global__ void __launch_bounds__(kThreads) k_adamw(const __grid_constant__ StagedArgs a)
{
    pdl_enter();
    const int r = blockIdx.y;
    const int64_t lo = (int64_t)r * a.S, len = shard_len(a.n, a.S, r);
    const int64_t nvec = len / kVec;
    for (int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x; q < nvec;
         q += (int64_t)gridDim.x * kThreads) {
        const int64_t e = lo + q * kVec;
        float4 g;
        if constexpr (SPLIT) {
            const uint2 l = ld_stream(a.g_lo + e), h = ld_stream(a.g_hi + e);
            g = make_float4(__uint_as_float(__byte_perm(l.x, h.x, 0x5410)),
                            __uint_as_float(__byte_perm(l.x, h.x, 0x7632)),
                            __uint_as_float(__byte_perm(l.y, h.y, 0x5410)),
                            __uint_as_float(__byte_perm(l.y, h.y, 0x7632)));
        } else {
            g = ld_stream(a.gs + e);
        }
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
            float g;
            if constexpr (SPLIT)
                g = __uint_as_float((uint32_t)a.g_lo[i] | ((uint32_t)a.g_hi[i] << 16));
            else
                g = a.gs[i];
            adamw(a.s, g, w, m, v);
            a.W[i] = w;
            a.m[i] = m;
            a.v[i] = v;
        }
    }
}

template <int RC, int VPT>
__global__ void __launch_bounds__(kThreads) k_ag_cast(const __grid_constant__ StagedArgs a)
{
    // VPT vectors of 8 elements per thread per iteration, blockDim vectors
    // apart (each warp instruction stays contiguous): two float4 loads of W
    // and one 16-byte store per replica each, every load issued first.  A
    // shard starts on a multiple of 4 elements only, so the vector loop
    // starts at the shard's first multiple of 8; the head before it and the
    // tail after the last full vector are done element by element.
    pdl_enter();
    const int R = RC > 0 ? RC : a.R;
    const int r = blockIdx.y;
    const int64_t lo = (int64_t)r * a.S, len = shard_len(a.n, a.S, r);
    const int64_t hi = lo + len;
    const int64_t v0 = (lo + 7) / 8 * 8;                  // first 8-aligned element
    const int64_t n8 = hi > v0 ? (hi - v0) / 8 : 0;
    for (int64_t q0 = (int64_t)blockIdx.x * kThreads * VPT + threadIdx.x; q0 < n8;
         q0 += (int64_t)gridDim.x * kThreads * VPT) {
        float4 w0[VPT], w1[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int64_t q = q0 + (int64_t)j * kThreads;
            if (q < n8) {
                w0[j] = ld_stream(a.W + v0 + q * 8);
                w1[j] = ld_stream(a.W + v0 + q * 8 + 4);
            }
        }
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int64_t q = q0 + (int64_t)j * kThreads;
            if (q >= n8) break;
            const int64_t e = v0 + q * 8;
            const uint4 p = make_uint4(pack_bf16x2(w0[j].x, w0[j].y), pack_bf16x2(w0[j].z, w0[j].w),
                                       pack_bf16x2(w1[j].x, w1[j].y), pack_bf16x2(w1[j].z, w1[j].w));
            if constexpr (RC > 0) {
#pragma unroll
                for (int k = 0; k < RC; ++k) __stcs(reinterpret_cast<uint4*>(a.P.p[k] + e), p);
            } else {
                for (int k = 0; k < R; ++k) __stcs(reinterpret_cast<uint4*>(a.P.p[k] + e), p);
            }
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
        return launch_pdl(kern, grid, kThreads, st, a);
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
    const int64_t work = (a.S / kVec + kThreads - 1) / kThreads;
    auto go = [&](auto kern) {
        const void* k = reinterpret_cast<const void*>(kern);
        const int64_t per_rank = (int64_t)grid_for(k, work * a.R) / a.R;    // never past one wave
        dim3 grid((unsigned)(per_rank < 1 ? 1 : per_rank), (unsigned)a.R);
        return launch_pdl(kern, grid, kThreads, st, a);
    };
    return a.g_lo ? go(k_adamw<true>) : go(k_adamw<false>);
}

// Vectors of 8 elements per thread per iteration, and the grid cap in quarter
// blocks per SM (0: every resident block).  2 vectors, and 2, 3 or 4 blocks
// per SM, measured within 0.5 % of this on the GPT-2, 1B and uneven staged
// steps.  On the uneven workload the kernel takes 306 us at its 4 resident
// blocks per SM (58 registers); bounded to 6 or 8 blocks per SM it took 308
// and 314 us, and 4 elements per thread with 8-byte stores at 8 blocks 359.
constexpr int kAgVecs = 1;
constexpr int kAgQuarterBlocks = 0;

cudaError_t launch_ag(const StagedArgs& a, cudaStream_t st)
{
    const int64_t work = (a.S / 8 + kThreads * kAgVecs - 1) / (kThreads * kAgVecs);
    auto go = [&](const void* k, auto kern) {
        const int64_t per_rank =
            (int64_t)grid_for(k, work * a.R, kAgQuarterBlocks) / a.R;    // never past one wave
        dim3 grid((unsigned)(per_rank < 1 ? 1 : per_rank), (unsigned)a.R);
        return launch_pdl(kern, grid, kThreads, st, a);
    };
#define ZERO_AG(r_) \
    return go(reinterpret_cast<const void*>(&k_ag_cast<r_, kAgVecs>), k_ag_cast<r_, kAgVecs>);
    switch (a.R) {
    case 8: ZERO_AG(8)
    case 7: ZERO_AG(7)
    case 4: ZERO_AG(4)
    case 2: ZERO_AG(2)
    default: ZERO_AG(0)
    }
#undef ZERO_AG
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
    std::sort(r, r + n, [](const Range& x, const Range& y) { return x.lo < y.lo; });
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
    // ZeRO-2 gives up the gradients once they are reduced: without scratch the
    // staged step keeps the reduced gradient in gradient buffers 0 and 1
    const bool in_grads = variant == ZERO_VARIANT_STAGED && !scratch && plan->stage == 2 &&
                          plan->R * plan->M >= 2;
    if (in_grads) {
        rs[0].out = rs[1].out = true;          // written: they may alias nothing
    } else if (variant == ZERO_VARIANT_STAGED) {
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
    if (in_grads) {
        a.g_lo = const_cast<uint16_t*>(rank_grads[0]);
        a.g_hi = const_cast<uint16_t*>(rank_grads[1]);
    }
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

extern "C" zero_status zero_get_device_status(const int32_t* dev_status, void* stream,
                                              int32_t* out)
{
    if (!dev_status) return ZERO_ERR_NULL;
    if ((uintptr_t)dev_status & 3u) return ZERO_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t word = 0;
    // ordered after the steps on `stream`; then wait for the stream to finish
    if (cudaMemcpyAsync(&word, dev_status, sizeof word, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return ZERO_ERR_CUDA;
    }
    if (out) *out = word;
    if (word & ZERO_DEV_TIMEOUT) return ZERO_ERR_DEVICE_TIMEOUT;
    if (word & ZERO_DEV_NONFINITE) return ZERO_ERR_NONFINITE;
    return ZERO_OK;
}

// The variants and the other entry points, in files of their own (one translation unit).
#include "zero_clip.cuh"
#include "zero_compress.cuh"
#include "zero_onebit.cuh"
#include "zero_tma.cuh"
#include "zero_check.cuh"
#include "zero3.cuh"

// ================================================ staged step, no allocation ==
// zero_step_staged_noalloc: the staged trio with its fp32 reduced-gradient
// scratch in a fixed device array of this file instead of a caller buffer,
// for callers that cannot allocate device memory.  The array's address is a
// device address only on the device side; host code looks it up once per
// device with cudaGetSymbolAddress (with that device current; again after
// the device's context has been replaced) and passes it to the kernels like
// any other scratch pointer.
namespace {

static __device__ __align__(256) float g_noalloc_scratch[ZERO_NOALLOC_MAX_ELEMS];

std::mutex g_noalloc_mu;
struct NoallocAddr {
    const void* ctx;                      // the context the address was looked up in
    float* addr;
};
NoallocAddr g_noalloc_addr[64] = {};      // per device ordinal

// The current context's handle, through the driver entry point the runtime
// hands out (no link to the driver library is needed).  A device reset
// replaces the primary context and may place the array elsewhere, so the
// cached address is only reused in the context it was looked up in.
const void* current_context()
{
    using GetCtx = int (*)(void**);
    static GetCtx fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<GetCtx>(f);
    }();
    void* ctx = nullptr;
    if (!fn || fn(&ctx) != 0) return nullptr;
    return ctx;
}

// The array's device address for the current device, looked up once per
// device (and again after the device's context has been replaced).
zero_status noalloc_scratch(float** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ZERO_ERR_CUDA;
    const void* ctx = current_context();
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoallocAddr& slot = g_noalloc_addr[dev];
    if (!slot.addr || !ctx || slot.ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();            // clear it so later launch checks do not see it
            return ZERO_ERR_CUDA;
        }
        slot.addr = static_cast<float*>(p);
        slot.ctx = current_context();      // the lookup has made the device's context current
    }
    *out = slot.addr;
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

    // the array's address belongs to the current device: the stream must too
    int dev = -1, sdev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ZERO_ERR_CUDA;
    if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
        cudaGetLastError();
        return ZERO_ERR_INVALID_ARG;
    }
    if (sdev != dev) return ZERO_ERR_INVALID_ARG;
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
