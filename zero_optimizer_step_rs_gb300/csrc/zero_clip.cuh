// zero_clip.cuh - the step with global-norm clipping (zero_step_clipped).
// Part of the zero_step.cu translation unit: included at its end, it uses that
// file's scalars, device helpers, launch helpers and argument checks.

// =========================================== step with global-norm clipping ==
// zero_step_clipped: the averaged gradient of every element is stashed in
// fp32 scratch while its square feeds a fixed pairwise tree (fp32, leaves
// g*g, zero padding to a power of two); a small second kernel finishes the
// tree and turns the squared norm into the clip coefficient (and the skip
// decision for a non-finite norm), and a last pass applies it with the AdamW
// update and the R-way bf16 all-gather: three launches.
//
// Tree decomposition: in the streaming pass each warp reduces 256
// consecutive leaves (32 lanes x 8 leaves: a 3-level tree in registers, then
// 5 levels of shuffles) - exactly an aligned subtree of the global tree - and
// writes one partial, with no block-wide barrier; each further level is a
// block reducing 2048 partials (8 per thread, the warp levels, then 3 levels
// across the 8 warps), again an aligned subtree.  Adding a zero (padding)
// changes no value, so the root equals the tree over the leaves padded to
// the next power of two for any N and any grid.
//
// The levels above the first are finished in one launch with arrival
// tickets, without any wait: the blocks reduce the groups of 2048 first-level
// partials; a block that has written its group's sum makes it visible
// (__threadfence) and takes a ticket on the counter of its group one level
// up, and the block that draws that group's last ticket reduces it in turn;
// the block that completes the root computes the coefficient.  No block ever
// waits for another.  The counters are zeroed by the streaming pass, which
// the tree launch follows in stream order.
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
    int64_t g_off, ctl_off, cnt_off, cnt_bytes, total;
    int levels;
    int64_t lvl_off[8], lvl_len[8];
    int64_t cnt_base[8];   // first counter of level k >= 2 (index into the counter array)
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
    L.cnt_off = off + round256((int64_t)sizeof(ClipCtl));
    int64_t cnt = 0;                              // one counter per group above level 1
    for (int k = 2; k < L.levels; ++k) {
        L.cnt_base[k] = cnt;
        cnt += L.lvl_len[k];
    }
    L.cnt_bytes = 4 * cnt;
    L.total = L.cnt_off + round256(L.cnt_bytes);
    return L;
}

// pairwise sum of 8 consecutive leaves (a perfect tree of 3 levels)
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
    v = warp_tree(v);
    if (lane == 0) warp_sum[warp] = v;
    __syncthreads();
    float r = 0.0f;
    if (threadIdx.x == 0) {
        const float* w = warp_sum;
        r = __fadd_rn(__fadd_rn(__fadd_rn(w[0], w[1]), __fadd_rn(w[2], w[3])),
                      __fadd_rn(__fadd_rn(w[4], w[5]), __fadd_rn(w[6], w[7])));
    }
    __syncthreads();                   // warp_sum is reused by the next group
    return r;                          // thread 0 holds the block's subtree
}

struct ClipArgs {
    GradPtrs g;
    ReplicaPtrs P;
    float* gs;             // averaged gradients (padded floats; [0, N) used)
    float* lvl[8];         // tree levels: level 0 has one partial per 256 elements (per warp)
    int64_t lvl_len[8];
    uint32_t* cnt[8];      // arrival counters of the groups of level k >= 2
    uint32_t* cnt_all;     // all counters, zeroed by the streaming pass
    int64_t n_cnt;
    int32_t levels;
    float* W;
    float* m;
    float* v;
    ClipCtl* ctl;
    int64_t n;
    int32_t R, M;
    StepScalars s;
    float max_norm;
    int32_t skip_nonfinite;
    int32_t* status;
    double* sumsq_out;
};

// The squared norm into the clip coefficient (double, as clip_grad_norm_
// computes it) and the skip decision, by the one thread that holds the root.
__device__ void clip_finish(const ClipArgs& a, float ss)
{
    const double norm = sqrt((double)ss);
    const double coef = (double)a.max_norm / (norm + 1e-6);
    ClipCtl c{};
    c.sumsq = (double)ss;
    c.clip = coef < 1.0 ? 1 : 0;
    c.coef = c.clip ? (float)coef : 1.0f;
    const bool finite = isfinite(ss);
    c.skip = (!finite && a.skip_nonfinite) ? 1 : 0;
    *a.ctl = c;
    if (a.status) {
        if (!finite) atomicOr(a.status, ZERO_DEV_NONFINITE);
        if (c.skip) atomicOr(a.status, ZERO_DEV_SKIPPED);
    }
    if (a.sumsq_out) *a.sumsq_out = c.sumsq;
}

// sum of group b of level k - 1 (at most 2048 partials, read from L2: other
// blocks wrote them) into partial b of level k; the value in thread 0
__device__ __forceinline__ float reduce_group(const ClipArgs& a, int k, int64_t b)
{
    const int64_t lo = b * kTreeLeaves;
    const int64_t n_in = a.lvl_len[k - 1];
    const float* in = a.lvl[k - 1];
    const int64_t e = lo + (int64_t)threadIdx.x * 8;
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = e + j < n_in ? __ldcg(in + e + j) : 0.0f;
    const float v = block_tree(tree8(x));
    if (threadIdx.x == 0) a.lvl[k][b] = v;
    return v;
}

// the levels above the first, then the coefficient: one launch
__global__ void __launch_bounds__(kThreads) k_norm_tree(const __grid_constant__ ClipArgs a)
{
    __shared__ uint32_t last;
    pdl_enter();
    if (a.levels == 1) {                           // a single first-level partial is the root
        if (blockIdx.x == 0 && threadIdx.x == 0) clip_finish(a, a.lvl[0][0]);
        return;
    }
    for (int64_t g = blockIdx.x; g < a.lvl_len[1]; g += gridDim.x) {
        float v = reduce_group(a, 1, g);
        int64_t idx = g;
        int k = 2;
        for (; k < a.levels; ++k) {                // climb while this block is the last arrival
            const int64_t b = idx / kTreeLeaves;
            const int64_t n_in = a.lvl_len[k - 1] - b * kTreeLeaves;
            const uint32_t expect = (uint32_t)(n_in < kTreeLeaves ? n_in : kTreeLeaves);
            if (threadIdx.x == 0) {
                __threadfence();                   // partial idx of level k - 1, before the ticket
                last = atomicAdd(&a.cnt[k][b], 1u) == expect - 1;
            }
            __syncthreads();
            const bool mine = last;
            __syncthreads();                       // `last` is reused at the next level
            if (!mine) break;
            __threadfence();                       // the group's partials, after the tickets
            v = reduce_group(a, k, b);
            idx = b;
        }
        if (k == a.levels && threadIdx.x == 0) clip_finish(a, v);
    }
}

// pass 1: averaged gradient of 8 consecutive elements per thread, stashed,
// and the tile's pairwise partial of their squares
template <int RC, int MC>
__global__ void __launch_bounds__(kThreads) k_rs_norm(const __grid_constant__ ClipArgs a)
{
    pdl_enter();
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
        if ((threadIdx.x & 31) == 0 && wpart * kWarpLeaves < n) a.lvl[0][wpart] = part;
    }
    // the tree launch that follows takes tickets on these counters
    if (blockIdx.x == 0)
        for (int64_t i = threadIdx.x; i < a.n_cnt; i += kThreads) a.cnt_all[i] = 0u;
}

// pass 2: g' = g * coef (when clipping), AdamW, bf16 all-gather; tiles of
// 256 threads x 4 elements x kAgUnits units with every load of a tile issued
// first, as in k_fused.  This pass writes 28 of its 44 bytes per parameter,
// and write-heavy streams ran faster with more warps per SM: one unit at 8
// blocks per SM (32 registers, 56 bytes spilled to L1) measured 0.951 of the
// copy peak for the whole step against 0.947 for 4 units at 2 blocks per SM
// (114 registers); 1 unit at 4 or 6, 2 units at 4 and 4 units at 3 blocks
// per SM measured 0.942-0.948.
constexpr int kAgUnits = 1;
template <int RC>
__global__ void __launch_bounds__(kThreads, 8) k_adamw_ag(const __grid_constant__ ClipArgs a)
{
    pdl_enter();
    const ClipCtl c = *a.ctl;
    if (c.skip) return;
    const int R = RC > 0 ? RC : a.R;
    constexpr int U = kAgUnits;
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
    return launch_pdl(k_rs_norm<RC, MC>, dim3(grid_for(k, tiles)), kThreads, st, a);
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
    const int64_t work = (a.n + kAgUnits * kUnit - 1) / (kAgUnits * kUnit);
    auto go = [&](const void* k, auto kern) {
        return launch_pdl(kern, dim3(grid_for(k, work < 1 ? 1 : work)), kThreads, st, a);
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
    uint32_t* counters = reinterpret_cast<uint32_t*>(base + L.cnt_off);
    a.levels = L.levels;
    for (int k = 0; k < L.levels; ++k) {
        a.lvl[k] = reinterpret_cast<float*>(base + L.lvl_off[k]);
        a.lvl_len[k] = L.lvl_len[k];
        a.cnt[k] = k >= 2 ? counters + L.cnt_base[k] : nullptr;
    }
    a.cnt_all = counters;
    a.n_cnt = L.cnt_bytes / 4;
    a.max_norm = max_norm;
    a.skip_nonfinite = (flags & ZERO_FLAG_SKIP_NONFINITE) ? 1 : 0;
    a.status = dev_status;
    a.sumsq_out = dev_sumsq;
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
    if (err == cudaSuccess) {
        const void* k = reinterpret_cast<const void*>(&k_norm_tree);
        err = launch_pdl(k_norm_tree, dim3(L.levels > 1 ? grid_for(k, L.lvl_len[1]) : 1),
                         kThreads, st, a);
    }
    if (err == cudaSuccess) err = launch_adamw_ag(a, st);
    return cuda_status(err);
}
