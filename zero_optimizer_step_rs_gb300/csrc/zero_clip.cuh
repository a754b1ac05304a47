// zero_clip.cuh - the step with global-norm clipping (zero_step_clipped).
// Part of the zero_step.cu translation unit: included at its end, it uses that
// file's scalars, device helpers, launch helpers and argument checks.

// =========================================== step with global-norm clipping ==
// zero_step_clipped: the averaged gradient of every element is stashed in
// fp32 scratch while its square feeds a fixed pairwise tree (fp32, leaves
// g*g, zero padding to a power of two); the update pass finishes the tree,
// turns the squared norm into the clip coefficient (and the skip decision for
// a non-finite norm), and applies it with the AdamW update and the R-way bf16
// all-gather: two launches.
//
// Tree decomposition.  The norm pass works in tiles of 2048 elements (256
// threads x 8) and takes them in groups of G consecutive tiles, G a power of
// two chosen from N alone so that there are at most 8192 groups; one block
// reduces a whole group (a block takes a run of consecutive groups), so every
// group is an aligned subtree of the global tree.  Inside a group each warp reduces its 256 leaves of a tile (a 3-level
// tree in registers, then 5 levels of shuffles) and leaves the partial in
// shared memory; every 32 tiles (or at the group's end) the block reduces
// those 256 partial slots, padded with zeros, and a group of more than 32
// tiles combines its rounds pairwise.  The update pass reduces the group
// partials, padded with zeros to 8192, again pairwise: each block redundantly,
// from L2, before its first element.  A zero (padding) leaf or subtree changes
// no value - the leaves are squares, so +0 or NaN, never -0 - and the root
// therefore equals the tree over the leaves padded to the next power of two,
// for any N and any grid.  No block ever waits for another, and the scratch
// holds no counter: any contents on entry.
namespace {

constexpr int kTreeLeaves = 2048;                 // elements per norm-pass tile (256 x 8)
constexpr int kWarpLeaves = 256;                  // leaves per warp and tile
constexpr int kRoundTiles = 32;                   // tiles per shared-memory round (256 slots)
constexpr int kMaxGroups = 8192;                  // group partials (256 threads x 32)

struct ClipCtl {
    double sumsq;          // squared norm (the fp32 tree value, widened)
    float coef;            // multiplier when clip != 0
    int32_t clip;          // 1: multiply the averaged gradients by coef
    int32_t skip;          // 1: non-finite norm and skipping requested
};

struct ClipLayout {
    int64_t g_off, part_off, total;
    int64_t tiles, group_tiles, groups;
};

int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

ClipLayout clip_layout(const zero_plan_t* plan)
{
    ClipLayout L{};
    L.tiles = (plan->N + kTreeLeaves - 1) / kTreeLeaves;
    if (L.tiles < 1) L.tiles = 1;
    L.group_tiles = 1;
    while ((L.tiles + L.group_tiles - 1) / L.group_tiles > kMaxGroups) L.group_tiles *= 2;
    L.groups = (L.tiles + L.group_tiles - 1) / L.group_tiles;
    L.g_off = 0;
    L.part_off = round256(4 * plan->padded);
    L.total = L.part_off + round256(4 * L.groups);
    return L;
}

// pairwise sum of 4 or 8 consecutive leaves (a perfect tree of 2 or 3 levels)
__device__ __forceinline__ float tree4(float a, float b, float c, float d)
{
    return __fadd_rn(__fadd_rn(a, b), __fadd_rn(c, d));
}

__device__ __forceinline__ float tree8(const float (&x)[8])
{
    return __fadd_rn(tree4(x[0], x[1], x[2], x[3]), tree4(x[4], x[5], x[6], x[7]));
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
        float w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = warp_sum[k];
        r = tree8(w);
    }
    __syncthreads();                   // warp_sum is reused by the next call
    return r;                          // thread 0 holds the block's subtree
}

struct ClipArgs {
    GradPtrs g;
    ReplicaPtrs P;
    float* gs;             // averaged gradients (padded floats; [0, N) used)
    float* part;           // one partial per group of group_tiles tiles
    int64_t tiles, group_tiles, groups;
    int64_t groups_per_block;   // the norm pass's blocks take consecutive runs of groups
    float* W;
    float* m;
    float* v;
    int64_t n;
    int32_t R, M;
    StepScalars s;
    float max_norm;
    int32_t skip_nonfinite;
    int32_t* status;
    double* sumsq_out;
};

// The squared norm into the clip coefficient (double, as clip_grad_norm_
// computes it) and the skip decision.
__device__ ClipCtl clip_control(const ClipArgs& a, float ss)
{
    const double norm = sqrt((double)ss);
    const double coef = (double)a.max_norm / (norm + 1e-6);
    ClipCtl c{};
    c.sumsq = (double)ss;
    c.clip = coef < 1.0 ? 1 : 0;
    c.coef = c.clip ? (float)coef : 1.0f;
    c.skip = (!isfinite(ss) && a.skip_nonfinite) ? 1 : 0;
    return c;
}

// pass 1: averaged gradient of 8 consecutive elements per thread, stashed,
// and the group's pairwise partial of their squares.  Every block takes the
// same number of consecutive groups (the last one fewer) and the grid is
// sized to it: the pass streams at a rate set by its active blocks, and on
// GB300 the 1B-shaped workload's 4,715 groups dealt round-robin to 760 blocks
// (7 rounds where 6.2 would do) took 4.53 ms against 3.70 for the earlier
// tile-by-tile pass; in runs of 6 groups over 786 blocks with 40 registers
// (6 blocks per SM; 5 at the unbounded 48) it takes 3.62 ms.  The generic
// (R, M) case runs 2 blocks per SM (128 registers, no spill); at 6 it
// spilled 380 bytes.
template <int RC, int MC>
__global__ void __launch_bounds__(kThreads, RC > 0 ? 6 : 2)
k_rs_norm(const __grid_constant__ ClipArgs a)
{
    __shared__ float slot[kRoundTiles * (kThreads / 32)];  // warp partials of one round
    pdl_enter();
    const int R = RC > 0 ? RC : a.R;
    const int M = MC > 0 ? MC : a.M;
    const int64_t n = a.n;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t GT = a.group_tiles;
    const int round_tiles = GT < kRoundTiles ? (int)GT : kRoundTiles;
    const int64_t g0 = (int64_t)blockIdx.x * a.groups_per_block;
    const int64_t g1 = g0 + a.groups_per_block < a.groups ? g0 + a.groups_per_block : a.groups;
    for (int64_t grp = g0; grp < g1; ++grp) {
        float stack[40];               // pairwise combination of the rounds (thread 0)
        int64_t rounds = 0;
        for (int64_t t0 = grp * GT; t0 < (grp + 1) * GT; t0 += round_tiles) {
            for (int j = 0; j < round_tiles; ++j) {
                const int64_t tile = t0 + j;
                float part = 0.0f;
                if (tile < a.tiles) {
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
                    for (int k = 0; k < 8; ++k) sq[k] = __fmul_rn(g[k], g[k]);  // padding: +0
                    part = warp_tree(tree8(sq));
                }
                if (lane == 0) slot[j * (kThreads / 32) + warp] = part;
            }
            __syncthreads();
            // the round's 256 slots, zero past round_tiles * 8: one per thread
            const int used = round_tiles * (kThreads / 32);
            const float v = block_tree((int)threadIdx.x < used ? slot[threadIdx.x] : 0.0f);
            if (threadIdx.x == 0) {    // push the round; merge equal-sized subtrees
                float x = v;
                int64_t c = rounds++;
                int top = __popcll(c);
                while (c & 1) {
                    x = __fadd_rn(stack[--top], x);
                    c >>= 1;
                }
                stack[top] = x;
            }
        }
        // rounds per group is 1 or a power of two: the stack holds one value
        if (threadIdx.x == 0) a.part[grp] = stack[0];
    }
}

// pass 2: the root of the tree over the group partials and the clip
// coefficient (every block, redundantly: 32 KB from L2 at most), then
// g' = g * coef (when clipping), AdamW, bf16 all-gather; tiles of 256 threads
// x 4 elements x kAgUnits units with every load of a tile issued first, as in
// k_fused.  This pass writes 28 of its 44 bytes per parameter, and
// write-heavy streams ran faster with more warps per SM: one unit at 8
// blocks per SM (32 registers, 56 bytes spilled to L1) measured 0.951 of the
// copy peak for the whole step against 0.947 for 4 units at 2 blocks per SM
// (114 registers); 1 unit at 4 or 6, 2 units at 4 and 4 units at 3 blocks
// per SM measured 0.942-0.948.  The replica tile staged in shared memory
// and written by R bulk copies (cp.async.bulk, one thread, double-buffered)
// measured 0.944 against 0.957 for the register stores.  The streaming cache
// hints stay: write-back stores for the replicas or for every store cost
// 0.3-3 %, and L2-only loads (ld.global.cg) 1-1.6 % on the uneven and
// 4B-shaped workloads.  8 consecutive elements a thread, taken as two
// 4-element halves to keep the registers of this loop, with one 16-byte
// store per replica (a third fewer store instructions) measured 0.74-0.78:
// each half's loads use every other 16 bytes of the lines they touch.  Lanes
// 2i and 2i+1 swapping their packed values by a shuffle, each then storing 8
// elements to half of the replicas (half the replica store instructions, the
// loads unchanged), measured the same as this within 0.2 %: the pass is bound
// by the DRAM's handling of its write-heavy mix, not by its store issue.
constexpr int kAgUnits = 1;

// Warp w reduces slots [1024 w, 1024 (w + 1)) of the 8192: lane l holds
// slots 128 q + 4 l .. + 3 of chunk q, so the lanes' shuffle tree spans the
// chunk's 128 consecutive slots, and the 8 chunks and then the 8 warps close
// the tree.  Slots past the last group are zero.
__device__ __forceinline__ float groups_root(const ClipArgs& a)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float c[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int64_t s = (int64_t)warp * 1024 + q * 128 + lane * 4;
        float4 x = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (s + 4 <= a.groups) {
            x = __ldcg(reinterpret_cast<const float4*>(a.part + s));
        } else if (s < a.groups) {
            x.x = __ldcg(a.part + s);
            if (s + 1 < a.groups) x.y = __ldcg(a.part + s + 1);
            if (s + 2 < a.groups) x.z = __ldcg(a.part + s + 2);
        }
        c[q] = warp_tree(tree4(x.x, x.y, x.z, x.w));
    }
    __shared__ float warp_sum[kThreads / 32];
    if (lane == 0) warp_sum[warp] = tree8(c);
    __syncthreads();
    float r = 0.0f;
    if (threadIdx.x == 0) {
        float w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = warp_sum[k];
        r = tree8(w);
    }
    return r;                          // thread 0 holds the root
}

template <int RC>
__global__ void __launch_bounds__(kThreads, 8) k_adamw_ag(const __grid_constant__ ClipArgs a)
{
    __shared__ ClipCtl ctl;
    pdl_enter();
    const float ss = groups_root(a);
    if (threadIdx.x == 0) {
        ctl = clip_control(a, ss);
        if (blockIdx.x == 0) {
            if (a.status) {
                if (!isfinite(ss)) atomicOr(a.status, ZERO_DEV_NONFINITE);
                if (ctl.skip) atomicOr(a.status, ZERO_DEV_SKIPPED);
            }
            if (a.sumsq_out) *a.sumsq_out = ctl.sumsq;
        }
    }
    __syncthreads();
    const ClipCtl c = ctl;
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
    const int64_t cap = grid_for(k, a.groups);
    ClipArgs b = a;
    b.groups_per_block = (a.groups + cap - 1) / cap;
    const int64_t grid = (a.groups + b.groups_per_block - 1) / b.groups_per_block;
    return launch_pdl(k_rs_norm<RC, MC>, dim3((unsigned)grid), kThreads, st, b);
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
    a.part = reinterpret_cast<float*>(base + L.part_off);
    a.tiles = L.tiles;
    a.group_tiles = L.group_tiles;
    a.groups = L.groups;
    a.max_norm = max_norm;
    a.skip_nonfinite = (flags & ZERO_FLAG_SKIP_NONFINITE) ? 1 : 0;
    a.status = dev_status;
    a.sumsq_out = dev_sumsq;
    a.W = master;
    a.m = m;
    a.v = v;
    a.n = plan->N;
    a.R = plan->R;
    a.M = plan->M;
    a.s = step_scalars(*hp, step, plan->R, plan->M);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    cudaError_t err = launch_rs_norm(a, st);
    if (err == cudaSuccess) err = launch_adamw_ag(a, st);
    return cuda_status(err);
}
