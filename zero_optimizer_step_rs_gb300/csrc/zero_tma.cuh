// zero_tma.cuh - the fused step with TMA bulk staging
// (ZERO_VARIANT_FUSED_TMA).  Part of the zero_step.cu translation unit:
// included at its end, it uses that file's scalars, device helpers, launch
// helpers and argument checks.

// ============================================== fused step, TMA bulk staging ==
// k_fused_tma: the fused step with the R*M gradient tiles and the three
// state tiles of each 1024-element tile brought into shared memory by
// cp.async.bulk (one elected thread, completion on an mbarrier, 3 stages
// in flight per block) and the replica tile written back by R bulk stores
// from a double-buffered shared tile.  Same arithmetic as k_fused, same bits.
// (Replicas stored from registers instead, as k_fused does, measured 0.904
// against 0.971 of the copy peak on the 1B-shaped workload: with its 2
// blocks per SM this kernel keeps its stores in the bulk copies.)
// On this access pattern it measures a few percent below the register-
// direct k_fused, which stays the default; it is the selectable variant
// ZERO_VARIANT_FUSED_TMA.
//
// Every mbarrier wait is bounded.  When a wait runs out, the whole block
// (the decision is block-uniform) stops, thread 0 waits - again bounded -
// for the stage loads it has issued and not consumed, and for its bulk
// stores, sets ZERO_DEV_TIMEOUT in the status word and the block returns, so
// no copy can land in shared memory after the block has left.  If that
// drain runs out as well, ZERO_DEV_DRAIN_FAILED is set beside it: the block
// has left with copies in flight and the context is suspect.
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
    pdl_enter();
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
            bool drained = true;
            for (int64_t kk = k_fail; kk < k_fail + kTmaStages && kk < my; ++kk)
                drained &= mbar_wait(&full[kk % kTmaStages], (uint32_t)((kk / kTmaStages) & 1),
                                     kDrainLimit);
            // copies may still land in this block's shared memory after it leaves
            if (!drained && a.status) atomicOr(a.status, ZERO_DEV_DRAIN_FAILED);
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
    // programmatic dependent launch, as the other step kernels (dynamic shared memory here)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L.smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_fused_tma, a, expire_waits ? 0u : kWaitLimit,
                              (int32_t)(check ? 1 : 0));
}

}  // namespace
