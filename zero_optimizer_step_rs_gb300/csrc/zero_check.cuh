// zero_check.cuh - the replica-consistency check (zero_check_replicas).  Part
// of the zero_step.cu translation unit: included at its end, it uses that
// file's scalars, device helpers, launch helpers and argument checks.

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
