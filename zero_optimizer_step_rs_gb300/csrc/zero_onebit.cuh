// zero_onebit.cuh - 1-bit Adam with a frozen variance (zero_step_onebit).
// Part of the zero_step.cu translation unit: included at its end, it uses that
// file's scalars, device helpers, launch helpers and argument checks.

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
    pdl_enter();
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
    return launch_pdl(k_onebit<RC, MC>, dim3(grid_for(k, work < 1 ? 1 : work)), kThreads, st, a);
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
