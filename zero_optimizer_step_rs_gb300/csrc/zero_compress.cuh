// zero_compress.cuh - the step with a compressed reduce-scatter
// (zero_step_compressed).  Part of the zero_step.cu translation unit: included
// at its end, it uses that file's scalars, device helpers, launch helpers and
// argument checks.

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
// (rint(RN(x * rc)) alone decides every quotient more than 2^-13 from a
// half-integer; taking it, with a warp vote per rank sending the rest to
// quot_by_recip, ran fewer instructions but measured 0.933 against 0.957 of
// the copy peak on the 1B-shaped workload: the votes serialise the ranks.)
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
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float4 w4, m4, v4;                        // the owner's state of a full block
        bool have_state = false;
        // every rank's loads first, then the codecs and their warp reductions,
        // so the loads are all in flight before the first sync.  Whether the
        // owner's state joins them was measured per codec: it does for int8
        // without error feedback while R*M <= 16 (0.86 -> 0.96 of peak at R=8,
        // M=1; at R=7, M=4 it would cost 0.97 -> 0.90), and slows the others.
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
                    if constexpr (RC * MC <= 16) {
                        w4 = ld_stream(a.W + e);
                        m4 = ld_stream(a.m + e);
                        v4 = ld_stream(a.v + e);
                        have_state = true;
                    }
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
    return launch_pdl(k_comp<RC, MC, KIND, EF>, dim3(grid_for(k, work < 1 ? 1 : work, quarters)),
                      kThreads, st, a);
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
