// plan.cpp - host-side shard layout and byte accounting (zero_plan_*).
//
// Layout: the tensors are concatenated in the given order into one flat
// vector of N elements; shard length S = roundup(ceil(N/R), align); rank r
// owns [r*S, min((r+1)*S, N)).  The state arrays hold R*S floats so that
// every shard starts on an aligned offset; the pad [N, R*S) is never read
// or written.  (CS25 V6 Lecture 4 notes, "ZeRO-1": each rank owns a part of
// the optimizer state and updates only its parameter shard.)
//
// Accounting per rank: CS25 V6 Lecture 4 notes, M_DP, M_Z1 and M_Z2
// equations; M_Z3 from CS324 Lecture 9 notes, exercise 1.  The sharded
// parts are counted with the padded shard length S.
#include <cstdlib>
#include <cstring>
#include <new>

#include "zero_step.h"

namespace {

struct PlanStorage {
    zero_plan_t pub;
    int64_t* offsets;
};

bool mul_overflows(int64_t a, int64_t b) { return a != 0 && b > INT64_MAX / a; }

}  // namespace

extern "C" int32_t zero_abi_version(void) { return ZERO_ABI_VERSION; }

extern "C" const char* zero_status_string(zero_status s)
{
    switch (s) {
    case ZERO_OK: return "ok";
    case ZERO_ERR_INVALID_ARG: return "invalid argument";
    case ZERO_ERR_NULL: return "null pointer";
    case ZERO_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case ZERO_ERR_SIZE: return "size out of range or scratch too small";
    case ZERO_ERR_OVERLAP: return "output buffer overlaps another buffer";
    case ZERO_ERR_CUDA: return "CUDA launch or copy failed";
    case ZERO_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case ZERO_ERR_NONFINITE: return "non-finite gradient";
    case ZERO_ERR_IO: return "checkpoint file could not be written or read";
    case ZERO_ERR_CORRUPT: return "checkpoint header or checksum is wrong";
    }
    return "unknown status";
}

extern "C" zero_status zero_plan_create(const int64_t* tensor_numels, int32_t n_tensors,
                                        int32_t R, int32_t M, int32_t stage,
                                        int32_t align_elems, zero_plan_t** out)
{
    if (!out) return ZERO_ERR_NULL;
    *out = nullptr;
    if (n_tensors < 0) return ZERO_ERR_INVALID_ARG;
    if (n_tensors > 0 && !tensor_numels) return ZERO_ERR_NULL;
    if (R < 1 || R > ZERO_MAX_R || M < 1 || (int64_t)R * M > ZERO_MAX_RM)
        return ZERO_ERR_INVALID_ARG;
    if (stage != 1 && stage != 2) return ZERO_ERR_INVALID_ARG;
    if (align_elems == 0) align_elems = 64;
    if (align_elems < 0 || align_elems % 4 != 0 || align_elems > (1 << 24))
        return ZERO_ERR_INVALID_ARG;

    int64_t N = 0;
    for (int32_t k = 0; k < n_tensors; ++k) {
        if (tensor_numels[k] < 0) return ZERO_ERR_INVALID_ARG;
        if (tensor_numels[k] > INT64_MAX / 64 - N) return ZERO_ERR_SIZE;
        N += tensor_numels[k];
    }
    const int64_t per = (N + R - 1) / R;
    const int64_t S = (per + align_elems - 1) / align_elems * align_elems;
    if (mul_overflows(S, R) || mul_overflows(S * R, 16)) return ZERO_ERR_SIZE;

    auto* ps = new (std::nothrow) PlanStorage();
    if (!ps) return ZERO_ERR_SIZE;
    ps->offsets = static_cast<int64_t*>(std::malloc(sizeof(int64_t) * (size_t)(n_tensors + 1)));
    if (!ps->offsets) { delete ps; return ZERO_ERR_SIZE; }
    ps->offsets[0] = 0;
    for (int32_t k = 0; k < n_tensors; ++k) ps->offsets[k + 1] = ps->offsets[k] + tensor_numels[k];

    zero_plan_t& p = ps->pub;
    std::memset(&p, 0, sizeof(p));
    p.N = N;
    p.S = S;
    p.padded = S * R;
    p.R = R;
    p.M = M;
    p.stage = stage;
    p.align_elems = align_elems;
    p.n_tensors = n_tensors;
    p.tensor_offsets = ps->offsets;
    const int64_t bp = 2, bg = 2, bo = 12;
    p.bytes_per_rank_dp = N * (bp + bg + bo);
    p.bytes_per_rank_z1 = N * (bp + bg) + S * bo;
    p.bytes_per_rank_z2 = N * bp + S * (bg + bo);
    p.bytes_per_rank_z3 = S * (bp + bg + bo);
    p.bytes_per_rank = stage == 1 ? p.bytes_per_rank_z1 : p.bytes_per_rank_z2;
    p.scratch_bytes_staged = 4 * S * R;
    *out = &p;
    return ZERO_OK;
}

extern "C" void zero_plan_destroy(zero_plan_t* plan)
{
    if (!plan) return;
    auto* ps = reinterpret_cast<PlanStorage*>(plan);   // pub is the first member
    std::free(ps->offsets);
    delete ps;
}

extern "C" int32_t zero_plan_owner(const zero_plan_t* plan, int64_t i)
{
    if (!plan || i < 0 || i >= plan->N || plan->S <= 0) return -1;
    return (int32_t)(i / plan->S);
}
