// ckpt.cpp - sharded optimizer-state checkpoints and R -> R' resharding.
//
// What the pages ask for:
//   - 14 bytes per parameter: bf16 parameter 2 + fp32 master 4 + Adam m, v 8
//     (BLOOM's checkpoint, CS324 Lecture 9 notes, section 2.1);
//   - restoring on a different card count needs the optimizer state of the
//     cards merged (same notes, exercise 11);
//   - bitwise-identical training from any checkpoint (PaLM, section 3.1);
//   - sharded parallel writes, atomic rename, asynchronous saves
//     (LLM infra 06, section 15.4, the failure mode of a crash while a
//     checkpoint is written).
//
// Format: one file per rank shard, "shard-RRRRR-of-NNNNN.zck", holding the
// rank's elements [lo, lo + len) of the flat vector: a 128-byte header, then
// bf16 params[len], fp32 master[len], m[len], v[len] (14 bytes/param).  The
// header carries the layout (R, rank, N, S, lo, len), the step count, the
// AdamW hyper-parameters, a Fletcher-64 checksum of the payload and one of
// the header itself.  A shard is written to "<name>.tmp", fsync'ed, then
// renamed, so a reader never sees a partial file.
//
// Resharding: element i sits at index i of the state arrays under every R
// (the layouts differ only in padding), so loading under R' reads, for each
// new shard, the byte ranges of the old shard files that overlap it.
//
// All little-endian; the header is written field by field (no struct
// padding assumptions).
#include <cuda_runtime.h>
#include <errno.h>
#include <fcntl.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include <sys/stat.h>
#include <unistd.h>

#include <atomic>
#include <cstdlib>
#include <string>
#include <thread>
#include <vector>

#include "zero_step.h"

namespace {

constexpr char kMagic[8] = {'Z', 'E', 'R', 'O', 'C', 'K', 'P', 'T'};
constexpr uint32_t kVersion = 1;
constexpr int64_t kHeaderBytes = 128;

// Fletcher-64: two running sums of 32-bit little-endian words modulo
// 2^32 - 1 (a trailing partial word is zero-padded).  Continuable across
// calls through the state pair.
struct Fletcher64 {
    uint64_t a = 0, b = 0;
    uint8_t pend[4];
    int npend = 0;
    void add_word(uint32_t w)
    {
        a = (a + w) % 0xFFFFFFFFull;
        b = (b + a) % 0xFFFFFFFFull;
    }
    void update(const void* data, size_t n)
    {
        const uint8_t* p = static_cast<const uint8_t*>(data);
        while (n && npend) {                       // finish a pending word
            pend[npend++] = *p++;
            --n;
            if (npend == 4) {
                add_word((uint32_t)pend[0] | (uint32_t)pend[1] << 8 | (uint32_t)pend[2] << 16 |
                         (uint32_t)pend[3] << 24);
                npend = 0;
            }
        }
        // bulk: defer the modulo, it cannot overflow within 2^16 words
        while (n >= 4) {
            size_t words = n / 4;
            if (words > 65536) words = 65536;
            for (size_t k = 0; k < words; ++k, p += 4) {
                const uint32_t w = (uint32_t)p[0] | (uint32_t)p[1] << 8 | (uint32_t)p[2] << 16 |
                                   (uint32_t)p[3] << 24;
                a += w;
                b += a;
            }
            a %= 0xFFFFFFFFull;
            b %= 0xFFFFFFFFull;
            n -= words * 4;
        }
        while (n) {
            pend[npend++] = *p++;
            --n;
        }
    }
    uint64_t finish()
    {
        if (npend) {
            while (npend < 4) pend[npend++] = 0;
            add_word((uint32_t)pend[0] | (uint32_t)pend[1] << 8 | (uint32_t)pend[2] << 16 |
                     (uint32_t)pend[3] << 24);
            npend = 0;
        }
        return b << 32 | a;
    }
};

struct Header {
    int32_t R, rank, M, stage;
    int64_t N, S, lo, len, step;
    zero_adamw_hparams hp;
    uint64_t payload_sum, header_sum;
};

void put32(uint8_t* p, uint32_t v) { for (int k = 0; k < 4; ++k) p[k] = (uint8_t)(v >> (8 * k)); }
void put64(uint8_t* p, uint64_t v) { for (int k = 0; k < 8; ++k) p[k] = (uint8_t)(v >> (8 * k)); }
uint32_t get32(const uint8_t* p)
{
    uint32_t v = 0;
    for (int k = 0; k < 4; ++k) v |= (uint32_t)p[k] << (8 * k);
    return v;
}
uint64_t get64(const uint8_t* p)
{
    uint64_t v = 0;
    for (int k = 0; k < 8; ++k) v |= (uint64_t)p[k] << (8 * k);
    return v;
}
uint32_t fbits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
float bitsf(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

// header layout (byte offsets): magic 0, version 8, header_bytes 12, R 16,
// rank 20, M 24, stage 28, N 32, S 40, lo 48, len 56, step 64, lr 72,
// beta1 76, beta2 80, eps 84, wd 88, payload_sum 96, header_sum 104, 112..127 zero
void encode(const Header& h, uint8_t* out)
{
    memset(out, 0, kHeaderBytes);
    memcpy(out, kMagic, 8);
    put32(out + 8, kVersion);
    put32(out + 12, (uint32_t)kHeaderBytes);
    put32(out + 16, (uint32_t)h.R);
    put32(out + 20, (uint32_t)h.rank);
    put32(out + 24, (uint32_t)h.M);
    put32(out + 28, (uint32_t)h.stage);
    put64(out + 32, (uint64_t)h.N);
    put64(out + 40, (uint64_t)h.S);
    put64(out + 48, (uint64_t)h.lo);
    put64(out + 56, (uint64_t)h.len);
    put64(out + 64, (uint64_t)h.step);
    put32(out + 72, fbits(h.hp.lr));
    put32(out + 76, fbits(h.hp.beta1));
    put32(out + 80, fbits(h.hp.beta2));
    put32(out + 84, fbits(h.hp.eps));
    put32(out + 88, fbits(h.hp.weight_decay));
    put64(out + 96, h.payload_sum);
    Fletcher64 f;
    f.update(out, kHeaderBytes);                 // header_sum field still zero
    put64(out + 104, f.finish());
}

zero_status decode(const uint8_t* in, Header* h)
{
    if (memcmp(in, kMagic, 8) != 0 || get32(in + 8) != kVersion ||
        get32(in + 12) != (uint32_t)kHeaderBytes)
        return ZERO_ERR_CORRUPT;
    uint8_t tmp[kHeaderBytes];
    memcpy(tmp, in, kHeaderBytes);
    put64(tmp + 104, 0);
    Fletcher64 f;
    f.update(tmp, kHeaderBytes);
    if (f.finish() != get64(in + 104)) return ZERO_ERR_CORRUPT;
    h->R = (int32_t)get32(in + 16);
    h->rank = (int32_t)get32(in + 20);
    h->M = (int32_t)get32(in + 24);
    h->stage = (int32_t)get32(in + 28);
    h->N = (int64_t)get64(in + 32);
    h->S = (int64_t)get64(in + 40);
    h->lo = (int64_t)get64(in + 48);
    h->len = (int64_t)get64(in + 56);
    h->step = (int64_t)get64(in + 64);
    h->hp.lr = bitsf(get32(in + 72));
    h->hp.beta1 = bitsf(get32(in + 76));
    h->hp.beta2 = bitsf(get32(in + 80));
    h->hp.eps = bitsf(get32(in + 84));
    h->hp.weight_decay = bitsf(get32(in + 88));
    h->payload_sum = get64(in + 96);
    h->header_sum = get64(in + 104);
    return ZERO_OK;
}

std::string shard_name(const std::string& dir, int r, int R)
{
    char buf[64];
    snprintf(buf, sizeof buf, "/shard-%05d-of-%05d.zck", r, R);
    return dir + buf;
}

bool write_all(int fd, const void* p, size_t n)
{
    const char* c = static_cast<const char*>(p);
    while (n) {
        const ssize_t w = ::write(fd, c, n > (1u << 30) ? (1u << 30) : n);
        if (w < 0) {
            if (errno == EINTR) continue;
            return false;
        }
        c += w;
        n -= (size_t)w;
    }
    return true;
}

bool pread_all(int fd, void* p, size_t n, int64_t off)
{
    char* c = static_cast<char*>(p);
    while (n) {
        const ssize_t r = ::pread(fd, c, n > (1u << 30) ? (1u << 30) : n, (off_t)off);
        if (r < 0) {
            if (errno == EINTR) continue;
            return false;
        }
        if (r == 0) return false;                 // short file
        c += r;
        n -= (size_t)r;
        off += r;
    }
    return true;
}

struct ShardSrc {
    const uint16_t* params;
    const float *master, *m, *v;
};

// write one shard file atomically: <name>.tmp, fsync, rename, fsync(dir)
zero_status write_shard(const std::string& dir, const Header& h0, const ShardSrc& src)
{
    Header h = h0;
    Fletcher64 f;
    const size_t n = (size_t)h.len;
    f.update(src.params + h.lo, 2 * n);
    f.update(src.master + h.lo, 4 * n);
    f.update(src.m + h.lo, 4 * n);
    f.update(src.v + h.lo, 4 * n);
    h.payload_sum = f.finish();
    uint8_t hdr[kHeaderBytes];
    encode(h, hdr);
    const std::string fin = shard_name(dir, h.rank, h.R);
    const std::string tmp = fin + ".tmp";
    const int fd = ::open(tmp.c_str(), O_WRONLY | O_CREAT | O_TRUNC, 0644);
    if (fd < 0) return ZERO_ERR_IO;
    bool ok = write_all(fd, hdr, kHeaderBytes) && write_all(fd, src.params + h.lo, 2 * n) &&
              write_all(fd, src.master + h.lo, 4 * n) && write_all(fd, src.m + h.lo, 4 * n) &&
              write_all(fd, src.v + h.lo, 4 * n) && ::fsync(fd) == 0;
    ok = (::close(fd) == 0) && ok;
    if (!ok || ::rename(tmp.c_str(), fin.c_str()) != 0) {
        ::unlink(tmp.c_str());
        return ZERO_ERR_IO;
    }
    const int dfd = ::open(dir.c_str(), O_RDONLY);
    if (dfd >= 0) {
        ::fsync(dfd);
        ::close(dfd);
    }
    return ZERO_OK;
}

zero_status write_all_shards(const zero_plan_t* plan, const ShardSrc& src, int64_t step,
                             const zero_adamw_hparams& hp, const std::string& dir, int threads)
{
    if (::mkdir(dir.c_str(), 0755) != 0 && errno != EEXIST) return ZERO_ERR_IO;
    const int R = plan->R;
    std::vector<zero_status> st((size_t)R, ZERO_OK);
    std::atomic<int> next{0};
    auto worker = [&]() {
        for (int r = next++; r < R; r = next++) {
            Header h{};
            h.R = R;
            h.rank = r;
            h.M = plan->M;
            h.stage = plan->stage;
            h.N = plan->N;
            h.S = plan->S;
            h.lo = (int64_t)r * plan->S;
            const int64_t len = plan->N - h.lo < plan->S ? plan->N - h.lo : plan->S;
            h.len = len > 0 ? len : 0;
            if (h.lo > plan->N) h.lo = plan->N;
            h.step = step;
            h.hp = hp;
            st[(size_t)r] = write_shard(dir, h, src);
        }
    };
    if (threads < 1) threads = 1;
    if (threads > R) threads = R;
    std::vector<std::thread> pool;
    for (int t = 1; t < threads; ++t) pool.emplace_back(worker);
    worker();
    for (auto& th : pool) th.join();
    for (zero_status s : st)
        if (s != ZERO_OK) return s;
    return ZERO_OK;
}

struct OldShards {
    int R = 0;
    int64_t N = 0, S = 0, step = 0;
    zero_adamw_hparams hp{};
    std::vector<Header> h;
};

// read and check every header of the checkpoint in dir
zero_status scan(const std::string& dir, OldShards* out)
{
    // the first shard tells R; every shard must agree
    int R = -1;
    for (int guess_R = 1; guess_R <= ZERO_MAX_R && R < 0; ++guess_R) {
        struct stat sb;
        if (::stat(shard_name(dir, 0, guess_R).c_str(), &sb) == 0) R = guess_R;
    }
    if (R < 0) return ZERO_ERR_IO;
    out->R = R;
    out->h.resize((size_t)R);
    for (int r = 0; r < R; ++r) {
        const int fd = ::open(shard_name(dir, r, R).c_str(), O_RDONLY);
        if (fd < 0) return ZERO_ERR_IO;
        uint8_t hdr[kHeaderBytes];
        const bool ok = pread_all(fd, hdr, kHeaderBytes, 0);
        struct stat sb;
        const bool st_ok = ::fstat(fd, &sb) == 0;
        ::close(fd);
        if (!ok || !st_ok) return ZERO_ERR_CORRUPT;
        Header h;
        if (zero_status e = decode(hdr, &h)) return e;
        if (h.R != R || h.rank != r) return ZERO_ERR_CORRUPT;
        if (sb.st_size != kHeaderBytes + 14 * h.len) return ZERO_ERR_CORRUPT;
        if (r == 0) {
            out->N = h.N;
            out->S = h.S;
            out->step = h.step;
            out->hp = h.hp;
        } else if (h.N != out->N || h.S != out->S || h.step != out->step) {
            return ZERO_ERR_CORRUPT;
        }
        out->h[(size_t)r] = h;
    }
    return ZERO_OK;
}

// verify one old shard's payload checksum (reads the whole file once)
zero_status verify(const std::string& dir, const OldShards& old, int r)
{
    const Header& h = old.h[(size_t)r];
    const int fd = ::open(shard_name(dir, r, old.R).c_str(), O_RDONLY);
    if (fd < 0) return ZERO_ERR_IO;
    std::vector<uint8_t> buf((size_t)1 << 24);
    Fletcher64 f;
    int64_t left = 14 * h.len, off = kHeaderBytes;
    bool ok = true;
    while (left > 0 && ok) {
        const size_t n = (size_t)(left < (int64_t)buf.size() ? left : (int64_t)buf.size());
        ok = pread_all(fd, buf.data(), n, off);
        f.update(buf.data(), n);
        left -= (int64_t)n;
        off += (int64_t)n;
    }
    ::close(fd);
    if (!ok) return ZERO_ERR_IO;
    return f.finish() == h.payload_sum ? ZERO_OK : ZERO_ERR_CORRUPT;
}

struct ShardDst {
    uint16_t* params;            // element i at params[i], i < N
    float *master, *m, *v;       // element i at [i]
};

// copy elements [lo, hi) of the flat vector from the old shards
zero_status read_range(const std::string& dir, const OldShards& old, int64_t lo, int64_t hi,
                       const ShardDst& dst)
{
    for (int r = 0; r < old.R && lo < hi; ++r) {
        const Header& h = old.h[(size_t)r];
        const int64_t a = lo > h.lo ? lo : h.lo;
        const int64_t b = hi < h.lo + h.len ? hi : h.lo + h.len;
        if (a >= b) continue;
        const int fd = ::open(shard_name(dir, r, old.R).c_str(), O_RDONLY);
        if (fd < 0) return ZERO_ERR_IO;
        const int64_t k = a - h.lo, n = b - a;
        const int64_t p_off = kHeaderBytes, w_off = p_off + 2 * h.len, m_off = w_off + 4 * h.len,
                      v_off = m_off + 4 * h.len;
        const bool ok = pread_all(fd, dst.params + a, 2 * (size_t)n, p_off + 2 * k) &&
                        pread_all(fd, dst.master + a, 4 * (size_t)n, w_off + 4 * k) &&
                        pread_all(fd, dst.m + a, 4 * (size_t)n, m_off + 4 * k) &&
                        pread_all(fd, dst.v + a, 4 * (size_t)n, v_off + 4 * k);
        ::close(fd);
        if (!ok) return ZERO_ERR_IO;
    }
    return ZERO_OK;
}

zero_status check_plan_basic(const zero_plan_t* plan)
{
    if (!plan) return ZERO_ERR_NULL;
    if (plan->R < 1 || plan->R > ZERO_MAX_R || plan->N < 0 || plan->S < 0 ||
        plan->S * plan->R < plan->N)
        return ZERO_ERR_INVALID_ARG;
    return ZERO_OK;
}

}  // namespace

// ----------------------------------------------------------- host layer --

extern "C" zero_status zero_ckpt_write_host(const zero_plan_t* plan, const uint16_t* params,
                                            const float* master, const float* m, const float* v,
                                            int64_t step, const zero_adamw_hparams* hp,
                                            const char* dir, int32_t n_threads)
{
    if (zero_status e = check_plan_basic(plan)) return e;
    if (!hp || !dir || (plan->N > 0 && (!params || !master || !m || !v))) return ZERO_ERR_NULL;
    if (step < 0) return ZERO_ERR_INVALID_ARG;
    ShardSrc src{params, master, m, v};
    return write_all_shards(plan, src, step, *hp, dir, n_threads);
}

extern "C" zero_status zero_ckpt_read_host(const zero_plan_t* plan, const char* dir, int32_t rank,
                                           uint16_t* params, float* master, float* m, float* v,
                                           int64_t* step_out, zero_adamw_hparams* hp_out)
{
    if (zero_status e = check_plan_basic(plan)) return e;
    if (!dir || (plan->N > 0 && (!params || !master || !m || !v))) return ZERO_ERR_NULL;
    if (rank < -1 || rank >= plan->R) return ZERO_ERR_INVALID_ARG;
    OldShards old;
    if (zero_status e = scan(dir, &old)) return e;
    if (old.N != plan->N) return ZERO_ERR_SIZE;
    // the new shard(s) to fill, and the old shards they touch
    int64_t lo = 0, hi = plan->N;
    if (rank >= 0) {
        lo = (int64_t)rank * plan->S;
        hi = lo + plan->S < plan->N ? lo + plan->S : plan->N;
        if (lo > plan->N) lo = hi = plan->N;
    }
    for (int r = 0; r < old.R; ++r) {
        const Header& h = old.h[(size_t)r];
        if (h.len > 0 && h.lo < hi && h.lo + h.len > lo)
            if (zero_status e = verify(dir, old, r)) return e;
    }
    ShardDst dst{params, master, m, v};
    if (zero_status e = read_range(dir, old, lo, hi, dst)) return e;
    if (step_out) *step_out = old.step;
    if (hp_out) *hp_out = old.hp;
    return ZERO_OK;
}

// --------------------------------------------------------- device layer --

struct zero_ckpt_job {
    std::thread writer;
    zero_status status = ZERO_OK;
    void* staging = nullptr;     // pinned host copy of the state
    cudaEvent_t copied = nullptr;
};

extern "C" zero_status zero_ckpt_save_async(const zero_plan_t* plan, const uint16_t* dev_params,
                                            const float* dev_master, const float* dev_m,
                                            const float* dev_v, int64_t step,
                                            const zero_adamw_hparams* hp, const char* dir,
                                            int32_t n_threads, void* stream,
                                            zero_ckpt_job** job_out)
{
    if (zero_status e = check_plan_basic(plan)) return e;
    if (!hp || !dir || !job_out) return ZERO_ERR_NULL;
    if (plan->N > 0 && (!dev_params || !dev_master || !dev_m || !dev_v)) return ZERO_ERR_NULL;
    if (step < 0) return ZERO_ERR_INVALID_ARG;
    *job_out = nullptr;
    const size_t n = (size_t)plan->N;
    auto* job = new (std::nothrow) zero_ckpt_job();
    if (!job) return ZERO_ERR_SIZE;
    const size_t bytes = 14 * n + 64;
    if (cudaMallocHost(&job->staging, bytes ? bytes : 64) != cudaSuccess) {
        delete job;
        return ZERO_ERR_CUDA;
    }
    char* base = static_cast<char*>(job->staging);
    uint16_t* hp_ = reinterpret_cast<uint16_t*>(base);
    float* hw = reinterpret_cast<float*>(base + ((2 * n + 15) & ~(size_t)15));
    float* hm = hw + n;
    float* hv = hm + n;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool ok = cudaEventCreateWithFlags(&job->copied, cudaEventDisableTiming) == cudaSuccess;
    if (ok && n) {
        ok = cudaMemcpyAsync(hp_, dev_params, 2 * n, cudaMemcpyDeviceToHost, st) == cudaSuccess &&
             cudaMemcpyAsync(hw, dev_master, 4 * n, cudaMemcpyDeviceToHost, st) == cudaSuccess &&
             cudaMemcpyAsync(hm, dev_m, 4 * n, cudaMemcpyDeviceToHost, st) == cudaSuccess &&
             cudaMemcpyAsync(hv, dev_v, 4 * n, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    }
    ok = ok && cudaEventRecord(job->copied, st) == cudaSuccess;
    if (!ok) {
        // copies already enqueued may still be writing into the staging
        // buffer: wait for the stream before freeing it
        cudaStreamSynchronize(st);
        if (job->copied) cudaEventDestroy(job->copied);
        cudaFreeHost(job->staging);
        delete job;
        return ZERO_ERR_CUDA;
    }
    // the state is in host memory once `copied` completes: later steps on
    // `stream` are ordered after the copies; the files are written here
    const zero_plan_t plan_copy = *plan;
    const zero_adamw_hparams hp_copy = *hp;
    const std::string d(dir);
    job->writer = std::thread([job, plan_copy, hp_copy, d, step, n_threads, hp_, hw, hm, hv]() {
        if (cudaEventSynchronize(job->copied) != cudaSuccess) {
            job->status = ZERO_ERR_CUDA;
            return;
        }
        // element i of the flat vector at index i: shift the fp32 views so
        // that [i] addresses element i (they start at element 0)
        ShardSrc src{hp_, hw, hm, hv};
        job->status = write_all_shards(&plan_copy, src, step, hp_copy, d, n_threads);
    });
    *job_out = job;
    return ZERO_OK;
}

extern "C" zero_status zero_ckpt_job_wait(zero_ckpt_job* job)
{
    if (!job) return ZERO_ERR_NULL;
    if (job->writer.joinable()) job->writer.join();
    const zero_status s = job->status;
    if (job->copied) cudaEventDestroy(job->copied);
    if (job->staging) cudaFreeHost(job->staging);
    delete job;
    return s;
}

extern "C" zero_status zero_ckpt_load(const zero_plan_t* plan, const char* dir,
                                      uint16_t* const* dev_params, int32_t n_params,
                                      float* dev_master, float* dev_m, float* dev_v,
                                      int64_t* step_out, zero_adamw_hparams* hp_out,
                                      void* stream)
{
    if (zero_status e = check_plan_basic(plan)) return e;
    if (!dir) return ZERO_ERR_NULL;
    if (n_params < 0 || n_params > plan->R) return ZERO_ERR_INVALID_ARG;
    if (plan->N > 0 && (!dev_master || !dev_m || !dev_v || (n_params > 0 && !dev_params)))
        return ZERO_ERR_NULL;
    const size_t n = (size_t)plan->N;
    void* stage = nullptr;
    if (cudaMallocHost(&stage, 14 * n + 64) != cudaSuccess) return ZERO_ERR_CUDA;
    char* base = static_cast<char*>(stage);
    uint16_t* hp_ = reinterpret_cast<uint16_t*>(base);
    float* hw = reinterpret_cast<float*>(base + ((2 * n + 15) & ~(size_t)15));
    float* hm = hw + n;
    float* hv = hm + n;
    zero_status e = zero_ckpt_read_host(plan, dir, -1, hp_, hw, hm, hv, step_out, hp_out);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (e == ZERO_OK && n) {
        bool ok = cudaMemcpyAsync(dev_master, hw, 4 * n, cudaMemcpyHostToDevice, st) == cudaSuccess &&
                  cudaMemcpyAsync(dev_m, hm, 4 * n, cudaMemcpyHostToDevice, st) == cudaSuccess &&
                  cudaMemcpyAsync(dev_v, hv, 4 * n, cudaMemcpyHostToDevice, st) == cudaSuccess;
        for (int k = 0; ok && k < n_params; ++k)
            ok = cudaMemcpyAsync(dev_params[k], hp_, 2 * n, cudaMemcpyHostToDevice, st) ==
                 cudaSuccess;
        ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
        if (!ok) e = ZERO_ERR_CUDA;
    }
    cudaFreeHost(stage);
    return e;
}
