// sv_api.cu -- host side of libsv: handle, argument checks, workspace and
// launch orchestration for the verify calls declared in sv.h.
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "sv_gumbel.cuh"
#include "sv_job.cuh"
#include "sv_topk.cuh"

namespace sv {
size_t pass_smem_bytes();
size_t rescue_scratch_doubles(int B);
cudaError_t pass_setup(int *blocks_per_sm);
cudaError_t pass_launch(const Job &j, int grid, cudaStream_t s);
cudaError_t spot_prep_launch(const Job &j, cudaStream_t s);
cudaError_t anyorder_prep_launch(const Job &j, cudaStream_t s);
cudaError_t seed_launch(const Job &j, int grid, cudaStream_t s);
cudaError_t seed_setup(int *blocks_per_sm);
cudaError_t post_setup(int occ[2]);
cudaError_t post_launch(const Job &j, int tv_grid, int resid_grid, int coop_grid, bool tv,
                        cudaStream_t s);
cudaError_t selftest_run(uint64_t seed, long long n, const uint64_t *skip, const float *gtab,
                         const float *gtop, double *res, cudaStream_t s);
cudaError_t wait_selftest_run(int *err, const unsigned *word, uint32_t limit, cudaStream_t s);
}  // namespace sv

using namespace sv;

struct sv_handle {
    int device = 0;
    int sms = 0;
    int pass_blocks = 1;   // resident streaming CTAs per SM
    int tv_blocks = 1;     // resident total-variation CTAs per SM
    int seed_blocks = 1;   // resident seed CTAs per SM
    bool resid_pair = false;  // two 512-thread residual CTAs fit on an SM
    int *d_err = nullptr;
    unsigned *d_ctl = nullptr;
    float *d_gtab = nullptr;      // [kGTab] G bounds of ordinary ids
    float *d_gtop = nullptr;      // [2 * kGTab] upper and lower G bounds of top ids
    uint64_t *d_skip = nullptr;   // [kSkipN] skip thresholds
    char *ws = nullptr;
    size_t ws_bytes = 0;
    unsigned *cnt = nullptr;  // completion counters: always zero between calls
    int cnt_B = 0;            // sequences the counter arena holds
    int force_rescue = 0;
    cudaEvent_t ev[2] = {nullptr, nullptr};  // caller-owned (SV_OPT_TIMING_EVENTS)
    bool timing = false;
    std::mutex mu;
};

namespace sv {
// Host fault injection for failure-path tests.  SV_FAULT_INJECT holds
// "call:code[,call:code...]"; a listed entry point returns the status
// `code` (1..6) at its launch point -- after its argument checks, before it
// enqueues anything -- without touching the GPU.  Unset, empty or malformed
// entries inject nothing.  The variable is read at every call.
sv_status fault_injected(const char *call)
{
    const char *env = getenv("SV_FAULT_INJECT");
    if (!env || !*env) return SV_OK;
    const size_t n = strlen(call);
    for (const char *p = env; *p;) {
        const char *end = strchr(p, ',');
        const size_t len = end ? (size_t)(end - p) : strlen(p);
        if (len > n + 1 && strncmp(p, call, n) == 0 && p[n] == ':') {
            char *stop = nullptr;
            const long code = strtol(p + n + 1, &stop, 10);
            if (stop == p + len && code >= 1 && code <= 6) return (sv_status)code;
        }
        if (!end) break;
        p = end + 1;
    }
    return SV_OK;
}
}  // namespace sv

namespace {

// Upper bounds of G = -log(-log u) for ordinary ids, rounded up to fp32 with
// one more ulp of slack: entry c bounds ids whose fine bits start with the
// byte c, i.e. w < (c + 1)/256 and u = w 255/256 < (c + 1) 255 / 65536.  The
// last entry bounds every ordinary id (u < 255/256).
static float up_f32(double g)
{
    float f = (float)g;
    if ((double)f < g) f = nextafterf(f, INFINITY);
    return nextafterf(f, INFINITY);
}

void gumbel_bound_table(float *t)
{
    for (int c = 0; c < kGTab; ++c)
        t[c] = up_f32(-log(-log((double)(c + 1) * 255.0 / 65536.0)));
}

static float down_f32(double g)
{
    float f = (float)g;
    if ((double)f > g) f = nextafterf(f, -INFINITY);
    return nextafterf(f, -INFINITY);
}

// The same for top ids: w < (c + 1)/256 gives 1 - u = (1 - w)/256 >
// (255 - c)/65536.  The last byte (w up to 1) has no finite bound.  Entries
// kGTab.. hold the lower bounds: w >= c/256 gives 1 - u <= (256 - c)/65536,
// rounded down with one more ulp of slack.
void gumbel_top_bound_table(float *t)
{
    for (int c = 0; c < kGTab - 1; ++c)
        t[c] = up_f32(-log(-log1p(-(double)(255 - c) / 65536.0)));
    t[kGTab - 1] = INFINITY;
    for (int c = 0; c < kGTab; ++c)
        t[kGTab + c] = down_f32(-log(-log1p(-(double)(256 - c) / 65536.0)));
}

// Skip thresholds C_g = ceil(2^64 (255/256)^g), g = 1..256 (entry 0 unused):
// 255^g as a little-endian byte string; C_g = 255^g * 256^(8-g) for g <= 8,
// else 255^g / 256^(g-8) rounded up (its bytes below 256^(g-8) dropped).
void skip_table(uint64_t *C)
{
    uint8_t n[272];
    memset(n, 0, sizeof n);
    n[0] = 1;
    int len = 1;
    C[0] = 0;
    for (int g = 1; g <= 256; ++g) {
        unsigned carry = 0;
        for (int i = 0; i < len; ++i) {
            const unsigned t = n[i] * 255u + carry;
            n[i] = (uint8_t)(t & 255u);
            carry = t >> 8;
        }
        while (carry) {
            n[len++] = (uint8_t)(carry & 255u);
            carry >>= 8;
        }
        uint64_t v = 0;
        if (g <= 8) {
            for (int i = len - 1; i >= 0; --i)
                v = (v << 8) | n[i];
            C[g] = v << (8 * (8 - g));
        } else {
            const int drop = g - 8;
            bool rest = false;
            for (int i = 0; i < drop && i < len; ++i)
                rest |= n[i] != 0;
            for (int i = len - 1; i >= drop; --i)
                v = (v << 8) | n[i];
            C[g] = v + (rest ? 1 : 0);
        }
    }
}

sv_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return SV_OK;
    if (e == cudaErrorMemoryAllocation) return SV_ERR_OOM;
    return SV_ERR_CUDA;
}

size_t align_up(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
    size_t rp, rs, resid, rescue, dtmp, tvpart, rpart, smask, svalid, seeds, total;
};

Layout layout(int B, int rows_per_seq, int parts, int K, int W, int tv_chunks, int states,
              size_t seed_recs)
{
    Layout L;
    size_t o = 0;
    L.rp = o;     o = align_up(o + (size_t)B * rows_per_seq * parts * sizeof(RowPart));
    L.rs = o;     o = align_up(o + (size_t)B * rows_per_seq * sizeof(RowStat));
    L.resid = o;  o = align_up(o + (size_t)B * sizeof(ResidEntry));
    L.rescue = o; o = align_up(o + (size_t)B * sizeof(RescueEntry));
    L.dtmp = o;   o = align_up(o + (size_t)B * std::max(W, 1) * sizeof(DraftTmp));
    L.tvpart = o; o = align_up(o + (size_t)B * std::max(K, 1) * tv_chunks * sizeof(float));
    L.rpart = o;  o = align_up(o + rescue_scratch_doubles(B) * sizeof(double));
    L.smask = o;  o = align_up(o + (size_t)B * states * sizeof(uint64_t));
    L.svalid = o; o = align_up(o + (size_t)B * sizeof(unsigned));
    L.seeds = o;  o = align_up(o + seed_recs * sizeof(SeedRec));
    L.total = o;
    return L;
}

// Grow the workspace (stream-ordered); new memory is zeroed so that every
// counter starts at zero.  Kernels return their counters to zero.
sv_status ensure_ws(sv_handle *h, size_t bytes, cudaStream_t s)
{
    if (bytes <= h->ws_bytes) return SV_OK;
    size_t nb = std::max(bytes, h->ws_bytes * 2);
    if (h->ws) {
        cudaError_t e = cudaFreeAsync(h->ws, s);
        if (e != cudaSuccess) return cuda_status(e);
        h->ws = nullptr;
        h->ws_bytes = 0;
    }
    void *p = nullptr;
    cudaError_t e = cudaMallocAsync(&p, nb, s);
    if (e != cudaSuccess) return cuda_status(e);
    e = cudaMemsetAsync(p, 0, nb, s);
    if (e != cudaSuccess) return cuda_status(e);
    h->ws = (char *)p;
    h->ws_bytes = nb;
    return SV_OK;
}

// Counter arena: seq_done [Bcap], tvdone [kMaxK * Bcap].
// The kernels return every counter they touch to zero, so the arena is zeroed
// only when it is (re)allocated.
constexpr int kCntPerSeq = 1 + kMaxK;

sv_status ensure_cnt(sv_handle *h, int B, cudaStream_t s)
{
    if (B <= h->cnt_B) return SV_OK;
    int nb = std::max(B, 2 * h->cnt_B);
    if (h->cnt) {
        cudaError_t e = cudaFreeAsync(h->cnt, s);
        if (e != cudaSuccess) return cuda_status(e);
        h->cnt = nullptr;
        h->cnt_B = 0;
    }
    void *p = nullptr;
    cudaError_t e = cudaMallocAsync(&p, (size_t)nb * kCntPerSeq * sizeof(unsigned), s);
    if (e != cudaSuccess) return cuda_status(e);
    e = cudaMemsetAsync(p, 0, (size_t)nb * kCntPerSeq * sizeof(unsigned), s);
    if (e != cudaSuccess) return cuda_status(e);
    h->cnt = (unsigned *)p;
    h->cnt_B = nb;
    return SV_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Shape checks shared by every logit tensor argument.
bool logits_ok(const void *p, sv_dtype dt, int64_t rs, int V)
{
    if (!p || !aligned16(p)) return false;
    if (dt != SV_F32 && dt != SV_BF16) return false;
    int esz = dt == SV_BF16 ? 2 : 4;
    if (V < 1 || (int64_t)V * esz % 16 != 0) return false;
    if (rs < V || (rs * esz) % 16 != 0) return false;
    if ((int64_t)V > (int64_t)1 << 30) return false;
    return true;
}

void fill_common(Job &j, sv_handle *h, const void *src0, sv_dtype dt, int64_t rs, int V)
{
    memset(&j, 0, sizeof j);
    j.dtype = dt;
    j.src0 = (const char *)src0;
    int esz = dt == SV_BF16 ? 2 : 4;
    j.rs = rs * esz;
    j.V = V;
    j.nvec = (int)((int64_t)V * esz / 16);
    j.err = h->d_err;
    j.ctl = h->d_ctl;
    j.gtab = h->d_gtab;
    j.gtop = h->d_gtop;
    j.skip = h->d_skip;
    j.force_rescue = h->force_rescue;
    j.c1 = 1.4426950408889634f;
    j.eos = -1;
}

// Choose the row split and bind the workspace; returns the pass grid size.
sv_status plan(sv_handle *h, Job &j, int rows_per_seq, cudaStream_t s, int tv_chunks, int *grid)
{
    const int resident = h->sms * h->pass_blocks;
    long long rows = (long long)j.B * rows_per_seq;
    int max_parts = std::max(1, (j.nvec + kStageVecs - 1) / kStageVecs);
    long long want = (4LL * resident + rows - 1) / std::max(rows, 1LL);
    int parts = (int)std::min<long long>(std::max<long long>(want, 1), std::min(max_parts, 16));
    j.rows_per_seq = rows_per_seq;
    j.parts = parts;
    j.part_vecs = (j.nvec + parts - 1) / parts;
    j.parts = (j.nvec + j.part_vecs - 1) / j.part_vecs;  // no empty part
    j.total_units = rows * j.parts;
    // longest fp32 summation path: the chunk tree, one addition per stage of a
    // unit, the warp sum and the sum over consumer warps (records are merged
    // in fp64)
    const int stages_per_unit = (j.part_vecs + kStageVecs - 1) / kStageVecs;
    // plus the absolute error of log2 S in the row merge (below 2^-22)
    j.eps_lse = lse_rel_bound_stream((double)j.V, kLseSumDepth + 2.0 + stages_per_unit) + 0x1p-22;
    // exact ratios (log2(e)/T) / fl32(log2(e)/T) and reciprocals, once per call
    auto ratio = [](float c, float T) {
        return (c > 0.f && T > 0.f) ? (1.4426950408889634 / (double)T) / (double)c : 1.0;
    };
    j.crp = ratio(j.cp, j.Tp);
    j.crq = ratio(j.cq, j.Tq);
    j.cr1 = ratio(j.c1, 1.f);
    j.rTp = j.Tp > 0.f ? 1.0 / (double)j.Tp : 0.0;
    j.rTq = j.Tq > 0.f ? 1.0 / (double)j.Tq : 0.0;
    j.tv_chunks = tv_chunks;
    // seed spans: the blocks of 256 ids of every Gumbel-max row, end to end,
    // in equal spans, one per seed warp of one resident wave (at least 32
    // blocks, one per lane).  A row meets at most ceil(nblk / span) span
    // boundaries, so it has that many records plus one.
    const int nblk = (j.V + 255) / 256;
    const long long grows = (long long)j.B * gumbel_rows(j);
    const long long sblocks = grows * nblk;
    const long long swarps = 8LL * h->seed_blocks * h->sms;
    j.seed_span = (int)std::min<long long>(
        std::max<long long>(32, (sblocks + swarps - 1) / swarps), 1LL << 30);
    j.seed_chunks = grows ? (nblk + j.seed_span - 1) / j.seed_span + 1 : 0;
    const size_t seed_recs = (size_t)j.B * gumbel_rows(j) * j.seed_chunks;
    Layout L = layout(j.B, rows_per_seq, j.parts, j.K, j.W, tv_chunks,
                      j.kind == K_SPOT ? j.N + 1 : (j.kind == K_ANYORDER ? 1 : 0), seed_recs);
    sv_status st = ensure_ws(h, L.total, s);
    if (st != SV_OK) return st;
    st = ensure_cnt(h, j.B, s);
    if (st != SV_OK) return st;
    j.seq_done = h->cnt;
    j.tvdone = h->cnt + h->cnt_B;
    char *w = h->ws;
    j.rp = (RowPart *)(w + L.rp);
    j.rs_stat = (RowStat *)(w + L.rs);
    j.resid = (ResidEntry *)(w + L.resid);
    j.rescue = (RescueEntry *)(w + L.rescue);
    j.dtmp = (DraftTmp *)(w + L.dtmp);
    j.tvpart = (float *)(w + L.tvpart);
    j.rpart = (double *)(w + L.rpart);
    j.smask = (uint64_t *)(w + L.smask);
    j.svalid = (unsigned *)(w + L.svalid);
    j.seeds = seed_recs ? (SeedRec *)(w + L.seeds) : nullptr;
    *grid = (int)std::min<long long>(j.total_units, resident);
    return SV_OK;
}

// The timing events (SV_OPT_TIMING_EVENTS) bracket the streaming pass with
// the kernels that prepare it (state masks, seed records).
sv_status launch(sv_handle *h, const Job &j, int grid, cudaStream_t s, bool post, bool tv)
{
    if (h->timing) cudaEventRecord(h->ev[0], s);
    if (j.kind == K_SPOT || j.kind == K_ANYORDER) {
        cudaError_t e = j.kind == K_SPOT ? spot_prep_launch(j, s) : anyorder_prep_launch(j, s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (j.seeds) {
        // one warp per span (8 warps a CTA): at most one resident wave
        const long long sblocks = (long long)j.B * gumbel_rows(j) * ((j.V + 255) / 256);
        const long long warps = (sblocks + j.seed_span - 1) / j.seed_span;
        const int grid = (int)((warps + 7) / 8);
        cudaError_t e = seed_launch(j, std::max(grid, 1), s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    cudaError_t e = pass_launch(j, grid, s);
    if (h->timing) cudaEventRecord(h->ev[1], s);
    if (e != cudaSuccess) return cuda_status(e);
    if (!post) return SV_OK;
    // the residual pass: a CTA per sequence, two per SM when there are more
    // sequences than SMs
    const int rgrid = j.B > h->sms && h->resid_pair ? std::min(j.B, 2 * h->sms)
                                                   : std::min(j.B, h->sms);
    return cuda_status(post_launch(j, h->sms * h->tv_blocks, rgrid, h->sms, tv, s));
}

}  // namespace

extern "C" {

const char *sv_status_string(sv_status s)
{
    switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARG: return "invalid argument";
    case SV_ERR_CUDA: return "CUDA runtime error";
    case SV_ERR_OOM: return "out of device memory";
    case SV_ERR_TIMEOUT: return "a bounded device wait expired";
    case SV_ERR_UNSUPPORTED: return "unsupported device or shape";
    case SV_ERR_DEVICE_BOUNDS: return "token id, position or parent out of range";
    }
    return "unknown status";
}

sv_status sv_create(sv_handle **out)
{
    if (!out) return SV_ERR_INVALID_ARG;
    *out = nullptr;
    if (sv_status fi = fault_injected("sv_create")) return fi;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_UNSUPPORTED;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return SV_ERR_UNSUPPORTED;
    if (prop.major != 10 || prop.minor != 3) return SV_ERR_UNSUPPORTED;  // built for sm_103a
    sv_handle *h = new sv_handle();
    h->device = dev;
    h->sms = prop.multiProcessorCount;
    int nb = 0, pb[2] = {0, 0};
    cudaError_t e = pass_setup(&nb);
    h->pass_blocks = std::max(nb, 1);
    if (e == cudaSuccess) e = post_setup(pb);
    h->tv_blocks = std::max(1, pb[0]);
    h->resid_pair = pb[1] >= 2;
    int sb = 0;
    if (e == cudaSuccess) e = seed_setup(&sb);
    h->seed_blocks = std::max(1, sb);
    if (e == cudaSuccess) e = cudaMalloc(&h->d_err, sizeof(int));
    if (e == cudaSuccess) e = cudaMalloc(&h->d_ctl, C_NCTL * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMalloc(&h->d_gtab, kGTab * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&h->d_gtop, 2 * kGTab * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&h->d_skip, kSkipN * sizeof(uint64_t));
    if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(h->d_ctl, 0, C_NCTL * sizeof(unsigned));
    if (e == cudaSuccess) {
        float t[2 * kGTab];
        gumbel_bound_table(t);
        e = cudaMemcpy(h->d_gtab, t, kGTab * sizeof(float), cudaMemcpyHostToDevice);
        gumbel_top_bound_table(t);
        if (e == cudaSuccess) e = cudaMemcpy(h->d_gtop, t, sizeof t, cudaMemcpyHostToDevice);
        uint64_t c[kSkipN];
        skip_table(c);
        if (e == cudaSuccess) e = cudaMemcpy(h->d_skip, c, sizeof c, cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
        sv_destroy(h);
        return cuda_status(e);
    }
    *out = h;
    return SV_OK;
}

sv_status sv_destroy(sv_handle *h)
{
    if (!h) return SV_OK;
    cudaDeviceSynchronize();
    if (h->ws) cudaFree(h->ws);
    if (h->cnt) cudaFree(h->cnt);
    if (h->d_err) cudaFree(h->d_err);
    if (h->d_ctl) cudaFree(h->d_ctl);
    if (h->d_gtab) cudaFree(h->d_gtab);
    if (h->d_gtop) cudaFree(h->d_gtop);
    if (h->d_skip) cudaFree(h->d_skip);
    delete h;
    return SV_OK;
}

sv_status sv_sync_status(sv_handle *h, void *stream)
{
    if (!h) return SV_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    int code = 0;
    e = cudaMemcpy(&code, h->d_err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    if (code != 0) {
        // A wait expired or an input was out of range: the counters may not
        // have returned to zero, so clear them with the error word.
        cudaMemset(h->d_err, 0, sizeof(int));
        unsigned keep = 0;
        cudaMemcpy(&keep, h->d_ctl + C_RESCUED, sizeof(unsigned), cudaMemcpyDeviceToHost);
        cudaMemset(h->d_ctl, 0, C_NCTL * sizeof(unsigned));
        cudaMemcpy(h->d_ctl + C_RESCUED, &keep, sizeof(unsigned), cudaMemcpyHostToDevice);
        if (h->cnt) cudaMemset(h->cnt, 0, (size_t)h->cnt_B * kCntPerSeq * sizeof(unsigned));
        cudaDeviceSynchronize();
    }
    return (sv_status)code;
}

sv_status sv_rescue_count(sv_handle *h, void *stream, int64_t *count)
{
    if (!h || !count) return SV_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e);
    unsigned c = 0;
    e = cudaMemcpy(&c, h->d_ctl + C_RESCUED, sizeof c, cudaMemcpyDeviceToHost);
    *count = c;
    return cuda_status(e);
}

sv_status sv_selftest(sv_handle *h, uint64_t seed, int64_t n, double *ratios, void *stream)
{
    if (!h || !ratios || n < 1) return SV_ERR_INVALID_ARG;
    return cuda_status(
        selftest_run(seed, n, h->d_skip, h->d_gtab, h->d_gtop, ratios, (cudaStream_t)stream));
}

sv_status sv_wait_selftest(sv_handle *h, int64_t limit, void *stream)
{
    if (!h || limit < 0 || limit > (int64_t)kSpinLimit) return SV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(h->mu);
    // the word waited on is the handle's control word C_RESCUED, which only
    // the fp64 path changes, and never while this kernel runs on the stream
    return cuda_status(wait_selftest_run(h->d_err, h->d_ctl + C_RESCUED, (uint32_t)limit,
                                         (cudaStream_t)stream));
}

sv_status sv_set_option(sv_handle *h, sv_option opt, int64_t value)
{
    if (!h) return SV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(h->mu);
    switch (opt) {
    case SV_OPT_FORCE_RESCUE:
        h->force_rescue = value ? 1 : 0;
        return SV_OK;
    case SV_OPT_TIMING_EVENTS:
        if (value == 0) {
            h->timing = false;
            return SV_OK;
        }
        memcpy(h->ev, (const void *)(intptr_t)value, sizeof h->ev);
        h->timing = true;
        return SV_OK;
    }
    return SV_ERR_INVALID_ARG;
}

sv_status sv_verify_greedy(sv_handle *h, const void *target, sv_dtype dtype, int64_t row_stride,
                           int B, int K, int V, const int32_t *draft_ids,
                           const int32_t *draft_len, int32_t *accept_len, int32_t *next_token,
                           void *stream)
{
    if (!h || B < 0 || K < 0 || K > kMaxK) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!logits_ok(target, dtype, row_stride, V) || !accept_len || !next_token ||
        (K > 0 && !draft_ids))
        return SV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(h->mu);
    cudaStream_t s = (cudaStream_t)stream;
    Job j;
    fill_common(j, h, target, dtype, row_stride, V);
    j.kind = K_GREEDY;
    j.B = B;
    j.K = K;
    j.ids = draft_ids;
    j.lens = draft_len;
    if (sv_status fi = fault_injected("sv_verify_greedy")) return fi;
    j.acc = accept_len;
    j.next = next_token;
    int grid;
    sv_status st = plan(h, j, K + 1, s, 1, &grid);
    if (st != SV_OK) return st;
    return launch(h, j, grid, s, false, false);
}

sv_status sv_verify_sample(sv_handle *h, const void *target, const void *draft, sv_dtype dtype,
                           int64_t row_stride, int B, int K, int V, const int32_t *draft_ids,
                           const int32_t *draft_len, float T_p, float T_q, sv_accept_mode mode,
                           float lam, uint64_t seed, const int64_t *pos_base,
                           int32_t *accept_len, int32_t *next_token, float *p_at_draft,
                           float *q_at_draft, float *lse_p, float *lse_q, float *tv,
                           int32_t *flags, void *stream)
{
    if (!h || B < 0 || K < 0 || K > kMaxK) return SV_ERR_INVALID_ARG;
    if (!(T_p >= 0.f) || !(T_q >= 0.f) || !isfinite(T_p) || !isfinite(T_q)) return SV_ERR_INVALID_ARG;
    if (mode == SV_LENIENT_RATIO && !(lam >= 1.f && isfinite(lam))) return SV_ERR_INVALID_ARG;
    if (mode == SV_LENIENT_LINEAR && !(lam >= 0.f && lam <= 1.f)) return SV_ERR_INVALID_ARG;
    if (mode == SV_LENIENT_CACTUS && !(lam >= 0.f && isfinite(lam))) return SV_ERR_INVALID_ARG;
    if (mode != SV_LOSSLESS && mode != SV_LENIENT_RATIO && mode != SV_LENIENT_LINEAR &&
        mode != SV_LENIENT_CACTUS)
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (T_p == 0.f) {  // greedy rule on the target rows
        if (T_q != 0.f) return SV_ERR_INVALID_ARG;
        return sv_verify_greedy(h, target, dtype, row_stride, B, K, V, draft_ids, draft_len,
                                accept_len, next_token, stream);
    }
    if (T_q == 0.f) return SV_ERR_INVALID_ARG;
    if (!logits_ok(target, dtype, row_stride, V) || !accept_len || !next_token ||
        (K > 0 && (!draft_ids || !logits_ok(draft, dtype, row_stride, V))))
        return SV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(h->mu);
    cudaStream_t s = (cudaStream_t)stream;
    Job j;
    fill_common(j, h, target, dtype, row_stride, V);
    j.kind = K_SAMPLE;
    j.src1 = (const char *)draft;
    j.B = B;
    j.K = K;
    j.Tp = T_p;
    j.Tq = T_q;
    j.cp = (float)(1.4426950408889634 / (double)T_p);
    j.cq = (float)(1.4426950408889634 / (double)T_q);
    j.invTp = (float)(1.0 / (double)T_p);
    j.amode = mode;
    j.lam = lam;
    j.cactus_emd = mode == SV_LENIENT_CACTUS ? exp(-(double)lam) * (1.0 - 1e-12) : 0.0;
    j.seed = seed;
    j.ids = draft_ids;
    j.lens = draft_len;
    j.pos_base = pos_base;
    j.acc = accept_len;
    j.next = next_token;
    j.flags = flags;
    j.p_at = p_at_draft;
    j.q_at = q_at_draft;
    j.lse_p = lse_p;
    j.lse_q = lse_q;
    j.tv = tv;
    const int tvc = (int)std::min<long long>(
        16, std::max<long long>(1, (4LL * h->sms + (long long)B * std::max(K, 1) - 1) /
                                       ((long long)B * std::max(K, 1))));
    if (sv_status fi = fault_injected("sv_verify_sample")) return fi;
    int grid;
    sv_status st = plan(h, j, 2 * K + 1, s, tvc, &grid);
    if (st != SV_OK) return st;
    return launch(h, j, grid, s, true, tv != nullptr && K > 0);
}

sv_status sv_verify_tree(sv_handle *h, const void *node_logits, sv_dtype dtype, int64_t row_stride,
                         int B, int N, int V, const int32_t *parent, const int32_t *node_pos,
                         const int32_t *node_tok, float T, uint64_t seed,
                         const int64_t *pos_base, int32_t *path_len, int32_t *path_nodes,
                         int max_depth, int32_t *commit_count, uint8_t *match, int32_t *flags,
                         void *stream)
{
    if (!h || B < 0 || N < 1 || N > kMaxN || max_depth < 0) return SV_ERR_INVALID_ARG;
    if (!(T >= 0.f) || !isfinite(T)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!path_len || !commit_count || (max_depth > 0 && !path_nodes)) return SV_ERR_INVALID_ARG;
    if (!logits_ok(node_logits, dtype, row_stride, V) || !parent || !node_pos || !node_tok)
        return SV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(h->mu);
    cudaStream_t s = (cudaStream_t)stream;
    Job j;
    fill_common(j, h, node_logits, dtype, row_stride, V);
    j.kind = K_TREE;
    j.B = B;
    j.N = N;
    j.Tp = T;
    j.invTp = T > 0.f ? (float)(1.0 / (double)T) : 0.f;
    j.seed = seed;
    j.pos_base = pos_base;
    j.parent = parent;
    j.node_pos = node_pos;
    j.node_tok = node_tok;
    j.path_len = path_len;
    j.path_nodes = path_nodes;
    j.max_depth = max_depth;
    j.commit_count = commit_count;
    j.match = match;
    j.flags = flags;
    if (sv_status fi = fault_injected("sv_verify_tree")) return fi;
    int grid;
    sv_status st = plan(h, j, N, s, 1, &grid);
    if (st != SV_OK) return st;
    return launch(h, j, grid, s, false, false);
}

sv_status sv_verify_spot(sv_handle *h, const void *state_logits, sv_dtype dtype,
                         int64_t row_stride, int B, int N, int L, int V, const int32_t *parent,
                         const int32_t *node_pos, const int32_t *node_tok,
                         const uint64_t *root_mask, float T, uint64_t seed,
                         const int64_t *pos_base, int32_t *path_len, int32_t *path_nodes,
                         int max_depth, int32_t *commit_count, int32_t *commit_pos,
                         int32_t *commit_tok, uint8_t *match, int32_t *state_pos,
                         int32_t *state_tok, int32_t *flags, void *stream)
{
    if (!h || B < 0 || N < 0 || N > kMaxN || L < 1 || L > kMaxL || max_depth < 0)
        return SV_ERR_INVALID_ARG;
    if (!(T >= 0.f) || !isfinite(T)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!path_len || !commit_count || !commit_pos || !commit_tok || !root_mask ||
        (max_depth > 0 && !path_nodes) || (N > 0 && (!parent || !node_pos || !node_tok)))
        return SV_ERR_INVALID_ARG;
    if (!logits_ok(state_logits, dtype, row_stride, V)) return SV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(h->mu);
    cudaStream_t s = (cudaStream_t)stream;
    Job j;
    fill_common(j, h, state_logits, dtype, row_stride, V);
    j.kind = K_SPOT;
    j.B = B;
    j.N = N;
    j.L = L;
    j.Tp = T;
    j.invTp = T > 0.f ? (float)(1.0 / (double)T) : 0.f;
    j.seed = seed;
    j.pos_base = pos_base;
    j.parent = parent;
    j.node_pos = node_pos;
    j.node_tok = node_tok;
    j.root_mask = root_mask;
    j.path_len = path_len;
    j.path_nodes = path_nodes;
    j.max_depth = max_depth;
    j.commit_count = commit_count;
    j.commit_pos = commit_pos;
    j.commit_tok = commit_tok;
    j.match = match;
    j.state_pos = state_pos;
    j.state_tok = state_tok;
    j.flags = flags;
    if (sv_status fi = fault_injected("sv_verify_spot")) return fi;
    int grid;
    sv_status st = plan(h, j, (N + 1) * L, s, 1, &grid);
    if (st != SV_OK) return st;
    return launch(h, j, grid, s, false, false);
}

sv_status sv_packed_anyorder_step(sv_handle *h, const void *logits, sv_dtype dtype,
                                  int64_t row_stride, int B, int Kv, int W, int V,
                                  const int32_t *u, const int32_t *win_pos, const int32_t *order,
                                  const int32_t *draft, const int32_t *end_pos, int32_t eos_id,
                                  int32_t *accept_len, int32_t *commit_len, int32_t *commit_pos,
                                  int32_t *commit_tok, int32_t *end_out, int32_t *next_draft,
                                  float *score, void *stream)
{
    if (!h || B < 0 || Kv < 1 || Kv > kMaxK || W < 1 || W > kMaxK) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!logits_ok(logits, dtype, row_stride, V) || !u || !win_pos || !order || !draft ||
        !end_pos || !accept_len || !commit_len || !commit_pos || !commit_tok || !end_out ||
        !next_draft)
        return SV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(h->mu);
    cudaStream_t s = (cudaStream_t)stream;
    Job j;
    fill_common(j, h, logits, dtype, row_stride, V);
    j.kind = K_ANYORDER;
    j.B = B;
    j.K = Kv;
    j.W = W;
    j.lens = u;
    j.win_pos = win_pos;
    j.order = order;
    j.ids = draft;
    j.end_in = end_pos;
    j.eos = eos_id;
    j.acc = accept_len;
    j.commit_len = commit_len;
    j.commit_pos = commit_pos;
    j.commit_tok = commit_tok;
    j.end_out = end_out;
    j.next_draft = next_draft;
    j.confidence = score;
    if (sv_status fi = fault_injected("sv_packed_anyorder_step")) return fi;
    int grid;
    sv_status st = plan(h, j, Kv + W, s, 1, &grid);
    if (st != SV_OK) return st;
    return launch(h, j, grid, s, false, false);
}

sv_status sv_packed_step(sv_handle *h, const void *logits, sv_dtype dtype, int64_t row_stride,
                         int B, int K, int W, int V, const int32_t *prev_draft,
                         const int32_t *prev_len, const float *prev_q_at_draft,
                         const void *prev_draft_logits, const int32_t *prev_q_offset, float T,
                         uint64_t seed, uint64_t iter, const int64_t *pos_base, int32_t eos_id,
                         const int32_t *remaining, int32_t *accept_len, int32_t *commit_len,
                         int32_t *committed, int32_t *next_draft, int32_t *next_len,
                         float *next_q_at_draft, float *confidence, int32_t *flags,
                         void *stream)
{
    if (!h || B < 0 || K < 1 || K > kMaxK || W < 1 || W > kMaxK) return SV_ERR_INVALID_ARG;
    if (!(T >= 0.f) || !isfinite(T)) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!logits_ok(logits, dtype, row_stride, V) || !prev_len || (K > 1 && !prev_draft) ||
        !accept_len || !commit_len || !committed || !next_draft || !next_len)
        return SV_ERR_INVALID_ARG;
    if (T > 0.f && ((K > 1 && !prev_q_at_draft) || !prev_q_offset ||
                    !logits_ok(prev_draft_logits, dtype, row_stride, V)))
        return SV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(h->mu);
    cudaStream_t s = (cudaStream_t)stream;
    Job j;
    fill_common(j, h, logits, dtype, row_stride, V);
    j.kind = K_PACKED;
    j.src2 = (const char *)prev_draft_logits;
    j.B = B;
    j.K = K;
    j.W = W;
    j.Tp = T;
    j.Tq = T;
    j.cp = T > 0.f ? (float)(1.4426950408889634 / (double)T) : 0.f;
    j.cq = j.cp;
    j.invTp = T > 0.f ? (float)(1.0 / (double)T) : 0.f;
    j.seed = seed;
    j.iter = iter;
    j.pos_base = pos_base;
    j.eos = eos_id;
    j.remaining = remaining;
    j.ids = prev_draft;
    j.lens = prev_len;
    j.prev_q = prev_q_at_draft;
    j.prev_off = prev_q_offset;
    j.acc = accept_len;
    j.commit_len = commit_len;
    j.committed = committed;
    j.next_draft = next_draft;
    j.next_len = next_len;
    j.next_q = next_q_at_draft;
    j.confidence = confidence;
    j.flags = flags;
    if (sv_status fi = fault_injected("sv_packed_step")) return fi;
    int grid;
    sv_status st = plan(h, j, K + W, s, 1, &grid);
    if (st != SV_OK) return st;
    return launch(h, j, grid, s, T > 0.f, false);
}

sv_status sv_packed_topk_step(sv_handle *h, const void *logits, sv_dtype dtype,
                              int64_t row_stride, int B, int K, int W, int V, int kp, int kq,
                              const int32_t *prev_draft, const int32_t *prev_len,
                              const int32_t *prev_q_ids, const float *prev_q_probs,
                              const int32_t *prev_q_offset, float T, uint64_t seed, uint64_t iter,
                              const int64_t *pos_base, int32_t eos_id, const int32_t *remaining,
                              int32_t *accept_len, int32_t *commit_len, int32_t *committed,
                              int32_t *next_draft, int32_t *next_len, float *next_q_at_draft,
                              int32_t *q_ids, float *q_probs, int32_t *flags, void *stream)
{
    if (!h || B < 0 || K < 1 || K > kMaxK || W < 1 || W > kMaxK) return SV_ERR_INVALID_ARG;
    if (!(T > 0.f) || !isfinite(T)) return SV_ERR_INVALID_ARG;
    if (kp < 1 || kq < 1 || kp > kTopkMax || kq > kTopkMax || kp > V || kq > V)
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    if (!logits_ok(logits, dtype, row_stride, V) || !prev_len || (K > 1 && !prev_draft) ||
        !prev_q_ids || !prev_q_probs || !prev_q_offset || !accept_len || !commit_len ||
        !committed || !next_draft || !next_len || !q_ids || !q_probs)
        return SV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(h->mu);
    cudaStream_t s = (cudaStream_t)stream;
    TopkJob t;
    memset(&t, 0, sizeof t);
    const int esz = dtype == SV_BF16 ? 2 : 4;
    t.src = (const char *)logits;
    t.rs = row_stride * esz;
    t.dtype = dtype;
    t.V = V;
    t.nvec = (int)((int64_t)V * esz / 16);
    t.B = B;
    t.K = K;
    t.W = W;
    t.kp = kp;
    t.kq = kq;
    t.T = T;
    t.seed = seed;
    t.iter = iter;
    t.pos_base = pos_base;
    t.eos = eos_id;
    t.remaining = remaining;
    t.prev_draft = prev_draft;
    t.prev_len = prev_len;
    t.prev_q_ids = prev_q_ids;
    t.prev_q_probs = prev_q_probs;
    t.prev_off = prev_q_offset;
    t.skip = h->d_skip;
    t.acc = accept_len;
    t.commit_len = commit_len;
    t.committed = committed;
    t.next_draft = next_draft;
    t.next_len = next_len;
    t.next_q = next_q_at_draft;
    t.q_ids = q_ids;
    t.q_probs = q_probs;
    t.flags = flags;
    t.err = h->d_err;
    if (sv_status fi = fault_injected("sv_packed_topk_step")) return fi;
    // workspace: the sorted list of every row (kTopkMax logits, ids and
    // Gumbel values) and its log-sum-exp
    const size_t rows = (size_t)B * (K + W);
    sv_status st = ensure_ws(h, rows * (kTopkMax * 16 + 8), s);
    if (st != SV_OK) return st;
    t.lg = (double *)h->ws;
    t.lL = (double *)(h->ws + rows * kTopkMax * 8);
    t.lval = (float *)(h->ws + rows * (kTopkMax * 8 + 8));
    t.lid = (int32_t *)(h->ws + rows * (kTopkMax * 12 + 8));
    if (h->timing) cudaEventRecord(h->ev[0], s);
    cudaError_t e = topk_select_launch(t, s);
    if (h->timing) cudaEventRecord(h->ev[1], s);
    if (e == cudaSuccess) e = topk_decide_launch(t, s);
    return cuda_status(e);
}

}  // extern "C"
