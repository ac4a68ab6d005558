// sv_job.cuh -- kernel-parameter and workspace structures of libsv.
#pragma once

#include "sv_dev.cuh"

namespace sv {

// A sequence whose correction must be drawn from the residual [p - q]_+ of
// one row pair, after the fast path proved every acceptance decision.
struct __align__(16) ResidEntry {
    int b;          // sequence
    int h;          // position of the first rejection (row index)
    int need_lq;    // 1: the q row's log-sum-exp is not known yet (Packed-SS)
    int bonus;      // 1: every draft was accepted; the draw is the bonus token,
                    // the Gumbel-max of x/Tp over the p row (no q row)
    const char *prow;  // target row at position h
    const char *qrow;  // proposal row at position h
    double Lp, Lq;     // natural log-sum-exps of x/Tp and y/Tq
    double epsp, epsq; // relative error bounds of exp(Lp), exp(Lq)
    double lclo, lchi; // bracket of log c: the residual is [c p - q]_+ (c = 1
                       // but for the modified Cactus rule)
};

// One seed record: the top ids (the ids whose uniform lies in the top 1/256)
// of one piece of a Gumbel-max row, scored before the stream: the piece's
// threshold (best lower end - 1e-9) and its candidates (Cand2 fields).  An
// unused record has threshold -inf and no candidate.
struct __align__(16) SeedRec {
    float thr;
    float hi1, lo1, hi2, lo2, hi3;
    int v1, v2;
};

// A sequence that goes to the fp64 path.
struct __align__(16) RescueEntry {
    int b;
    int kind;       // 0: acceptance decisions, 1: residual draw at position h
    int h;          // kind 1: the rejected position; set for kind 0 by the fp64 path
    int resid;      // the fp64 path draws a residual at position h
    double Lp, Lq;  // fp64 log-sum-exps of the residual pair
    int flags;      // near-threshold decisions found by the fp64 path so far
    int bonus;      // the draw at h is the bonus token (every draft accepted)
    int pad[2];
};

// Per-draft-row results of a Packed-SS proposal, kept for the fp64 path.
struct __align__(16) DraftTmp {
    int z;
    int gflag;
    float q;
    float pad;
};

// Control words in the workspace (all return to zero after each call).
enum : int {
    C_UNIT = 0,       // streaming kernel: next unit
    C_EXIT = 1,       // streaming kernel: finished CTAs
    C_RESID_N = 2,    // residual entries
    C_RESCUE_N = 3,   // rescue entries
    // 4: unused
    C_REXIT = 5,      // residual kernel: finished CTAs
    C_TWORK = 6,      // total-variation kernel: next work item
    C_TEXIT = 7,      // total-variation kernel: finished CTAs
    C_GBAR = 8,       // fp64 kernel: grid barrier arrivals
    C_GGEN = 9,       // fp64 kernel: grid barrier generation
    C_GWORK = 10,     // fp64 kernel: next work item
    C_ABORT = 11,     // fp64 kernel: a barrier timed out
    C_RESCUED = 12,   // running count of rescued sequences (read by the host)
    C_NCTL = 16
};

struct Job {
    int kind, dtype;
    const char *src0;   // target / node / packed logits
    const char *src1;   // drafter logits (sample)
    const char *src2;   // previous drafter logits (packed, T > 0)
    int64_t rs;         // row stride, bytes
    int V, nvec;        // vocabulary; 16-byte vectors per row
    int B, K, N, W;
    int rows_per_seq, parts, part_vecs;
    long long total_units;
    float Tp, Tq;       // temperatures (tree / packed: Tp = T)
    float cp, cq, c1;   // log2(e)/Tp, log2(e)/Tq, log2(e)
    float invTp;        // 1/Tp rounded to fp32 (Gumbel filter)
    double eps_lse;     // relative error bound of exp(L) for streamed log-sum-exps
    double crp, crq, cr1;  // (log2(e)/T) / c for cp, cq, c1 (exact ratios, fp64)
    double rTp, rTq;    // 1/Tp, 1/Tq in fp64
    int amode;          // acceptance rule
    float lam;
    double cactus_emd;  // exp(-lam) (1 - 1e-12): below it, gamma* < 1 (modified Cactus)
    uint64_t seed, iter;
    int eos;
    int force_rescue;
    int max_depth;
    // inputs
    const int32_t *ids, *lens;
    const int64_t *pos_base;
    const int32_t *parent, *node_pos, *node_tok;
    const float *prev_q;
    const int32_t *prev_off, *remaining;
    // outputs
    int32_t *acc, *next, *flags;
    float *p_at, *q_at, *lse_p, *lse_q, *tv;
    int32_t *path_len, *path_nodes, *commit_count;
    uint8_t *match;
    int32_t *commit_len, *committed, *next_draft, *next_len;
    float *next_q, *confidence;
    // SPOT (K_SPOT): L positions per block state, root masks, Phi outputs
    int L;
    const uint64_t *root_mask;
    int32_t *commit_pos, *commit_tok, *state_pos, *state_tok;
    // any-order Packed-SS (K_ANYORDER): window positions, rank order, end
    // position in and out
    const int32_t *win_pos, *order, *end_in;
    int32_t *end_out;
    // workspace
    RowPart *rp;        // [B * rows_per_seq * parts]
    RowStat *rs_stat;   // [B * rows_per_seq]
    unsigned *seq_done; // [B]
    unsigned *ctl;      // [C_NCTL]
    ResidEntry *resid;  // [B]
    RescueEntry *rescue;// [B]
    DraftTmp *dtmp;     // [B * W]
    float *tvpart;      // [B * K * tv_chunks]
    unsigned *tvdone;   // [B * K]
    int tv_chunks;
    double *rpart;      // residual / fp64 scratch
    SeedRec *seeds;     // [gumbel rows * seed_chunks] (see gumbel_rows)
    int seed_chunks;    // seed records per Gumbel-max row
    int seed_span;      // blocks of 256 ids a seed warp lists (the Gumbel-max
                        // rows' blocks laid end to end, split into equal spans)
    uint64_t *smask;    // SPOT: masked positions of every state [B * (N + 1)];
                        // any-order: verify rows needed per sequence [B]
    unsigned *svalid;   // SPOT, any-order: rows to stream per sequence [B]
    int *err;
    const float *gtab;     // [kGTab] G bounds of ordinary ids
    const float *gtop;     // [2 * kGTab] upper, then lower G bounds of top ids by
                           // the top byte of their fine bits (the seed kernel's)
    const uint64_t *skip;  // [kSkipN] skip thresholds of the top-id draws
};

// Row slot bookkeeping shared by the kernels.
__device__ __forceinline__ int seq_len(const Job &j, int b)
{
    if (j.kind == K_TREE || j.kind == K_SPOT)
        return j.N;
    if (!j.lens)
        return j.kind == K_PACKED ? 0 : j.K;
    return __ldg(j.lens + b);
}

// Number of valid row slots of sequence b (clamped lengths).
__device__ __forceinline__ int valid_slots(const Job &j, int b)
{
    switch (j.kind) {
    case K_GREEDY: {
        int n = min(max(seq_len(j, b), 0), j.K);
        return n + 1;
    }
    case K_SAMPLE: {
        int n = min(max(seq_len(j, b), 0), j.K);
        return 2 * n + 1;
    }
    case K_TREE:
        return j.N;
    case K_SPOT:
    case K_ANYORDER:
        return (int)__ldg(j.svalid + b);
    default: {
        int n = min(max(seq_len(j, b), 0), j.K - 1);
        return n + 1 + j.W;
    }
    }
}

__device__ __forceinline__ bool slot_valid(const Job &j, int b, int slot)
{
    switch (j.kind) {
    case K_GREEDY:
        return slot <= min(max(seq_len(j, b), 0), j.K);
    case K_SAMPLE: {
        int n = min(max(seq_len(j, b), 0), j.K);
        return slot <= n || (slot > j.K && slot - j.K - 1 < n);
    }
    case K_TREE:
        return true;
    case K_SPOT:
        return ((__ldg(j.smask + (int64_t)b * (j.N + 1) + slot / j.L) >> (slot % j.L)) & 1ull) != 0;
    case K_ANYORDER: {
        const int u = min(max(seq_len(j, b), 0), j.W);
        return slot < (int)__ldg(j.smask + b) || (slot >= j.K && slot - j.K < u);
    }
    default: {
        int n = min(max(seq_len(j, b), 0), j.K - 1);
        return slot <= n || slot >= j.K;
    }
    }
}

__device__ __forceinline__ const char *slot_row(const Job &j, int b, int slot)
{
    switch (j.kind) {
    case K_GREEDY:
        return j.src0 + ((int64_t)b * (j.K + 1) + slot) * j.rs;
    case K_SAMPLE:
        return slot <= j.K ? j.src0 + ((int64_t)b * (j.K + 1) + slot) * j.rs
                           : j.src1 + ((int64_t)b * j.K + (slot - j.K - 1)) * j.rs;
    case K_TREE:
        return j.src0 + ((int64_t)b * j.N + slot) * j.rs;
    case K_SPOT:  // slot = state * L + position
        return j.src0 + ((int64_t)b * (j.N + 1) * j.L + slot) * j.rs;
    case K_ANYORDER:
        return j.src0 + ((int64_t)b * (j.K + j.W) + slot) * j.rs;
    default:
        return j.src0 + ((int64_t)b * (j.K + j.W) + slot) * j.rs;
    }
}

__device__ __forceinline__ int64_t pos0_of(const Job &j, int b)
{
    return j.pos_base ? __ldg(j.pos_base + b) : 0;
}

// Gumbel-max rows of the streaming pass: per sequence, the W proposal rows
// of a Packed-SS step at T > 0; every node row of a tree at T > 0; every
// (state, position) row of a SPOT call at T > 0.  Row k of sequence b has
// index b * gumbel_rows(j) + k.  (The bonus draw of a sampling call or a
// Packed-SS step is needed only when every draft is accepted; the residual
// pass takes it then, from the bonus row alone.)
__host__ __device__ __forceinline__ int gumbel_rows(const Job &j)
{
    switch (j.kind) {
    case K_PACKED: return j.Tp != 0.f ? j.W : 0;
    case K_TREE: return j.Tp != 0.f ? j.N : 0;
    case K_SPOT: return j.Tp != 0.f ? (j.N + 1) * j.L : 0;
    default: return 0;
    }
}

// Row slot of Gumbel-max row k of a sequence.
__device__ __forceinline__ int gumbel_slot(const Job &j, int k)
{
    return j.kind == K_PACKED ? j.K + k : k;  // proposal rows; tree and SPOT rows
}

// Index k of the Gumbel-max row in `slot`, or -1 when that row carries no
// Gumbel-max.
__device__ __forceinline__ int gumbel_index(const Job &j, int slot)
{
    switch (j.kind) {
    case K_PACKED: return (j.Tp != 0.f && slot >= j.K) ? slot - j.K : -1;
    case K_TREE:
    case K_SPOT: return j.Tp != 0.f ? slot : -1;
    default: return -1;
    }
}

}  // namespace sv
