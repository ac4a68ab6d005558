// sv_pass.cu -- the streaming kernel of libsv.
//
// One persistent CTA per SM streams logit rows from HBM exactly once.  A
// producer warp takes work units (a contiguous part of one row) from a global
// counter and moves them into a shared-memory ring with bulk copies
// (cp.async.bulk, completion on an mbarrier); the consumer warps compute the
// row statistics the verify rules need:
//   - max / lowest-index argmax                 (greedy rules, [PackedSS] eq. 1)
//   - sum 2^(x c - e) for log-sum-exp at T      (p, q of [PackedSS] §2.2, [SPOT] eq. 2)
//   - Gumbel-max with exact fp64 candidates     ([SPOT] eq. 4, eqs. 5-7)
// The producer prepares each unit's row mode one unit ahead, so the consumer
// warps read everything they need from shared memory.  Consumer warps never
// wait for one another or for global memory: at the end of a unit each drops
// its warp-reduced partial into a shared-memory unit slot, and the Gumbel
// threshold of a unit is shared through another slot.  A finalizer warp
// merges the partials into the unit's record, counts records per sequence,
// and runs a sequence's decision step (prefix scan, stopping index, tree
// path) once its last record is in, so the ring never waits for any of it.
// Each entry-point kind has its own kernel instance holding only the row
// modes that kind uses.
#include <math.h>

#include "sv_common.cuh"

namespace sv {

constexpr int kFinQ = 32;      // decision steps queued per CTA
constexpr int kUnitSlots = 8;  // units whose partials wait for the finalizer
constexpr int kGQ = 64;        // queued Gumbel vectors per consumer warp
constexpr int kSeedCap = 2048; // top ids gathered per seeding round

struct RowMode {
    int mode;
    float c1, c2, invT;
    double T;
    uint64_t key;
};

struct StageMeta {
    int unit;         // -1: end of work
    int nv;           // 16-byte vectors in this stage
    int vbase;        // row vector index of the stage's first vector
    int first, last;  // first / last stage of its unit
    int lu;           // this CTA's running unit number
    int b;            // sequence of the unit
    unsigned expect;  // records that complete sequence b
    int xid;          // vocabulary id whose logit the unit records (-1: none)
    int vend;         // end (vector index) of the unit's part of the row
    const char *row;  // the unit's logit row
    // first stage: the next unit this CTA streams, if it carries a Gumbel-max
    // (its top ids are prefetched while this unit streams)
    const char *nrow;
    uint64_t nkey;
    int nrec, nlo, nhi, npad;
    RowMode rm;       // row mode of the unit
};

// The planner warp's plan of the units this CTA streams next, handed to the
// producer through a small queue: everything the producer needs, so that no
// global-memory latency sits between two units' copies.
constexpr int kPlanQ = 8;
struct PlanEntry {
    int kind;         // 0: part of a row, -1: no more units
    int rec, b;       // record; sequence
    unsigned expect;  // records that complete sequence b
    int xid;          // vocabulary id whose logit the unit records (-1: none)
    int vs, ve;       // the unit's vectors [vs, ve) of the row
    int pad;
    const char *row;  // the unit's logit row
    RowMode rm;
};

// One consumer warp's share of a unit.
struct WarpPart {
    float m;
    int amax;
    float e1, s1, e2, s2;
    float hi1, lo1, hi2, lo2, hi3;
    int v1, v2;
    float xd;  // logit at the draft token (the one lane that held it), else NaN
    int pad[2];
};

struct PassShared {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    StageMeta meta[kStages];
    // Gumbel threshold of local unit lu, in slot lu % kStages: the ring holds
    // stages of at most kStages - 1 other units when a unit starts, so no warp
    // still uses the slot that unit takes over.
    uint32_t thr[kStages];
    volatile int abort;
    // Gumbel vectors that passed level 1, per consumer warp: raw data and
    // the vector's index in the row
    uint4 gqd[kConsumerWarps][kGQ];
    uint32_t gqv[kConsumerWarps][kGQ];
    uint64_t skip[kSkipN];   // skip thresholds of the top-id draws
    // unit slots: consumer warps write their partials and arrive on ubar; the
    // finalizer merges them and arrives on ufree
    uint64_t ubar[kUnitSlots];
    uint64_t ufree[kUnitSlots];
    WarpPart up[kUnitSlots][kConsumerWarps];
    int uunit[kUnitSlots], ub[kUnitSlots];
    unsigned uexpect[kUnitSlots];
    // top ids of a unit being seeded, and their logits' 32-bit words (copied
    // ahead, one unit early); buffer lu & 1 belongs to local unit lu
    uint32_t seed_ids[2][kSeedCap];
    uint32_t seed_x[2][kSeedCap];
    int seed_cnt[2];     // ids listed in a buffer
    int seed_n;
    int seed_more;
    // barrier among the consumer warps (see csync) and each warp's phase
    uint64_t csync;
    uint32_t cph[kConsumerWarps];
    PlanEntry plan[kPlanQ];
    uint64_t plan_full[kPlanQ], plan_empty[kPlanQ];
    volatile int nunits;     // units this CTA streamed (set when the producer is done)
    volatile int prod_done;
    int todo[kFinQ];         // sequences whose decision step is due (finalizer only)
    int fin_qh, fin_qt;      // decision steps the finalizer left for the whole CTA
};

// Per-sequence values a unit's bookkeeping needs, loaded one unit ahead.
struct UnitPre {
    int len;       // draft length as given (unclamped)
    int64_t p0;    // absolute position of the sequence's first row
    int np;        // tree: position of the node (T > 0)
    int ida, idb;  // draft tokens of the two slots a light unit can map to
    uint64_t smask;   // SPOT: masked positions of the unit's state
    unsigned svalid;  // SPOT: rows the tree streams
};

// Unit order.  Rows that carry a Gumbel-max (a few times the work of a plain
// row) are streamed first, H per sequence, so that the last units of the pass
// are light ones and CTAs finish together; the other rows follow sequence by
// sequence.  A unit is one part of one row.
__device__ __forceinline__ int heavy_rows(const Job &j)
{
    if (j.kind == K_SAMPLE)
        return 1;  // the bonus row
    if (j.kind == K_PACKED && j.Tp != 0.f)
        return 1 + j.W;  // the bonus row and the proposal rows
    return 0;
}

// Sequence of unit u (needs no per-sequence data).
__device__ __forceinline__ int unit_seq(const Job &j, long long u)
{
    const int H = heavy_rows(j);
    const long long nh = (long long)j.B * H * j.parts;
    if (u < nh)
        return (int)(u / ((long long)H * j.parts));
    return (int)((u - nh) / ((long long)(j.rows_per_seq - H) * j.parts));
}

// Row slot and part of unit u of sequence b with clamped length n.
__device__ __forceinline__ void unit_map(const Job &j, long long u, int b, int n, int &slot,
                                         int &part)
{
    const int H = heavy_rows(j);
    const long long nh = (long long)j.B * H * j.parts;
    if (u < nh) {
        const long long rem = u - (long long)b * H * j.parts;
        const int r = (int)(rem / j.parts);
        part = (int)(rem - (long long)r * j.parts);
        slot = r == 0 ? n : j.K + r - 1;
    } else {
        const long long rem = (u - nh) - (long long)b * (j.rows_per_seq - H) * j.parts;
        const int r = (int)(rem / j.parts);
        part = (int)(rem - (long long)r * j.parts);
        slot = (H > 0 && r >= n) ? r + 1 : r;
    }
}

// Draft position whose token the row in `slot` is tested on (sample: target
// and drafter rows; Packed-SS at T > 0: verify rows), or -1.
__device__ __forceinline__ int draft_pos(const Job &j, int slot)
{
    if (j.kind == K_SAMPLE)
        return slot < j.K ? slot : (slot > j.K ? slot - j.K - 1 : -1);
    if (j.kind == K_PACKED && j.Tp != 0.f)
        return slot < j.K - 1 ? slot : -1;
    return -1;
}

__device__ __forceinline__ int draft_token(const Job &j, int b, int slot)
{
    const int pos = draft_pos(j, slot);
    if (pos < 0 || !j.ids)
        return -1;
    const int per = j.kind == K_PACKED ? j.K - 1 : j.K;
    return __ldg(j.ids + (int64_t)b * per + pos);
}

__device__ __forceinline__ UnitPre unit_prefetch(const Job &j, long long u)
{
    UnitPre p{0, 0, 0, -1, -1, 0ull, 0u};
    if (u >= j.total_units)
        return p;
    const int b = unit_seq(j, u);
    const int H = heavy_rows(j);
    const long long nh = (long long)j.B * H * j.parts;
    if (H > 0 && u >= nh) {
        // a light unit's slot is r or r + 1 (the bonus slot is skipped)
        const long long rem = (u - nh) - (long long)b * (j.rows_per_seq - H) * j.parts;
        const int r = (int)(rem / j.parts);
        p.ida = draft_token(j, b, r);
        p.idb = draft_token(j, b, r + 1);
    }
    p.len = j.kind == K_TREE ? j.N : (j.lens ? __ldg(j.lens + b) : (j.kind == K_PACKED ? 0 : j.K));
    p.p0 = j.pos_base ? __ldg(j.pos_base + b) : 0;
    if (j.kind == K_TREE && j.Tp != 0.f) {
        int slot, part;
        unit_map(j, u, b, 0, slot, part);
        p.np = __ldg(j.node_pos + (int64_t)b * j.N + slot);
    }
    if (j.kind == K_SPOT) {
        int slot, part;
        unit_map(j, u, b, 0, slot, part);
        p.smask = __ldg(j.smask + (int64_t)b * (j.N + 1) + slot / j.L);
        p.svalid = __ldg(j.svalid + b);
    }
    if (j.kind == K_ANYORDER) {
        p.smask = __ldg(j.smask + b);  // verify rows needed
        p.svalid = __ldg(j.svalid + b);
    }
    return p;
}

__device__ __forceinline__ int clamp_n(const Job &j, int len)
{
    const int hi = (j.kind == K_PACKED) ? j.K - 1 : j.K;
    return min(max(len, 0), hi);
}

// Row slots that exist for a sequence of clamped length n.
__device__ __forceinline__ int valid_slots_n(const Job &j, int n)
{
    switch (j.kind) {
    case K_GREEDY: return n + 1;
    case K_SAMPLE: return 2 * n + 1;
    case K_TREE: return j.N;
    default: return n + 1 + j.W;
    }
}
__device__ __forceinline__ bool slot_valid_n(const Job &j, int n, int slot)
{
    switch (j.kind) {
    case K_GREEDY: return slot <= n;
    case K_SAMPLE: return slot <= n || (slot > j.K && slot - j.K - 1 < n);
    case K_TREE: return true;
    default: return slot <= n || slot >= j.K;
    }
}

__device__ __forceinline__ RowMode row_mode(const Job &j, int b, int slot, int n, int64_t p0,
                                            int np)
{
    RowMode r;
    r.mode = 0;
    r.c1 = r.c2 = r.invT = 0.f;
    r.T = 1.0;
    r.key = 0;
    switch (j.kind) {
    case K_GREEDY:
        r.mode = M_ARGMAX;
        break;
    case K_SAMPLE:
        r.mode = M_LSE;
        if (slot <= j.K) {
            r.c1 = j.cp;
            if (slot == n) {  // bonus row: Gumbel-max of x_n / Tp
                r.mode |= M_GUMBEL;
                r.invT = j.invTp;
                r.T = j.Tp;
                r.key = rng_key(j.seed, kSample, (uint64_t)b, p0 + n, 0);
            }
        } else {
            r.c1 = j.cq;
        }
        break;
    case K_TREE:
        if (j.Tp == 0.f) {
            r.mode = M_ARGMAX;
        } else {
            r.mode = M_GUMBEL;
            r.invT = j.invTp;
            r.T = j.Tp;
            r.key = rng_key(j.seed, kTree, (uint64_t)b, p0 + np, 0);
        }
        break;
    case K_ANYORDER:
        // verify rows: the argmax; proposal rows: the argmax and the
        // log-sum-exp at temperature 1 of their confidence
        if (slot < j.K) {
            r.mode = M_ARGMAX;
        } else {
            r.mode = M_ARGMAX | M_LSE;
            r.c1 = j.c1;
        }
        break;
    case K_SPOT:
        // the confidence max_v softmax(x)_v needs the row max and its
        // log-sum-exp at temperature 1; the token, the argmax (T = 0) or the
        // coupled-noise Gumbel-max at the row's absolute position (T > 0)
        r.c1 = j.c1;
        if (j.Tp == 0.f) {
            r.mode = M_ARGMAX | M_LSE;
        } else {
            r.mode = M_GUMBEL | M_LSE | M_MAX;
            r.invT = j.invTp;
            r.T = j.Tp;
            r.key = rng_key(j.seed, kTree, (uint64_t)b, p0 + slot % j.L, 0);
        }
        break;
    default:  // Packed-SS
        if (slot < j.K) {
            if (j.Tp == 0.f) {
                r.mode = M_ARGMAX;
            } else {
                r.mode = M_LSE;
                r.c1 = j.cp;
                if (slot == n) {
                    r.mode |= M_GUMBEL;
                    r.invT = j.invTp;
                    r.T = j.Tp;
                    r.key = rng_key(j.seed, kSample, (uint64_t)b, p0 + n, 0);
                }
            }
        } else {
            const int jj = slot - j.K;
            if (j.Tp == 0.f) {
                r.mode = M_ARGMAX | M_LSE;  // confidence needs the T = 1 normaliser
                r.c1 = j.c1;
            } else {
                r.mode = M_GUMBEL | M_LSE | M_MAX;
                r.c1 = j.cp;
                r.invT = j.invTp;
                r.T = j.Tp;
                r.key = rng_key(j.seed, kDraft, (uint64_t)b, p0 + jj, j.iter);
                if (j.Tp != 1.f) {
                    r.mode |= M_LSE2;
                    r.c2 = j.c1;
                }
            }
        }
    }
    return r;
}

// Everything the producer needs to stream unit u (u < total_units).
struct UnitInfo {
    int rec;  // record index of the unit: (b * rows_per_seq + slot) * parts + part
    int b, slot, part;
    bool valid;
    unsigned expect;
    int xid;  // draft token whose logit the unit records, or -1
    RowMode rm;
};

__device__ __forceinline__ UnitInfo unit_info(const Job &j, long long u, const UnitPre &p)
{
    UnitInfo i;
    i.b = unit_seq(j, u);
    const int n = j.kind == K_TREE ? j.N : clamp_n(j, p.len);
    unit_map(j, u, i.b, n, i.slot, i.part);
    i.rec = (int)(((long long)i.b * j.rows_per_seq + i.slot) * j.parts + i.part);
    i.xid = -1;
    const int H = heavy_rows(j);
    if (H > 0 && u >= (long long)j.B * H * j.parts) {
        const int pos = draft_pos(j, i.slot);
        if (pos >= 0 && pos < n) {
            const long long rem =
                (u - (long long)j.B * H * j.parts) - (long long)i.b * (j.rows_per_seq - H) * j.parts;
            const int d = (i.slot == (int)(rem / j.parts)) ? p.ida : p.idb;
            if (d < 0 || d >= j.V)
                latch(j.err, SV_ERR_DEVICE_BOUNDS);  // tested as probability 0
            else
                i.xid = d;
        }
    }
    if (j.kind == K_SPOT) {
        i.valid = ((p.smask >> (i.slot % j.L)) & 1ull) != 0;
        i.expect = p.svalid * (unsigned)j.parts;
    } else if (j.kind == K_ANYORDER) {
        const int u = min(max(p.len, 0), j.W);
        i.valid = i.slot < (int)p.smask || (i.slot >= j.K && i.slot - j.K < u);
        i.expect = p.svalid * (unsigned)j.parts;
    } else {
        i.valid = slot_valid_n(j, n, i.slot);
        i.expect = (unsigned)(valid_slots_n(j, n) * j.parts);
    }
    i.rm = row_mode(j, i.b, i.slot, n, p.p0, p.np);
    return i;
}

// Gumbel part of a thread's state (passed by value to the out-of-line queue
// screen, so that the state stays in registers).
struct GState {
    Cand2 c;           // candidates
    float lomax;       // best lower end seen
    float thr, thrS;   // level-2 and level-1 thresholds
};

// Per-thread running state of one unit.
struct TState {
    float e1, e2;      // integer reference exponents of the sums (-inf: none yet)
    float2 acc1, acc2; // sums of 2^fl(x c - e), as fp32 pairs
    float mx;          // running max
    int amax;
    GState g;
    float pub;         // threshold last published to the CTA
    int gqn;           // groups in this warp's queue (warp-uniform)
    float xd;          // logit at the unit's draft token (its owner thread), else NaN
};

__device__ __forceinline__ void tstate_init(TState &s)
{
    s.e1 = s.e2 = -INFINITY;
    s.acc1 = s.acc2 = make_float2(0.f, 0.f);
    s.mx = -INFINITY;
    s.amax = 0x7FFFFFFF;
    s.g.c.init();
    s.g.lomax = -INFINITY;
    s.g.thr = s.g.thrS = s.pub = -INFINITY;
    s.gqn = 0;
    s.xd = __int_as_float(0x7FC00000);
}

__device__ __forceinline__ void raise_thr(GState &s, float t)
{
    if (t > s.thr) {
        s.thr = t;
        s.thrS = level1_thr(t);
    }
}

// Level 2: fp32 interval of x/T + G; candidates whose upper end reaches the
// threshold are kept, and the best lower end raises the threshold (anything
// below it - 1e-9 can neither win nor tie within 1e-9).
__device__ __forceinline__ void gumbel_level2(float x, uint32_t v, bool top, GState &s,
                                              const RowMode &rm)
{
    const float2 iv = logit_interval_at(x, rm.invT, rm.key, v, top);
    const float lo = iv.x, hi = iv.y;
    if (hi < s.thr)
        return;
    s.c.add(lo, hi, (int)v);
    if (lo > s.lomax) {
        s.lomax = lo;
        raise_thr(s, __fsub_rd(lo, 1e-9f));
    }
}

// ---------------------------------------------------------------------------
// One stage = one chunk: each consumer thread holds kVecsPerThread vectors.
// Vectors past the end of the stage read as -inf, which adds nothing to a
// sum and never wins a max.
// ---------------------------------------------------------------------------
using Chunk = uint4[kVecsPerThread];

template <typename In>
__device__ __forceinline__ void load_chunk(const uint4 *__restrict__ st, int nv, Chunk &q)
{
    const int t = threadIdx.x;
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k) {
        int idx = t + k * kConsumers;
        q[k] = idx < nv ? st[idx] : VecTraits<In>::neg_inf_vec();
    }
}

template <typename In>
__device__ __forceinline__ float chunk_max(const Chunk &q)
{
    using VT = VecTraits<In>;
    uint32_t pm = VT::pmax(q[0]);
#pragma unroll
    for (int k = 1; k < kVecsPerThread; ++k)
        pm = VT::bmax(pm, VT::pmax(q[k]));
    return VT::hi_of(pm);
}

// Sum of 2^fl(x c - e) over the chunk: one packed FFMA per two elements, one
// ex2 per element, a packed-add tree.
template <typename In>
__device__ __forceinline__ float2 lse_terms(const Chunk &q, float c, float e)
{
    using VT = VecTraits<In>;
    constexpr int P = VT::P;  // element pairs per vector
    float2 t[kVecsPerThread * P];
    const float2 cc = make_float2(c, c), ne = make_float2(-e, -e);
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k)
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const float2 y = fma2(VT::pair(q[k], i), cc, ne);
            t[k * P + i] = make_float2(ex2f(y.x), ex2f(y.y));
        }
    // pairwise tree over any number of terms (depth ceil(log2 N))
    constexpr int N = kVecsPerThread * P;
#pragma unroll
    for (int w = 1; w < N; w <<= 1)
#pragma unroll
        for (int i = 0; i + w < N; i += 2 * w)
            t[i] = add2(t[i], t[i + w]);
    return t[0];
}

// Adds the chunk to one log-sum-exp accumulator.  The first chunk with an
// element sets the reference to its max, rounded up to an integer; later, a
// partial sum of 2^20 or more moves the reference up to the chunk max and
// rescales the accumulator exactly.
template <typename In>
__device__ __forceinline__ void lse_chunk(const Chunk &q, float c, float &e, float2 &acc)
{
    if (e == -INFINITY) {
        const float cm = chunk_max<In>(q);
        if (cm == -INFINITY)
            return;  // no element yet
        e = ceilf(__fmul_ru(cm, c));
    }
    float2 part = lse_terms<In>(q, c, e);
    if (!(part.x + part.y < 0x1p20f)) {
        const float cm = chunk_max<In>(q);
        if (cm == -INFINITY) {
            part = make_float2(0.f, 0.f);
        } else {
            const float en = fmaxf(e, ceilf(__fmul_ru(cm, c)));
            if (e > -INFINITY) {
                const float sc = pow2_int(e - en);
                acc.x *= sc;
                acc.y *= sc;
            }
            e = en;
            part = lse_terms<In>(q, c, e);
        }
    }
    acc = add2(acc, part);
}

// Running max, and with ARG its lowest index: the first vector whose max is
// the chunk max, then the first element of it that equals it (predicated
// selects, no search loop).
template <typename In, bool ARG>
__device__ __forceinline__ void max_chunk(const Chunk &q, int vbase, TState &s)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    float vm[kVecsPerThread];
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k)
        vm[k] = VT::hi_of(VT::pmax(q[k]));
    float cm = vm[0];
#pragma unroll
    for (int k = 1; k < kVecsPerThread; ++k)
        cm = fmaxf(cm, vm[k]);
    if (ARG && cm > s.mx) {
        int kk = kVecsPerThread - 1;
        uint4 v = q[kVecsPerThread - 1];
#pragma unroll
        for (int k = kVecsPerThread - 2; k >= 0; --k)
            if (vm[k] == cm) {
                kk = k;
                v = q[k];
            }
        int ii = E - 1;
#pragma unroll
        for (int i = E - 2; i >= 0; --i)
            if (VT::elem(v, i) == cm)
                ii = i;
        s.amax = (vbase + (int)threadIdx.x + kk * kConsumers) * E + ii;
    }
    s.mx = fmaxf(s.mx, cm);
}

// Per-id screen of the queued vectors, 32 at a time, a vector per lane: its
// top ids are skipped (the seeding warp scored every top id of the unit);
// an ordinary id is bounded by the top byte of its fine bits, and survivors
// get the fp32 interval of level 2.
template <typename In>
__device__ __noinline__ GState gumbel_flush(const uint4 *__restrict__ qd,
                                            const uint32_t *__restrict__ qv, int n, GState s,
                                            const RowMode &rm, const float *__restrict__ gt,
                                            const uint64_t *__restrict__ skip)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    __syncwarp();
    for (int i = (int)(threadIdx.x & 31); i < n; i += 32) {
        const uint4 d = qd[i];
        const uint32_t v0 = qv[i] * E;
        const uint32_t tm = top_mask(rm.key, v0 >> 8, (int)(v0 & 255u), E, skip);
#pragma unroll 1
        for (int e = 0; e < E; ++e) {
            if ((tm >> e) & 1u)
                continue;
            const uint32_t v = v0 + e;
            const float x = VT::elem(d, e);
            const uint64_t m = fine52(rm.key, v);
            if (fmaf(x, rm.invT, gt[(int)(m >> 44)]) >= s.thrS)
                gumbel_level2(x, v, false, s, rm);
        }
    }
    __syncwarp();
    return s;
}

// Level 1 on whole vectors: an ordinary id's G stays below the table's last
// entry, so a vector is queued only if its largest logit can reach the
// threshold with that bound.  The queue is compacted with a ballot, so a warp
// does not diverge per vector.
template <typename In>
__device__ __forceinline__ void gumbel_chunk(const Chunk &q, int nv, int vbase, TState &s,
                                             const RowMode &rm, const float *__restrict__ gt,
                                             const uint64_t *__restrict__ skip, PassShared &sm)
{
    using VT = VecTraits<In>;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const float gmax = g_ordinary_max(gt);
    uint4 *qd = sm.gqd[w];
    uint32_t *qv = sm.gqv[w];
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k) {
        const int idx = t + k * kConsumers;
        const bool pass =
            fmaf(VT::hi_of(VT::pmax(q[k])), rm.invT, gmax) >= s.g.thrS && idx < nv;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, pass);
        if (bal) {
            if (pass) {
                const int r = s.gqn + __popc(bal & ((1u << lane) - 1u));
                qd[r] = q[k];
                qv[r] = (uint32_t)(vbase + idx);
            }
            s.gqn += __popc(bal);
            if (s.gqn > kGQ - 32) {
                s.g = gumbel_flush<In>(qd, qv, s.gqn, s.g, rm, gt, skip);
                s.gqn = 0;
            }
        }
    }
}

template <typename In, int MODE>
__device__ __forceinline__ void do_chunk(const uint4 *__restrict__ st, int nv, int vbase, TState &s,
                                         const RowMode &rm, const float *__restrict__ gt,
                                         PassShared &sm)
{
    Chunk q;
    load_chunk<In>(st, nv, q);
    if (MODE & (M_ARGMAX | M_MAX))
        max_chunk<In, (MODE & M_ARGMAX) != 0>(q, vbase, s);
    if (MODE & M_LSE)
        lse_chunk<In>(q, rm.c1, s.e1, s.acc1);
    if (MODE & M_LSE2)
        lse_chunk<In>(q, rm.c2, s.e2, s.acc2);
    if (MODE & M_GUMBEL)
        gumbel_chunk<In>(q, nv, vbase, s, rm, gt, sm.skip, sm);
}

// ---------------------------------------------------------------------------
// Decision steps (one warp; lane = draft position).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void check_len(const Job &j, int b)
{
    int n = seq_len(j, b);
    int hi = (j.kind == K_PACKED) ? j.K - 1 : j.K;
    if (n < 0 || n > hi)
        latch(j.err, SV_ERR_DEVICE_BOUNDS);
}

static __device__ __noinline__ void fin_greedy(const Job &j, int b)
{
    const int lane = threadIdx.x & 31;
    int n = clamp_len(j, b);
    if (lane == 0) check_len(j, b);
    bool match = false;
    if (lane < n) {
        RowM r = merge_row(j, b, lane, 1.0, 1.0);
        int d = __ldg(j.ids + (int64_t)b * j.K + lane);
        match = (d == r.amax);
    }
    unsigned mm = __ballot_sync(0xFFFFFFFFu, match);
    int h = (~mm == 0u) ? 32 : __ffs(~mm) - 1;
    h = min(h, n);
    if (lane == 0) {
        RowM r = merge_row(j, b, h, 1.0, 1.0);
        j.acc[b] = h;
        j.next[b] = r.amax;
    }
}

static __device__ __noinline__ void fin_sample(const Job &j, int b)
{
    const int lane = threadIdx.x & 31;
    // Every load of the step is independent of the draft length, so they are
    // issued together: the length, the position base and the unit records of
    // target rows 0..K (lane i) and drafter rows (lane i < K).  Records of rows
    // beyond the length are not used.  The logits at the draft tokens were
    // recorded during the stream.
    const int len = seq_len(j, b);
    const int64_t p0 = pos0_of(j, b);
    RowM rp, rq;
    rp.gc.init();
    rq.gc.init();
    if (lane <= j.K) rp = merge_row(j, b, lane, j.crp, 1.0);
    if (lane < j.K) rq = merge_row(j, b, j.K + 1 + lane, j.crq, 1.0);
    const int n = min(max(len, 0), j.K);
    if (lane == 0 && (len < 0 || len > j.K)) latch(j.err, SV_ERR_DEVICE_BOUNDS);
    bool acc = false, und = false;
    double Lp = 0, Lq = 0;
    double lclo = 0.0, lchi = 0.0;  // bracket of log c (modified Cactus residual)
    const double ep = j.eps_lse, eq = j.eps_lse;
    if (lane < n) {
        Lp = rp.L1a;
        Lq = rq.L1a;
        double lp = -INFINITY, lq = 0.0;
        if (!isnan(rp.xd) && !isnan(rq.xd)) {  // NaN: the draft token was out of range
            lp = (double)rp.xd * j.rTp - Lp;
            lq = (double)rq.xd * j.rTq - Lq;
        }
        // r in fp32 (exp_fast: 2^-21); x * (1/T) for x / T: 1e-13 of slack
        double r = (double)exp_fast(lp - lq);
        double rel = 1.01 * (ep + eq) + 0x1p-21 + 1e-13;
        double alo = alpha_of(j.amode, r * (1.0 - rel), j.lam);
        double ahi = alpha_of(j.amode, r * (1.0 + rel), j.lam);
        if (j.amode == SV_LENIENT_CACTUS && r * (1.0 - rel) < 1.0) {
            // gamma* grows with p: bracket p and q, then gamma* at both ends
            // of p's bracket; alpha = gamma* / q and c = (1 - gamma*)/(1 - p)
            const double plo = exp(lp - 1.01 * ep - 1e-13), phi = exp(lp + 1.01 * ep + 1e-13);
            const double qlo = exp(lq - 1.01 * eq - 1e-13), qhi = exp(lq + 1.01 * eq + 1e-13);
            double g0, g1, g2, g3;
            const bool ok = cactus_bracket(plo, (double)j.lam, &g0, &g1) &&
                            cactus_bracket(phi, (double)j.lam, &g2, &g3);
            alo = ok ? fmin(1.0, g0 / qhi) : 0.0;
            ahi = ok ? fmin(1.0, g3 / qlo) : 1.0;
            lclo = (g3 < 1.0) ? log1p(-g3) - log1p(-plo) : -INFINITY;
            lchi = log1p(-g0) - log1p(-phi);
        }
        double u = uniform_at(rng_key(j.seed, kAccept, (uint64_t)b, p0 + lane, 0), 0, j.skip);
        acc = u < alo - kFlagEps;
        bool rej = u >= ahi + kFlagEps;
        und = !(acc || rej) || j.force_rescue;
        if (j.force_rescue)
            acc = false;
        if (j.p_at) j.p_at[(int64_t)b * j.K + lane] = exp_fast(lp);
        if (j.q_at) j.q_at[(int64_t)b * j.K + lane] = exp_fast(lq);
        if (j.lse_p) j.lse_p[(int64_t)b * (j.K + 1) + lane] = (float)Lp;
        if (j.lse_q) j.lse_q[(int64_t)b * j.K + lane] = (float)Lq;
        RowStat *sp = j.rs_stat + (int64_t)b * j.rows_per_seq + lane;
        sp->L1 = Lp;
        sp->L2 = rp.L2c1;
        sp->m = rp.m;
        sp->eps = (float)ep;
        RowStat *sq = j.rs_stat + (int64_t)b * j.rows_per_seq + j.K + 1 + lane;
        sq->L1 = Lq;
        sq->L2 = rq.L2c1;
        sq->m = rq.m;
        sq->eps = (float)eq;
    } else if (lane < j.K) {
        const float nan = __int_as_float(0x7FC00000);
        if (j.p_at) j.p_at[(int64_t)b * j.K + lane] = nan;
        if (j.q_at) j.q_at[(int64_t)b * j.K + lane] = nan;
        if (j.lse_q) j.lse_q[(int64_t)b * j.K + lane] = nan;
        if (j.tv) j.tv[(int64_t)b * j.K + lane] = nan;
        if (j.lse_p) j.lse_p[(int64_t)b * (j.K + 1) + lane + 1] = nan;
    }
    unsigned am = __ballot_sync(0xFFFFFFFFu, acc);
    unsigned um = __ballot_sync(0xFFFFFFFFu, und);
    int f = (~am == 0u) ? 32 : __ffs(~am) - 1;
    f = min(f, n);  // first position not proved accepted
    unsigned upto = (f >= 31) ? 0xFFFFFFFFu : ((2u << f) - 1u);
    bool rescue = (um & upto) != 0u || j.force_rescue;
    double Lph = __shfl_sync(0xFFFFFFFFu, Lp, f & 31);
    double Lqh = __shfl_sync(0xFFFFFFFFu, Lq, f & 31);
    double eph = __shfl_sync(0xFFFFFFFFu, ep, f & 31);
    double eqh = __shfl_sync(0xFFFFFFFFu, eq, f & 31);
    const double lcloh = __shfl_sync(0xFFFFFFFFu, lclo, f & 31);
    const double lchih = __shfl_sync(0xFFFFFFFFu, lchi, f & 31);
    // bonus row n (always valid): its Gumbel-max with key (SAMPLE, pos + n),
    // resolved by the lane that holds its record
    GRes g = resolve_lanes(j, row_ptr(j, b, lane <= j.K ? lane : 0),
                           rng_key(j.seed, kSample, (uint64_t)b, p0 + lane, 0), (double)j.Tp,
                           j.invTp, rp.gc, lane == n);
    const int gbv = __shfl_sync(0xFFFFFFFFu, g.v, n);
    const int gbf = __shfl_sync(0xFFFFFFFFu, g.flag, n);
    const double Lb = __shfl_sync(0xFFFFFFFFu, rp.L1a, n);
    const float mb = __shfl_sync(0xFFFFFFFFu, rp.m, n);
    if (lane == 0) {
        if (j.lse_p) j.lse_p[(int64_t)b * (j.K + 1) + n] = (float)Lb;
        RowStat *sb = j.rs_stat + (int64_t)b * j.rows_per_seq + n;
        sb->L1 = Lb;
        sb->m = mb;
        sb->gidx = gbv;
        sb->gflag = gbf;
        if (rescue) {
            unsigned e = atomicAdd(j.ctl + C_RESCUE_N, 1u);
            j.rescue[e].b = b;
            j.rescue[e].kind = 0;
            j.rescue[e].h = 0;
        } else if (f == n) {
            j.acc[b] = n;
            j.next[b] = gbv;
            if (j.flags) j.flags[b] = gbf;
        } else {
            j.acc[b] = f;
            unsigned e = atomicAdd(j.ctl + C_RESID_N, 1u);
            ResidEntry re;
            re.b = b;
            re.h = f;
            re.need_lq = 0;
            re.pad = 0;
            re.prow = row_ptr(j, b, f);
            re.qrow = row_ptr(j, b, j.K + 1 + f);
            re.Lp = Lph;
            re.Lq = Lqh;
            re.epsp = eph;
            re.epsq = eqh;
            re.lclo = lcloh;
            re.lchi = lchih;
            j.resid[e] = re;
        }
    }
}

// Value v held for node a (lane a mod 32, half a div 32) by a warp holding
// nodes lane and lane + 32.
__device__ __forceinline__ int node_val(int v0, int v1, int a)
{
    const int x0 = __shfl_sync(0xFFFFFFFFu, v0, a & 31);
    const int x1 = __shfl_sync(0xFFFFFFFFu, v1, a & 31);
    return (a >> 5) ? x1 : x0;
}

static __device__ __noinline__ void fin_tree(const Job &j, int b)
{
    const int lane = threadIdx.x & 31;
    const int64_t p0 = pos0_of(j, b);
    int par[2], ok[2], dep[2], anc[2];
    int nflag = 0;
    for (int half = 0; half < 2; ++half) {
        const int n = lane + 32 * half;
        const bool has = n < j.N;
        int pn = -1, np = 0;
        if (has) {
            pn = __ldg(j.parent + (int64_t)b * j.N + n);
            np = __ldg(j.node_pos + (int64_t)b * j.N + n);
        }
        const bool bad = has && (pn < -1 || pn >= n || np < 0);
        if (bad)
            latch(j.err, SV_ERR_DEVICE_BOUNDS);
        RowM r = merge_row(j, b, has ? n : 0, 1.0, 1.0);
        int win;
        if (j.Tp == 0.f) {
            win = r.amax;
        } else {
            GRes g = resolve_lanes(j, row_ptr(j, b, has ? n : 0),
                                   rng_key(j.seed, kTree, (uint64_t)b, p0 + np, 0),
                                   (double)j.Tp, j.invTp, r.gc, has);
            win = g.v;
            if (has)
                nflag += g.flag;
        }
        const bool m = has && (win == __ldg(j.node_tok + (int64_t)b * j.N + n));
        if (has && j.match) j.match[(int64_t)b * j.N + n] = m ? 1 : 0;
        // a node with a bad parent index is treated as a root that is not
        // accepted (depth 0, so its children sit at depth 1)
        par[half] = (has && !bad) ? pn : -1;
        ok[half] = (m && !bad) ? 1 : 0;
        dep[half] = (has && !bad) ? 1 : 0;
        anc[half] = par[half];
    }
    for (int o = 16; o; o >>= 1)
        nflag += __shfl_xor_sync(0xFFFFFFFFu, nflag, o);
    // Pointer jumping over the parent links (parents precede their children,
    // N <= 64): depth = nodes on the path from the root, ok = every node on it
    // matched.
    for (int it = 0; it < 6; ++it) {
        int na[2], nd[2], no[2];
        for (int half = 0; half < 2; ++half) {
            const int a = anc[half] < 0 ? 0 : anc[half];
            const int da = node_val(dep[0], dep[1], a);
            const int oa = node_val(ok[0], ok[1], a);
            const int aa = node_val(anc[0], anc[1], a);
            const bool up = anc[half] >= 0;
            nd[half] = up ? dep[half] + da : dep[half];
            no[half] = up ? (ok[half] & oa) : ok[half];
            na[half] = up ? aa : -1;
        }
        for (int half = 0; half < 2; ++half) {
            dep[half] = nd[half];
            ok[half] = no[half];
            anc[half] = na[half];
        }
    }
    // deepest accepted node, lowest index among equals
    int key = -1;
    for (int half = 0; half < 2; ++half) {
        const int n = lane + 32 * half;
        if (n < j.N && ok[half])
            key = max(key, (dep[half] << 8) | (255 - n));
    }
    for (int o = 16; o; o >>= 1)
        key = max(key, __shfl_xor_sync(0xFFFFFFFFu, key, o));
    const int best = key < 0 ? -1 : 255 - (key & 255);
    const int bestd = key < 0 ? 0 : (key >> 8);
    for (int k = lane; k < j.max_depth; k += 32)
        j.path_nodes[(int64_t)b * j.max_depth + k] = -1;
    __syncwarp();
    // walk from the best node to the root (warp-uniform)
    for (int n = best, d = bestd; n >= 0 && d > 0; --d) {
        if (lane == 0 && d - 1 < j.max_depth)
            j.path_nodes[(int64_t)b * j.max_depth + d - 1] = n;
        n = node_val(par[0], par[1], n);
    }
    if (lane == 0) {
        j.path_len[b] = bestd;
        j.commit_count[b] = bestd + 1;
        if (j.flags) j.flags[b] = nflag;
    }
}

static __device__ __noinline__ void fin_packed(const Job &j, int b)
{
    const int lane = threadIdx.x & 31;
    const int n = clamp_len(j, b);
    const int Km1 = j.K - 1;
    const bool greedy = (j.Tp == 0.f);
    if (lane == 0) check_len(j, b);
    // The stored proposal rows a_{t-1} .. a_{t-1} + n - 1 must exist.
    bool bad_off = false;
    if (!greedy) {
        int off = __ldg(j.prev_off + b);
        bad_off = off < 0 || off + n > j.W;
        if (bad_off && lane == 0)
            latch(j.err, SV_ERR_DEVICE_BOUNDS);
    }
    // ---- proposals Z_t (every draft row) ----
    {
        const bool has = lane < j.W;
        const int slot = j.K + (has ? lane : 0);
        RowM r = greedy ? merge_row(j, b, slot, j.cr1, 1.0) : merge_row(j, b, slot, j.crp, j.cr1);
        GRes g{r.amax, 0};
        if (!greedy)
            g = resolve_lanes(j, row_ptr(j, b, slot),
                              rng_key(j.seed, kDraft, (uint64_t)b, pos0_of(j, b) + lane, j.iter),
                              (double)j.Tp, j.invTp, r.gc, has);
        DraftTmp t;
        t.pad = 0.f;
        double conf;
        if (!has) {
        } else if (greedy) {
            t.z = r.amax;
            t.gflag = 0;
            t.q = 1.f;
            conf = exp_fast((double)r.m - r.L1a);
        } else {
            t.z = g.v;
            t.gflag = g.flag;
            float yz = load_logit(j, row_ptr(j, b, slot), t.z);
            t.q = exp_fast((double)yz * j.rTp - r.L1a);
            // confidence is the largest probability at T = 1
            conf = exp_fast((double)r.m - ((j.Tp == 1.f) ? r.L1a : r.L1b));
        }
        if (has) {
            j.dtmp[(int64_t)b * j.W + lane] = t;
            if (j.confidence) j.confidence[(int64_t)b * j.W + lane] = (float)conf;
        }
    }
    __syncwarp();
    // ---- verification of D_{t-1} ----
    if (greedy) {
        int v = -1;
        if (lane <= n) {
            RowM r = merge_row(j, b, lane, 1.0, 1.0);
            v = r.amax;
        }
        bool match = (lane < n) && (__ldg(j.ids + (int64_t)b * Km1 + lane) == v);
        unsigned mm = __ballot_sync(0xFFFFFFFFu, match);
        int h = (~mm == 0u) ? 32 : __ffs(~mm) - 1;
        h = min(h, n);
        int c = __shfl_sync(0xFFFFFFFFu, v, h & 31);
        packed_commit(j, b, h, c, true, 0);
        return;
    }
    const int64_t p0 = pos0_of(j, b);
    bool acc = false, und = false;
    double Lp = 0, ep = 0;
    if (lane < n) {
        RowM rp = merge_row(j, b, lane, j.crp, 1.0);
        Lp = rp.L1a;
        ep = j.eps_lse;
        // the logit at the draft token was recorded during the stream (NaN:
        // the token was out of range, already reported)
        double lp = -INFINITY;
        if (!isnan(rp.xd))
            lp = (double)rp.xd * j.rTp - Lp;
        // log q in fp32 (logf within 1 ulp of |log q|): 2^-22 (1 + |log q|)
        const float qd = __ldg(j.prev_q + (int64_t)b * Km1 + lane);
        double lq = (double)logf(qd);
        double r = (double)exp_fast(lp - lq);
        double rel = 1.01 * ep + 0x1p-21 + 0x1p-22 * (1.0 + fabs(lq)) + 1e-13;
        double alo = fmin(1.0, r * (1.0 - rel)), ahi = fmin(1.0, r * (1.0 + rel));
        double u = uniform_at(rng_key(j.seed, kAccept, (uint64_t)b, p0 + lane, 0), 0, j.skip);
        acc = u < alo - kFlagEps;
        und = !(acc || u >= ahi + kFlagEps) || j.force_rescue;
        if (j.force_rescue)
            acc = false;
        RowStat *sp = j.rs_stat + (int64_t)b * j.rows_per_seq + lane;
        sp->L1 = Lp;
        sp->m = rp.m;
        sp->eps = (float)ep;
    }
    unsigned am = __ballot_sync(0xFFFFFFFFu, acc);
    unsigned um = __ballot_sync(0xFFFFFFFFu, und);
    int f = (~am == 0u) ? 32 : __ffs(~am) - 1;
    f = min(f, n);
    unsigned upto = (f >= 31) ? 0xFFFFFFFFu : ((2u << f) - 1u);
    bool rescue = (um & upto) != 0u || j.force_rescue;
    double Lph = __shfl_sync(0xFFFFFFFFu, Lp, f & 31);
    double eph = __shfl_sync(0xFFFFFFFFu, ep, f & 31);
    if (bad_off && (rescue || f < n)) {
        // no residual row to read: commit the proven prefix only
        packed_commit(j, b, f, -1, false, 0);
        return;
    }
    if (rescue) {
        if (lane == 0) {
            unsigned e = atomicAdd(j.ctl + C_RESCUE_N, 1u);
            j.rescue[e].b = b;
            j.rescue[e].kind = 0;
            j.rescue[e].h = 0;
        }
        return;
    }
    if (f == n) {
        RowM rb = merge_row(j, b, n, j.crp, 1.0);
        GRes g = resolve_lanes(j, row_ptr(j, b, n),
                               rng_key(j.seed, kSample, (uint64_t)b, p0 + n, 0), (double)j.Tp,
                               j.invTp, rb.gc, lane == 0);
        int c = __shfl_sync(0xFFFFFFFFu, g.v, 0);
        int fl = __shfl_sync(0xFFFFFFFFu, g.flag, 0);
        packed_commit(j, b, n, c, true, fl);
        return;
    }
    packed_commit(j, b, f, -1, false, 0);
    if (lane == 0) {
        int off = __ldg(j.prev_off + b);
        unsigned e = atomicAdd(j.ctl + C_RESID_N, 1u);
        ResidEntry re;
        re.b = b;
        re.h = f;
        re.need_lq = 1;
        re.pad = 0;
        re.prow = row_ptr(j, b, f);
        re.qrow = j.src2 + ((int64_t)b * j.W + off + f) * j.rs;
        re.Lp = Lph;
        re.Lq = 0.0;
        re.epsp = eph;
        re.epsq = 0.0;
        re.lclo = re.lchi = 0.0;
        j.resid[e] = re;
    }
}

// ---------------------------------------------------------------------------
// SPOT decision step ([SPOT] App. A.1): the target's transition Phi at every
// state of the tree (position s* by the largest probability over the state's
// masked positions, then its token), the match bit of every node, and the
// walk from the root through accepted children.  One warp; lane a holds
// states a, a + 32 and a + 64.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int state_val(const int (&v)[3], int a)
{
    const int x0 = __shfl_sync(0xFFFFFFFFu, v[0], a & 31);
    const int x1 = __shfl_sync(0xFFFFFFFFu, v[1], a & 31);
    const int x2 = __shfl_sync(0xFFFFFFFFu, v[2], a & 31);
    return (a >> 5) == 0 ? x0 : ((a >> 5) == 1 ? x1 : x2);
}

// max_v softmax(x)_v = 1 / sum_v exp(x_v - max x) of one row in fp64, by the
// whole warp: the rare states whose fp32 confidences do not separate their
// best position by the 1e-9 window.
static __device__ __noinline__ double conf64_row(const Job &j, const char *row)
{
    const int lane = threadIdx.x & 31;
    float m = -INFINITY;
    for (int v = lane; v < j.V; v += 32)
        m = fmaxf(m, load_logit(j, row, v));
    m = warp_max(m);
    double sum = 0.0;
    for (int v = lane; v < j.V; v += 32)
        sum += exp((double)load_logit(j, row, v) - (double)m);
    return 1.0 / warp_sumd(sum);
}

static __device__ __noinline__ void fin_spot(const Job &j, int b)
{
    const int lane = threadIdx.x & 31;
    const int S = j.N + 1, L = j.L;
    const int64_t p0 = pos0_of(j, b);
    // relative error of a confidence exp(m - L1) from the streamed sums
    const double e = 1.01 * j.eps_lse + 0x1p-21 + 1e-13;
    int sp[3], sv[3], nflag = 0;
    for (int r = 0; r < 3; ++r) {
        const int st = lane + 32 * r;
        const uint64_t mk = st < S ? __ldg(j.smask + (int64_t)b * S + st) : 0ull;
        // best position by fp32 confidence (lowest s among equal values) and
        // the largest upper end among the other masked positions
        float bc = -1.f;
        double blo = 0.0, bhi = 0.0, ohi = -1.0;
        int bs = -1, bam = -1;
        Cand2 bgc;
        bgc.init();
        for (int s = 0; s < L; ++s) {
            if (!((mk >> s) & 1ull))
                continue;
            const RowM rm = merge_row(j, b, st * L + s, j.cr1, 1.0);
            const float c = exp_fast((double)rm.m - rm.L1a);
            const double lo = (double)c * (1.0 - e), hi = (double)c * (1.0 + e);
            if (c > bc) {
                if (bs >= 0)
                    ohi = fmax(ohi, bhi);
                bc = c;
                blo = lo;
                bhi = hi;
                bs = s;
                bam = rm.amax;
                bgc = rm.gc;
            } else {
                ohi = fmax(ohi, hi);
            }
        }
        // settled in fp32 when the best's lower end clears every other upper
        // end by the flag window; else the contenders in fp64, by the warp
        const bool unsure = bs >= 0 && ohi >= 0.0 && blo - ohi < kFlagEps;
        unsigned um = __ballot_sync(0xFFFFFFFFu, unsure);
        while (um) {
            const int src = __ffs(um) - 1;
            um &= um - 1;
            const int ost = src + 32 * r;
            const uint64_t omk = __shfl_sync(0xFFFFFFFFu, mk, src);
            const double oblo = __shfl_sync(0xFFFFFFFFu, blo, src);
            // contenders: masked positions whose upper end reaches the best's
            // lower end - 1e-9 (lane = position)
            bool cont = false;
            if (lane < L && ((omk >> lane) & 1ull)) {
                const RowM rm = merge_row(j, b, ost * L + lane, j.cr1, 1.0);
                const double c = (double)exp_fast((double)rm.m - rm.L1a);
                cont = c * (1.0 + e) >= oblo - kFlagEps;
            }
            unsigned cm = __ballot_sync(0xFFFFFFFFu, cont);
            double c1 = -1.0, c2 = -1.0;
            int s1 = -1;
            while (cm) {  // ascending positions: the lowest wins exact ties
                const int s = __ffs(cm) - 1;
                cm &= cm - 1;
                const double c = conf64_row(j, row_ptr(j, b, ost * L + s));
                if (c > c1) {
                    c2 = c1;
                    c1 = c;
                    s1 = s;
                } else if (c > c2) {
                    c2 = c;
                }
            }
            if (lane == src) {
                bs = s1;
                if (c1 - c2 > 0.0 && c1 - c2 < kFlagEps)
                    ++nflag;
            }
        }
        // the token at s*: its row's argmax (T = 0) or coupled-noise
        // Gumbel-max (T > 0)
        const bool has = bs >= 0;
        const RowM rb = (has && unsure) ? merge_row(j, b, st * L + bs, j.cr1, 1.0) : RowM{};
        if (has && unsure) {
            bam = rb.amax;
            bgc = rb.gc;
        }
        int v = has ? bam : -1;
        if (j.Tp != 0.f) {
            const GRes g = resolve_lanes(j, row_ptr(j, b, has ? st * L + bs : 0),
                                         rng_key(j.seed, kTree, (uint64_t)b, p0 + (has ? bs : 0), 0),
                                         (double)j.Tp, j.invTp, bgc, has);
            v = has ? g.v : -1;
            if (has)
                nflag += g.flag;
        }
        sp[r] = bs;
        sv[r] = v;
        if (st < S) {
            if (j.state_pos) j.state_pos[(int64_t)b * S + st] = bs;
            if (j.state_tok) j.state_tok[(int64_t)b * S + st] = v;
        }
    }
    // match bits: a node's commitment equals Phi of its parent's state
    bool mt[2];
    int par[2];
    for (int h = 0; h < 2; ++h) {
        const int n = lane + 32 * h;
        const bool in = n < j.N;
        par[h] = in ? __ldg(j.parent + (int64_t)b * j.N + n) : -2;
        const int pos = in ? __ldg(j.node_pos + (int64_t)b * j.N + n) : -1;
        const int tok = in ? __ldg(j.node_tok + (int64_t)b * j.N + n) : -1;
        const bool ok = in && par[h] >= -1 && par[h] < n;
        const int a = ok ? par[h] + 1 : 0;
        const int ps = state_val(sp, a), pv = state_val(sv, a);
        mt[h] = ok && ps >= 0 && pos == ps && tok == pv;
        if (in && j.match) j.match[(int64_t)b * j.N + n] = mt[h] ? 1 : 0;
    }
    for (int k = lane; k < j.max_depth; k += 32)
        j.path_nodes[(int64_t)b * j.max_depth + k] = -1;
    __syncwarp();
    // the walk: the lowest-index accepted child of the state reached
    int y = -1, len = 0;
    for (int it = 0; it < j.N; ++it) {
        const unsigned c0 = __ballot_sync(0xFFFFFFFFu, mt[0] && par[0] == y);
        const unsigned c1 = __ballot_sync(0xFFFFFFFFu, mt[1] && par[1] == y);
        if (!c0 && !c1)
            break;
        const int nx = c0 ? __ffs(c0) - 1 : 32 + __ffs(c1) - 1;
        if (lane == 0 && len < j.max_depth)
            j.path_nodes[(int64_t)b * j.max_depth + len] = nx;
        ++len;
        y = nx;
    }
    const int cs = state_val(sp, y + 1), ct = state_val(sv, y + 1);
    for (int o = 16; o; o >>= 1)
        nflag += __shfl_xor_sync(0xFFFFFFFFu, nflag, o);
    if (lane == 0) {
        j.path_len[b] = len;
        j.commit_count[b] = len + (cs >= 0 ? 1 : 0);
        j.commit_pos[b] = cs;
        j.commit_tok[b] = ct;
        if (j.flags) j.flags[b] = nflag;
    }
}

// ---------------------------------------------------------------------------
// Any-order Packed-SS decision step ([PackedSS] App. C, Alg. 3 lines 6-15,
// eq. 8; scores of App. E.6).  One warp; lane r is rank r of the verify
// order and also window index r.
// ---------------------------------------------------------------------------
static __device__ __noinline__ void fin_anyorder(const Job &j, int b)
{
    const int lane = threadIdx.x & 31;
    const int W = j.W;
    const int u = min(max(__ldg(j.lens + b), 0), W);
    const int nreq = (int)__ldg(j.smask + b);
    const int32_t *wp = j.win_pos + (int64_t)b * W, *od = j.order + (int64_t)b * W;
    const int32_t *dr = j.ids + (int64_t)b * W;
    // rank r: its window index, position and draft; kappa = leading ranks
    // with a draft (the preparation checked that order is a permutation)
    const int oi = lane < u ? __ldg(od + lane) : 0;
    const int pos = lane < u ? __ldg(wp + oi) : 0;
    const int d = lane < u ? __ldg(dr + oi) : -1;
    const unsigned hasd = __ballot_sync(0xFFFFFFFFu, lane < u && d >= 0);
    const int kappa = min((~hasd == 0u) ? 32 : __ffs(~hasd) - 1, u);
    int v = -1;
    if (lane < nreq)
        v = merge_row(j, b, lane, 1.0, 1.0).amax;  // eq. 8: the verifier's argmax
    const unsigned mm = __ballot_sync(0xFFFFFFFFu, lane < kappa && d == v);
    const int h = min((~mm == 0u) ? 32 : __ffs(~mm) - 1, kappa);
    const int A = min(h + 1, u);
    // an accepted EOS at position p lowers the end to min(E, p)
    const int E0 = __ldg(j.end_in + b);
    int ecut = 0x7FFFFFFF;
    if (lane < A && j.eos >= 0 && v == j.eos)
        ecut = pos;
    const int E = min(E0, __reduce_min_sync(0xFFFFFFFFu, ecut));
    // accepted pairs within E, rank order
    const bool keep = lane < A && pos <= E;
    const unsigned km = __ballot_sync(0xFFFFFFFFu, keep);
    const int kept = __popc(km);
    const int slot = __popc(km & ((1u << lane) - 1u));
    if (keep) {
        j.commit_pos[(int64_t)b * W + slot] = pos;
        j.commit_tok[(int64_t)b * W + slot] = v;
    }
    if (lane >= kept && lane < W) {
        j.commit_pos[(int64_t)b * W + lane] = -1;
        j.commit_tok[(int64_t)b * W + lane] = -1;
    }
    const unsigned accd = __reduce_or_sync(0xFFFFFFFFu, keep ? (1u << oi) : 0u);
    // proposals (window index = lane): argmax, and its probability at
    // temperature 1 with a relative error bound
    const double e = 1.01 * j.eps_lse + 0x1p-21 + 1e-13;
    int z = -1;
    double sc = -1.0;
    if (lane < u) {
        const RowM rm = merge_row(j, b, j.K + lane, j.cr1, 1.0);
        z = rm.amax;
        sc = (double)exp_fast((double)rm.m - rm.L1a);
    }
    const int wpos = lane < u ? __ldg(wp + lane) : 0x7FFFFFFF;
    const bool ret = lane < u && !((accd >> lane) & 1u) && wpos <= E;
    // scores whose intervals overlap another retained score's are recomputed
    // in fp64 (by the warp), so that the order below is exact
    bool unsure = false;
    for (int o = 0; o < 32; ++o) {
        const double so = __shfl_sync(0xFFFFFFFFu, sc, o);
        const bool ro = __shfl_sync(0xFFFFFFFFu, ret, o);
        if (ret && ro && o != lane && fabs(sc - so) <= (sc + so) * e)
            unsure = true;
    }
    unsigned um = __ballot_sync(0xFFFFFFFFu, unsure);
    while (um) {
        const int src = __ffs(um) - 1;
        um &= um - 1;
        const double c = conf64_row(j, row_ptr(j, b, j.K + src));
        if (lane == src)
            sc = c;
    }
    // rank of each retained position: decreasing score, ties by position
    int rank = 0;
    for (int o = 0; o < 32; ++o) {
        const double so = __shfl_sync(0xFFFFFFFFu, sc, o);
        const bool ro = __shfl_sync(0xFFFFFFFFu, ret, o);
        if (ro && (so > sc || (so == sc && o < lane)))
            ++rank;
    }
    const int nret = __popc(__ballot_sync(0xFFFFFFFFu, ret));
    if (lane < W) {
        j.next_draft[(int64_t)b * W + lane] = ret ? z : -1;
        if (j.confidence)
            j.confidence[(int64_t)b * W + lane] =
                lane < u ? (float)sc : __int_as_float(0x7FC00000);
        if (ret)
            j.next_order[(int64_t)b * W + rank] = lane;
        if (lane >= nret)
            j.next_order[(int64_t)b * W + lane] = -1;
    }
    if (lane == 0) {
        j.acc[b] = h;
        j.commit_len[b] = kept;
        j.end_out[b] = E;
    }
}

// ---------------------------------------------------------------------------
// The streaming kernel.
// ---------------------------------------------------------------------------
template <int KIND>
__device__ __forceinline__ void fin_kind(const Job &j, int b)
{
    if constexpr (KIND == K_GREEDY)
        fin_greedy(j, b);
    else if constexpr (KIND == K_SAMPLE)
        fin_sample(j, b);
    else if constexpr (KIND == K_TREE)
        fin_tree(j, b);
    else if constexpr (KIND == K_SPOT)
        fin_spot(j, b);
    else if constexpr (KIND == K_ANYORDER)
        fin_anyorder(j, b);
    else
        fin_packed(j, b);
}

// A thread's sum moved to the warp's reference E (exact scaling).
__device__ __forceinline__ float rebased(float2 acc, float e, float E)
{
    return e > -INFINITY ? (acc.x + acc.y) * pow2_int(e - E) : 0.f;
}

// End of a unit for one consumer warp: reduce the warp's state and hand it to
// the finalizer through unit slot lu % kUnitSlots.
// Unit header values the consumers keep after the unit's stages are released.
struct UnitHead {
    int unit, lu, b;
    unsigned expect;
    int xid;
};

__device__ __forceinline__ void finish_unit(const Job &j, const UnitHead &mt, TState &s,
                                            const RowMode &rm, PassShared &sm)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int us = mt.lu % kUnitSlots;
    const bool gum = (rm.mode & M_GUMBEL) != 0;
    const bool lse = (rm.mode & M_LSE) != 0, lse2 = (rm.mode & M_LSE2) != 0;
    const bool hasmax = (rm.mode & (M_ARGMAX | M_MAX)) != 0;
    float mx = s.mx;
    int am = s.amax;
    if (hasmax)
        warp_argmax(mx, am);
    Cand2 g = s.g.c;
    if (gum)
        warp_cand2(g);
    const float xd = warp_max(s.xd);  // NaN except at one lane (fmaxf drops NaN)
    float E1 = -INFINITY, E2 = -INFINITY, S1 = 0.f, S2 = 0.f;
    if (lse) {
        E1 = warp_max(s.e1);
        S1 = warp_sum(rebased(s.acc1, s.e1, E1));
    }
    if (lse2) {
        E2 = warp_max(s.e2);
        S2 = warp_sum(rebased(s.acc2, s.e2, E2));
    }
    if (lane == 0) {
        // the slot's previous unit must have been merged (normally long ago)
        if (!mbar_wait(&sm.ufree[us], ((mt.lu / kUnitSlots) & 1) ^ 1))
            latch(j.err, SV_ERR_TIMEOUT);
        WarpPart &p = sm.up[us][w];
        p.m = hasmax ? mx : -INFINITY;
        p.amax = hasmax ? am : 0x7FFFFFFF;
        p.e1 = E1;
        p.s1 = S1;
        p.e2 = E2;
        p.s2 = S2;
        p.hi1 = g.hi1;
        p.lo1 = g.lo1;
        p.hi2 = g.hi2;
        p.lo2 = g.lo2;
        p.hi3 = g.hi3;
        p.v1 = g.v1;
        p.v2 = g.v2;
        p.xd = xd;
        if (w == 0) {
            sm.uunit[us] = mt.unit;
            sm.ub[us] = mt.b;
            sm.uexpect[us] = mt.expect;
        }
        mbar_arrive(&sm.ubar[us]);
    }
}

// Merge the consumer warps' partials of local units cu .. cu + n - 1 (n <=
// kUnitSlots, all complete), one unit per lane, into their records and count
// them towards their sequences.  Returns a lane mask of the units whose record
// completed a sequence; lane i's seq is its unit's sequence.  Whole warp.
__device__ __forceinline__ unsigned merge_units(const Job &j, PassShared &sm, int cu, int n,
                                                int &seq)
{
    const int lane = threadIdx.x & 31;
    bool done = false;
    seq = -1;
    if (lane < n) {
        const int us = (cu + lane) % kUnitSlots;
        float m = -INFINITY, e1 = -INFINITY, e2 = -INFINITY;
        float xd = __int_as_float(0x7FC00000);
        int am = 0x7FFFFFFF;
        Cand2 g;
        g.init();
#pragma unroll 1
        for (int w = 0; w < kConsumerWarps; ++w) {
            const WarpPart &p = sm.up[us][w];
            if (p.m > m || (p.m == m && (unsigned)p.amax < (unsigned)am)) {
                m = p.m;
                am = p.amax;
            }
            e1 = fmaxf(e1, p.e1);
            e2 = fmaxf(e2, p.e2);
            xd = fmaxf(xd, p.xd);
            Cand2 o;
            o.hi1 = p.hi1;
            o.lo1 = p.lo1;
            o.hi2 = p.hi2;
            o.lo2 = p.lo2;
            o.hi3 = p.hi3;
            o.v1 = p.v1;
            o.v2 = p.v2;
            g.merge(o);
        }
        float S1 = 0.f, S2 = 0.f;
#pragma unroll 1
        for (int w = 0; w < kConsumerWarps; ++w) {
            const WarpPart &p = sm.up[us][w];
            if (p.s1 > 0.f) S1 += p.s1 * pow2_int(p.e1 - e1);
            if (p.s2 > 0.f) S2 += p.s2 * pow2_int(p.e2 - e2);
        }
        const int unit = sm.uunit[us], b = sm.ub[us];
        const unsigned expect = sm.uexpect[us];
        seq = b;
        RowPart r;
        r.m = m;
        r.e1 = e1;
        r.e2 = e2;
        r.s1 = S1;
        r.s2 = S2;
        r.amax = am;
        r.ghi1 = g.hi1;
        r.glo1 = g.lo1;
        r.ghi2 = g.hi2;
        r.glo2 = g.lo2;
        r.ghi3 = g.hi3;
        r.gv1 = g.v1;
        r.gv2 = g.v2;
        r.xd = xd;
        r.pad[0] = r.pad[1] = 0;
        j.rp[unit] = r;
        __threadfence();
        const unsigned old = atomicAdd(j.seq_done + b, 1u);
        done = (old + 1u == expect);
        if (done)
            __threadfence();  // acquire: every record of the sequence is visible
        mbar_arrive(&sm.ufree[us]);
    }
    return __ballot_sync(0xFFFFFFFFu, done);
}

// The finalizer warp: merges unit partials in local-unit order, all units
// that are complete at once, and runs the decision steps of completed
// sequences, until the producer is done and every unit it streamed is
// merged.  Once the producer is done it only queues decision steps: the
// steps still queued when it returns are run by every warp of the CTA at
// once (end_decisions), so that a CTA that completes several sequences at the
// end of the pass does not run their steps one after another.  Waits are
// bounded by a spin limit that restarts whenever work is found.
template <int KIND>
__device__ void finalizer_loop(const Job &j, PassShared &sm)
{
    const int lane = threadIdx.x & 31;
    int cu = 0, qh = 0, qt = 0;
    uint32_t spin = 0;
    for (;;) {
        // complete slots from cu on (each lane tests one; a completed phase
        // stays complete until the slot is freed)
        const int u = cu + lane;
        const bool rdy = lane < kUnitSlots && mbar_try(&sm.ubar[u % kUnitSlots],
                                                       (u / kUnitSlots) & 1);
        const unsigned rm = __ballot_sync(0xFFFFFFFFu, rdy);
        const int n = __ffs(~rm) - 1;  // leading complete slots
        if (n > 0) {
            int seq;
            unsigned dm = merge_units(j, sm, cu, n, seq);
            while (dm) {
                const int i = __ffs(dm) - 1;
                dm &= dm - 1;
                const int b = __shfl_sync(0xFFFFFFFFu, seq, i);
                if (qt - qh < kFinQ) {
                    __syncwarp();  // every lane has read the slot it may overwrite
                    if (lane == 0)
                        sm.todo[qt % kFinQ] = b;
                    ++qt;
                } else {
                    fin_kind<KIND>(j, b);
                }
            }
            __syncwarp();
            cu += n;
            spin = 0;
            continue;
        }
        int pdone = 0;
        if (lane == 0)
            pdone = sm.prod_done;
        pdone = __shfl_sync(0xFFFFFFFFu, pdone, 0);
        if (qh < qt && !pdone) {
            const int b = sm.todo[qh % kFinQ];
            ++qh;
            fin_kind<KIND>(j, b);
            spin = 0;
            continue;
        }
        int fin = 0;
        if (lane == 0)
            fin = pdone && cu >= sm.nunits;
        if (__shfl_sync(0xFFFFFFFFu, fin, 0))
            break;
        if (++spin > kSpinLimit) {
            if (lane == 0)
                latch(j.err, SV_ERR_TIMEOUT);
            break;
        }
        if (spin > 64)
            __nanosleep(SV_SPIN_SLEEP_NS);
    }
    __syncwarp();
    if (lane == 0) {
        sm.fin_qh = qh;
        sm.fin_qt = qt;
    }
}

// The decision steps the finalizer left queued, a warp per step (every warp
// of the CTA calls it after the CTA-wide barrier that follows the loops).
template <int KIND>
__device__ __forceinline__ void end_decisions(const Job &j, PassShared &sm)
{
    constexpr int kWarps = kPassThreads / 32;
    const int qh = sm.fin_qh, qt = sm.fin_qt;
    for (int i = qh + (int)(threadIdx.x >> 5); i < qt; i += kWarps)
        fin_kind<KIND>(j, sm.todo[i % kFinQ]);
}

// ---------------------------------------------------------------------------
// Seeding of Gumbel units by the consumer threads.  Every top id of a unit's
// id range is found (a couple of skip draws per block of 256 ids; threads take
// blocks in turn and list the ids in shared memory), its logit is copied to
// shared memory (cp.async, issued one unit ahead when the producer names the
// next unit), and it is scored in an fp32 interval.  The top ids join the
// candidates and the best lower end - 1e-9 starts the unit's shared
// threshold; the consumers' scan then skips top ids.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// The aligned 32-bit word that holds the logit of id v, and the logit in it.
template <typename In>
__device__ __forceinline__ const void *logit_word(const char *row, uint32_t v)
{
    return row + (sizeof(In) == 2 ? (((size_t)v * 2) & ~(size_t)3) : (size_t)v * 4);
}
template <typename In>
__device__ __forceinline__ float logit_of_word(uint32_t w, uint32_t v)
{
    if (sizeof(In) == 2)
        return __uint_as_float((v & 1u) ? (w & 0xFFFF0000u) : (w << 16));
    return __uint_as_float(w);
}

// Barrier among the consumer warps on an mbarrier (kConsumerWarps arrivals)
// with a bounded wait.  A hardware barrier would wait without end for a warp
// that gave up after an expired wait; this one gives up too (latching
// SV_ERR_TIMEOUT), and the CTA's abort flag then makes every later wait
// return at once and the consumers leave the stream.  Every consumer thread
// calls it; returns false when the barrier did not complete.  The mbarrier's
// release / acquire order the consumers' shared-memory accesses around it.
__device__ __noinline__ bool csync(PassShared &sm, const Job &j)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t ph = sm.cph[w];
    __syncwarp();
    if (lane == 0)
        mbar_arrive(&sm.csync);
    bool ok = false;
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try(&sm.csync, ph)) {
            ok = true;
            break;
        }
        if (sm.abort)
            break;
        if (SV_SPIN_SLEEP_NS > 0 && i > 64)
            __nanosleep(SV_SPIN_SLEEP_NS);
    }
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (lane == 0) {
        sm.cph[w] = ph ^ 1u;
        if (!ok) {
            latch(j.err, SV_ERR_TIMEOUT);
            sm.abort = 1;
        }
    }
    __syncwarp();
    return ok;
}

// Lists the top ids of [lo, hi) in buffer b; false if they did not all fit
// (the count is then larger than the list).  *listed receives the number of
// ids in the list, the same in every thread.  Every consumer thread calls
// it.  After a barrier that did not complete the list is left empty.
__device__ __noinline__ bool seed_list(PassShared &sm, const Job &j, int b, uint64_t key, int lo,
                                       int hi, int *listed)
{
    const int t = threadIdx.x;
    *listed = 0;
    if (t == 0)
        sm.seed_n = 0;
    if (!csync(sm, j)) {
        if (t == 0)
            sm.seed_cnt[b] = 0;
        return true;
    }
    const uint32_t bhi = (uint32_t)(hi - 1) >> 8;
    uint32_t beta = ((uint32_t)lo >> 8) + t;
    int pos = -1, i = 0;
    while (beta <= bhi) {
        pos = next_top(key, beta, i++, pos, sm.skip);
        const uint32_t v = beta * 256u + (uint32_t)pos;
        if (pos > 255 || v >= (uint32_t)hi) {  // block done
            beta += kConsumers;
            pos = -1;
            i = 0;
        } else if (v >= (uint32_t)lo) {
            const int idx = atomicAdd(&sm.seed_n, 1);
            if (idx < kSeedCap)
                sm.seed_ids[b][idx] = v;
        }
    }
    const bool ok = csync(sm, j);
    const int n = ok ? sm.seed_n : 0;
    *listed = min(n, kSeedCap);
    if (t == 0)
        sm.seed_cnt[b] = min(n, kSeedCap);
    return n <= kSeedCap;
}

// Starts the copies of the n listed ids' logit words into buffer b.
template <typename In>
__device__ __forceinline__ void seed_copy(PassShared &sm, int b, const char *row, int n)
{
    for (int e = threadIdx.x; e < n; e += kConsumers)
        cp_async4(&sm.seed_x[b][e], logit_word<In>(row, sm.seed_ids[b][e]));
    cp_async_commit();
}

// Scores buffer b (its copies must have been started) and starts the unit's
// threshold.
template <typename In>
__device__ __noinline__ GState seed_eval(PassShared &sm, const Job &j, int b, GState g,
                                         const RowMode &rm, int tslot)
{
    cp_async_wait_all();
    const bool ok = csync(sm, j);  // every thread's copies have landed
    const int n = ok ? min(max(sm.seed_cnt[b], 0), kSeedCap) : 0;
    for (int e = threadIdx.x; e < n; e += kConsumers) {
        const uint32_t v = sm.seed_ids[b][e];
        const float2 iv = logit_interval_m(logit_of_word<In>(sm.seed_x[b][e], v), rm.invT,
                                           fine52(rm.key, v), true);
        g.c.add(iv.x, iv.y, (int)v);
        if (iv.x > g.lomax) {
            g.lomax = iv.x;
            raise_thr(g, __fsub_rd(iv.x, 1e-9f));
        }
    }
    atomicMax(&sm.thr[tslot], f2ord(g.thr));
    if (csync(sm, j))
        raise_thr(g, ord2f(*(volatile uint32_t *)&sm.thr[tslot]));
    return g;
}

// Seeding without a prefetched list: in rounds of at most kSeedCap ids,
// loading the logits directly (the fallback for units with more top ids than
// a list holds).
template <typename In>
__device__ __noinline__ GState seed_rounds(PassShared &sm, const Job &j, int b, const char *row,
                                           int lo, int hi, GState g, const RowMode &rm, int tslot)
{
    using VT = VecTraits<In>;
    constexpr uint32_t kNone = 0xFFFFFFFFu;
    constexpr int kPer = (kSeedCap + kConsumers - 1) / kConsumers;
    const int t = threadIdx.x;
    const uint32_t bhi = (uint32_t)(hi - 1) >> 8;
    uint32_t beta = ((uint32_t)lo >> 8) + t;
    int pos = -1, i = 0;
    bool more = beta <= bhi;
    uint32_t pend = kNone;  // a top id found but not listed yet
    for (;;) {
        if (t == 0) {
            sm.seed_n = 0;
            sm.seed_more = 0;
        }
        if (!csync(sm, j))
            return g;
        for (;;) {
            if (pend != kNone) {
                const int idx = atomicAdd(&sm.seed_n, 1);
                if (idx >= kSeedCap)
                    break;  // the list is full: keep it for the next round
                sm.seed_ids[b][idx] = pend;
                pend = kNone;
            }
            if (!more)
                break;
            pos = next_top(rm.key, beta, i++, pos, sm.skip);
            const uint32_t v = beta * 256u + (uint32_t)pos;
            if (pos > 255 || v >= (uint32_t)hi) {  // block done
                beta += kConsumers;
                pos = -1;
                i = 0;
                more = beta <= bhi;
            } else if (v >= (uint32_t)lo) {
                pend = v;
            }
        }
        if (more || pend != kNone)
            sm.seed_more = 1;
        if (!csync(sm, j))
            return g;
        const int n = min(sm.seed_n, kSeedCap);
        uint32_t id[kPer];
        float x[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int e = t + k * kConsumers;
            id[k] = e < n ? sm.seed_ids[b][e] : kNone;
            x[k] = id[k] != kNone ? VT::load1(row, (int)id[k]) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k)
            if (id[k] != kNone) {
                const float2 iv =
                    logit_interval_m(x[k], rm.invT, fine52(rm.key, id[k]), true);
                g.c.add(iv.x, iv.y, (int)id[k]);
                if (iv.x > g.lomax) {
                    g.lomax = iv.x;
                    raise_thr(g, __fsub_rd(iv.x, 1e-9f));
                }
            }
        const int again = sm.seed_more;
        if (!csync(sm, j))  // the list is reused by the next round
            return g;
        if (!again)
            break;
    }
    atomicMax(&sm.thr[tslot], f2ord(g.thr));
    if (csync(sm, j))
        raise_thr(g, ord2f(*(volatile uint32_t *)&sm.thr[tslot]));
    return g;
}

// Streams one unit whose first stage is ready in `stage`: every stage of the
// unit with the row mode fixed at compile time, then the unit's partial.
// Returns false if a wait timed out or the producer aborted.
template <typename In, int MODE>
__device__ __forceinline__ bool unit_loop(const Job &j, PassShared &sm, unsigned char *stages,
                                          const float *gt, int &stage, uint32_t &phase,
                                          const RowMode &rm, int &pf_next)
{
    const int lane = threadIdx.x & 31;
    const StageMeta &m0 = sm.meta[stage];
    const UnitHead uh{m0.unit, m0.lu, m0.b, m0.expect, m0.xid};
    const int tslot = uh.lu % kStages;
    TState s;
    tstate_init(s);
    constexpr int E = VecTraits<In>::N;
    // pf_next: (record << 1 | buffer) of the unit whose top ids were listed
    // and copied a unit ago, or -1.  Residual units may stream between a unit
    // and the one it prefetched for, so the buffer travels with the record.
    const bool pre = pf_next >= 0 && (pf_next >> 1) == uh.unit;
    const int sb = pre ? (pf_next & 1) : (pf_next >= 0 ? (pf_next & 1) ^ 1 : 0);
    int listed = 0;
    if (MODE & M_GUMBEL) {
        if (pre) {
            s.g = seed_eval<In>(sm, j, sb, s.g, rm, tslot);  // listed and copied a unit ago
        } else if (seed_list(sm, j, sb, rm.key, m0.vbase * E, m0.vend * E, &listed)) {
            seed_copy<In>(sm, sb, m0.row, listed);
            s.g = seed_eval<In>(sm, j, sb, s.g, rm, tslot);
        } else {
            s.g = seed_rounds<In>(sm, j, sb, m0.row, m0.vbase * E, m0.vend * E, s.g, rm, tslot);
        }
    }
    if (m0.nrec >= 0) {
        // the next unit carries a Gumbel-max: list its top ids and start
        // their copies now, so that they land while this unit streams
        const int nb = sb ^ 1;
        const bool fits = seed_list(sm, j, nb, m0.nkey, m0.nlo, m0.nhi, &listed);
        if (fits)
            seed_copy<In>(sm, nb, m0.nrow, listed);
        pf_next = fits ? (m0.nrec << 1) | nb : -1;  // the same on every consumer thread
    } else {
        pf_next = -1;
    }
    for (;;) {
        const StageMeta &mt = sm.meta[stage];
        const int nv = mt.nv, vbase = mt.vbase, last = mt.last;
        const uint4 *st = reinterpret_cast<const uint4 *>(stages + (size_t)stage * kStageBytes);
        if (MODE & M_GUMBEL)
            raise_thr(s.g, ord2f(*(volatile uint32_t *)&sm.thr[tslot]));
        do_chunk<In, MODE>(st, nv, vbase, s, rm, gt, sm);
        if (uh.xid >= 0) {
            // the thread that holds the draft token's vector records its logit
            constexpr int E = VecTraits<In>::N;
            const int iv = uh.xid / E - vbase;
            if (iv >= 0 && iv < nv && (int)threadIdx.x == iv % kConsumers)
                s.xd = VecTraits<In>::elem(st[iv], uh.xid % E);
        }
        if ((MODE & M_GUMBEL) && s.g.thr > s.pub) {
            atomicMax(&sm.thr[tslot], f2ord(s.g.thr));
            s.pub = s.g.thr;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.empty[stage]);
        if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
        }
        if (last)
            break;
        if (!mbar_wait(&sm.full[stage], phase)) {
            latch(j.err, SV_ERR_TIMEOUT);
            return false;
        }
        if (sm.meta[stage].unit != uh.unit || sm.abort)  // the producer or a consumer aborted
            return false;
    }
    if ((MODE & M_GUMBEL) && s.gqn > 0) {
        const int w = threadIdx.x >> 5;
        s.g = gumbel_flush<In>(sm.gqd[w], sm.gqv[w], s.gqn, s.g, rm, gt, sm.skip);
        s.gqn = 0;
    }
    finish_unit(j, uh, s, rm, sm);
    return true;
}

// Only the row modes of entry-point kind KIND are instantiated.
template <typename In, int KIND>
__device__ __forceinline__ bool unit_dispatch(const Job &j, PassShared &sm, unsigned char *stages,
                                              const float *gt, int &stage, uint32_t &phase,
                                              const RowMode &rm, int &pf_next)
{
    const int m = rm.mode;
    if constexpr (KIND == K_GREEDY) {
        return unit_loop<In, M_ARGMAX>(j, sm, stages, gt, stage, phase, rm, pf_next);
    } else if constexpr (KIND == K_SAMPLE) {
        if (m & M_GUMBEL)
            return unit_loop<In, M_LSE | M_GUMBEL>(j, sm, stages, gt, stage, phase, rm, pf_next);
        return unit_loop<In, M_LSE>(j, sm, stages, gt, stage, phase, rm, pf_next);
    } else if constexpr (KIND == K_TREE) {
        if (m & M_GUMBEL)
            return unit_loop<In, M_GUMBEL>(j, sm, stages, gt, stage, phase, rm, pf_next);
        return unit_loop<In, M_ARGMAX>(j, sm, stages, gt, stage, phase, rm, pf_next);
    } else if constexpr (KIND == K_ANYORDER) {
        if (m & M_LSE)
            return unit_loop<In, M_ARGMAX | M_LSE>(j, sm, stages, gt, stage, phase, rm, pf_next);
        return unit_loop<In, M_ARGMAX>(j, sm, stages, gt, stage, phase, rm, pf_next);
    } else if constexpr (KIND == K_SPOT) {
        if (m & M_GUMBEL)
            return unit_loop<In, M_GUMBEL | M_LSE | M_MAX>(j, sm, stages, gt, stage, phase, rm,
                                                           pf_next);
        return unit_loop<In, M_ARGMAX | M_LSE>(j, sm, stages, gt, stage, phase, rm, pf_next);
    } else {
        switch (m) {
        case M_ARGMAX: return unit_loop<In, M_ARGMAX>(j, sm, stages, gt, stage, phase, rm, pf_next);
        case M_LSE: return unit_loop<In, M_LSE>(j, sm, stages, gt, stage, phase, rm, pf_next);
        case M_LSE | M_GUMBEL:
            return unit_loop<In, M_LSE | M_GUMBEL>(j, sm, stages, gt, stage, phase, rm, pf_next);
        case M_ARGMAX | M_LSE:
            return unit_loop<In, M_ARGMAX | M_LSE>(j, sm, stages, gt, stage, phase, rm, pf_next);
        case M_GUMBEL | M_LSE | M_MAX:
            return unit_loop<In, M_GUMBEL | M_LSE | M_MAX>(j, sm, stages, gt, stage, phase, rm, pf_next);
        default:
            return unit_loop<In, M_GUMBEL | M_LSE | M_LSE2 | M_MAX>(j, sm, stages, gt, stage,
                                                                     phase, rm, pf_next);
        }
    }
}

// ---------------------------------------------------------------------------
// The planner warp (lane 0): takes units from the global counter, loads their
// per-sequence values and works out their row modes and records, and queues
// them for the producer -- kPlanQ units ahead, so the producer never waits on
// global memory between two units.  Ends the queue with a kind -1 entry.
// ---------------------------------------------------------------------------
template <int KIND>
__device__ void planner_loop(const Job &j, PassShared &sm)
{
    if ((threadIdx.x & 31) != 0)
        return;
    long long n = 0;  // entries queued
    bool ok = true;
    auto push = [&](const PlanEntry &pe) {
        const int q = (int)(n % kPlanQ);
        if (!mbar_wait(&sm.plan_empty[q], (uint32_t)((n / kPlanQ) & 1) ^ 1u)) {
            ok = false;
            return;
        }
        sm.plan[q] = pe;
        mbar_arrive(&sm.plan_full[q]);  // release: the producer sees the entry
        ++n;
    };
    long long u = (long long)atomicAdd(j.ctl + C_UNIT, 1u);
    UnitPre pre = unit_prefetch(j, u);
    while (ok && u < j.total_units) {
        // Near the end of the pass, claim a unit only once the producer has
        // taken all but one queued entry: units claimed ahead are this CTA's
        // alone, and a deep queue at the end would leave CTAs finishing
        // several units apart.
        if (j.total_units - u < 2LL * gridDim.x && n >= 2 &&
            !mbar_wait(&sm.plan_empty[(n - 2) % kPlanQ], (uint32_t)(((n - 2) / kPlanQ) & 1))) {
            ok = false;
            break;
        }
        const long long un = (long long)atomicAdd(j.ctl + C_UNIT, 1u);
        const UnitPre pn = unit_prefetch(j, un);
        const UnitInfo ci = unit_info(j, u, pre);
        if (ci.valid) {
            PlanEntry pe;
            pe.kind = 0;
            pe.rec = ci.rec;
            pe.b = ci.b;
            pe.expect = ci.expect;
            pe.xid = ci.xid;
            pe.vs = ci.part * j.part_vecs;
            pe.ve = min(j.nvec, pe.vs + j.part_vecs);
            pe.row = slot_row(j, ci.b, ci.slot);
            pe.rm = ci.rm;
            push(pe);
        }
        u = un;
        pre = pn;
    }
    if (!ok)
        latch(j.err, SV_ERR_TIMEOUT);
    PlanEntry end;
    end.kind = -1;
    push(end);
}

template <typename In, int KIND>
__global__ void __launch_bounds__(kPassThreads, SV_MIN_BLOCKS)
    pass_kernel(const __grid_constant__ Job j)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    PassShared &sm = *reinterpret_cast<PassShared *>(smem_raw);
    float *gt = reinterpret_cast<float *>(smem_raw + ((sizeof(PassShared) + 127) & ~size_t(127)));
    unsigned char *stages = reinterpret_cast<unsigned char *>(gt) +
                            ((kGTab * sizeof(float) + 127) & ~size_t(127));
    const int t = threadIdx.x;
    if (t == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        for (int s = 0; s < kStages; ++s)
            sm.thr[s] = f2ord(-INFINITY);
        for (int q = 0; q < kUnitSlots; ++q) {
            mbar_init(&sm.ubar[q], kConsumerWarps);
            mbar_init(&sm.ufree[q], 1);
        }
        for (int q = 0; q < kPlanQ; ++q) {
            mbar_init(&sm.plan_full[q], 1);
            mbar_init(&sm.plan_empty[q], 1);
        }
        mbar_init(&sm.csync, kConsumerWarps);
        for (int w = 0; w < kConsumerWarps; ++w)
            sm.cph[w] = 0u;
        sm.seed_cnt[0] = sm.seed_cnt[1] = 0;
        sm.seed_n = 0;
        sm.abort = 0;
        sm.nunits = 0;
        sm.prod_done = 0;
        sm.fin_qh = sm.fin_qt = 0;
        mbar_fence_init();
    }
    pdl_wait();
    pdl_trigger();
    for (int i = t; i < kGTab; i += blockDim.x)
        gt[i] = __ldg(j.gtab + i);
    if (j.skip)
        for (int i = t; i < kSkipN; i += blockDim.x)
            sm.skip[i] = __ldg(j.skip + i);
    __syncthreads();

    if (t >= kConsumers + 64) {
        // ---------------- planner warp ----------------
        planner_loop<KIND>(j, sm);
    } else if (t >= kConsumers + 32) {
        // ---------------- finalizer warp ----------------
        finalizer_loop<KIND>(j, sm);
    } else if (t >= kConsumers) {
        // ---------------- producer warp ----------------
        // Lane 0 streams the planned units in order.  The entry after the
        // current one is read too: if it carries a Gumbel-max, the current
        // unit's first stage names it, so that the consumers list and copy
        // its top ids while this unit streams.
        if (t == kConsumers) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t pend = 0, pend_par = 0;  // stages with a copy not yet re-acquired
            int lu = 0;                       // local unit number
            bool ok = true;
            const int E = j.dtype == SV_BF16 ? 8 : 4;
            for (long long pi = 0;; ++pi) {
                const int q = (int)(pi % kPlanQ);
                if (!mbar_wait(&sm.plan_full[q], (uint32_t)((pi / kPlanQ) & 1))) {
                    ok = false;
                    break;
                }
                const PlanEntry &ce = sm.plan[q];
                if (ce.kind < 0)
                    break;
                // The next entry only if it is already queued: waiting for it
                // here could wait on a decision that needs this very unit.
                const int q1 = (int)((pi + 1) % kPlanQ);
                const bool have_next =
                    mbar_test(&sm.plan_full[q1], (uint32_t)(((pi + 1) / kPlanQ) & 1));
                const PlanEntry &ne = sm.plan[q1];
                const int step = kStageVecs;
                const bool nseed = have_next && ne.kind == 0 && (ne.rm.mode & M_GUMBEL);
                for (int v = ce.vs; v < ce.ve; v += step) {
                    const int nv = min(step, ce.ve - v);
                    if (!mbar_wait(&sm.empty[stage], phase ^ 1u)) {
                        ok = false;
                        break;
                    }
                    pend &= ~(1u << stage);  // the consumers released it: its copy landed
                    StageMeta &mt = sm.meta[stage];
                    mt.unit = ce.rec;
                    mt.nv = nv;
                    mt.vbase = v;
                    mt.first = (v == ce.vs);
                    mt.last = (v + step >= ce.ve);
                    mt.lu = lu;
                    mt.b = ce.b;
                    mt.expect = ce.expect;
                    mt.xid = ce.xid;
                    mt.row = ce.row;
                    mt.vend = ce.ve;
                    mt.rm = ce.rm;
                    mt.nrec = -1;
                    if (v == ce.vs) {
                        sm.thr[lu % kStages] = f2ord(-INFINITY);
                        if (nseed) {
                            mt.nrec = ne.rec;
                            mt.nrow = ne.row;
                            mt.nkey = ne.rm.key;
                            mt.nlo = ne.vs * E;
                            mt.nhi = ne.ve * E;
                        }
                    }
                    mbar_arrive_tx(&sm.full[stage], (uint32_t)nv * 16u);
                    bulk_g2s(stages + (size_t)stage * kStageBytes, ce.row + (int64_t)v * 16,
                             (uint32_t)nv * 16u, &sm.full[stage]);
                    pend |= 1u << stage;
                    pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                ++lu;
                mbar_arrive(&sm.plan_empty[q]);  // the planner may reuse the slot
            }
            if (ok && mbar_wait(&sm.empty[stage], phase ^ 1u)) {
                pend &= ~(1u << stage);
                sm.meta[stage].unit = -1;
                mbar_arrive(&sm.full[stage]);
            } else {
                latch(j.err, SV_ERR_TIMEOUT);
                sm.abort = 1;
                // Release consumers that wait on the next stage.
                sm.meta[stage].unit = -1;
                mbar_arrive(&sm.full[stage]);
            }
            // units the consumers will hand to the finalizer
            sm.nunits = lu;
            __threadfence_block();
            sm.prod_done = 1;
            // Every copy this warp issued must land before the CTA exits; a
            // stage whose copy was consumed has completed that phase, so the
            // wait returns at once.
            for (int s = 0; s < kStages; ++s)
                if (pend & (1u << s))
                    mbar_wait(&sm.full[s], (pend_par >> s) & 1u);
        }
    } else {
        // ---------------- consumer warps ----------------
        int stage = 0;
        uint32_t phase = 0;
        int pf_next = -1;  // (record << 1 | buffer) of a unit whose top ids were prefetched
        for (;;) {
            if (!mbar_wait(&sm.full[stage], phase)) {
                latch(j.err, SV_ERR_TIMEOUT);
                break;
            }
            if (sm.meta[stage].unit < 0 || sm.abort)
                break;
            const RowMode rm = sm.meta[stage].rm;
            if (!unit_dispatch<In, KIND>(j, sm, stages, gt, stage, phase, rm, pf_next))
                break;
        }
        cp_async_wait_all();  // no copy may be in flight when the CTA exits
    }
    __syncthreads();
    end_decisions<KIND>(j, sm);
    __syncthreads();
    if (t == 0) {
        __threadfence();
        unsigned old = atomicAdd(j.ctl + C_EXIT, 1u);
        if (old + 1u == gridDim.x) {
            // Last CTA out: every decision step has run; reset the counters.
            __threadfence();
            j.ctl[C_UNIT] = 0u;
            j.ctl[C_EXIT] = 0u;
            for (int b = 0; b < j.B; ++b)
                j.seq_done[b] = 0u;
            __threadfence();
        }
    }
}

size_t pass_smem_bytes()
{
    size_t a = (sizeof(PassShared) + 127) & ~size_t(127);
    size_t b = (kGTab * sizeof(float) + 127) & ~size_t(127);
    return a + b + (size_t)kStages * kStageBytes;
}

template <typename In, int KIND>
static cudaError_t set_smem(int smem)
{
    return cudaFuncSetAttribute(pass_kernel<In, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem);
}

// Host-side launchers (the kernels are templates of this translation unit).
cudaError_t pass_setup(int *blocks_per_sm)
{
    const int smem = (int)pass_smem_bytes();
    cudaError_t e = cudaSuccess;
    cudaError_t (*fns[])(int) = {
        set_smem<uint16_t, K_GREEDY>, set_smem<uint16_t, K_SAMPLE>, set_smem<uint16_t, K_TREE>,
        set_smem<uint16_t, K_PACKED>, set_smem<uint16_t, K_SPOT>,   set_smem<uint16_t, K_ANYORDER>,
        set_smem<float, K_GREEDY>,    set_smem<float, K_SAMPLE>,    set_smem<float, K_TREE>,
        set_smem<float, K_PACKED>,    set_smem<float, K_SPOT>,      set_smem<float, K_ANYORDER>};
    for (auto f : fns)
        if (e == cudaSuccess)
            e = f(smem);
    // the grid is sized for the instance with the fewest resident CTAs
    const void *ks[] = {
        (const void *)pass_kernel<uint16_t, K_GREEDY>, (const void *)pass_kernel<uint16_t, K_SAMPLE>,
        (const void *)pass_kernel<uint16_t, K_TREE>,   (const void *)pass_kernel<uint16_t, K_PACKED>,
        (const void *)pass_kernel<uint16_t, K_SPOT>,   (const void *)pass_kernel<uint16_t, K_ANYORDER>,
        (const void *)pass_kernel<float, K_GREEDY>,    (const void *)pass_kernel<float, K_SAMPLE>,
        (const void *)pass_kernel<float, K_TREE>,      (const void *)pass_kernel<float, K_PACKED>,
        (const void *)pass_kernel<float, K_SPOT>,      (const void *)pass_kernel<float, K_ANYORDER>};
    int best = 1 << 30;
    for (const void *k : ks) {
        int n = 0;
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kPassThreads, smem);
        best = n < best ? n : best;
    }
    *blocks_per_sm = best;
    return e;
}

template <typename In>
static cudaError_t launch_in(const Job &j, int grid, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    pdl_config(cfg, at, dim3(grid), dim3(kPassThreads), pass_smem_bytes(), s);
    switch (j.kind) {
    case K_GREEDY: return cudaLaunchKernelEx(&cfg, pass_kernel<In, K_GREEDY>, j);
    case K_SAMPLE: return cudaLaunchKernelEx(&cfg, pass_kernel<In, K_SAMPLE>, j);
    case K_TREE: return cudaLaunchKernelEx(&cfg, pass_kernel<In, K_TREE>, j);
    case K_SPOT: return cudaLaunchKernelEx(&cfg, pass_kernel<In, K_SPOT>, j);
    case K_ANYORDER: return cudaLaunchKernelEx(&cfg, pass_kernel<In, K_ANYORDER>, j);
    default: return cudaLaunchKernelEx(&cfg, pass_kernel<In, K_PACKED>, j);
    }
}

// SPOT preparation, one thread per tree: the masked positions of every state
// (the root's from root_mask; a node's state is its parent's with the
// node's position filled) and the number of rows the tree streams.  A node
// whose parent index is out of range, or whose position is not masked in its
// parent's state, latches SV_ERR_DEVICE_BOUNDS and gets a full state.  A
// tree with nothing masked anywhere has no row to stream, so its outputs
// are written here: nothing accepted and nothing committed.
__global__ void __launch_bounds__(128) spot_prep_kernel(const __grid_constant__ Job j)
{
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= j.B)
        return;
    const int S = j.N + 1;
    const uint64_t all = j.L >= 64 ? ~0ull : ((1ull << j.L) - 1ull);
    uint64_t *mk = j.smask + (int64_t)b * S;
    uint64_t m0 = __ldg(j.root_mask + b) & all;
    mk[0] = m0;
    unsigned cnt = (unsigned)__popcll(m0);
    for (int n = 0; n < j.N; ++n) {
        const int par = __ldg(j.parent + (int64_t)b * j.N + n);
        const int pos = __ldg(j.node_pos + (int64_t)b * j.N + n);
        uint64_t m = 0ull;
        if (par < -1 || par >= n || pos < 0 || pos >= j.L ||
            !((mk[par + 1] >> pos) & 1ull))
            latch(j.err, SV_ERR_DEVICE_BOUNDS);
        else
            m = mk[par + 1] & ~(1ull << pos);
        mk[n + 1] = m;
        cnt += (unsigned)__popcll(m);
    }
    j.svalid[b] = cnt;
    if (cnt == 0u) {
        j.path_len[b] = 0;
        j.commit_count[b] = 0;
        j.commit_pos[b] = -1;
        j.commit_tok[b] = -1;
        if (j.flags) j.flags[b] = 0;
        for (int k = 0; k < j.max_depth; ++k)
            j.path_nodes[(int64_t)b * j.max_depth + k] = -1;
        for (int n = 0; n < j.N && j.match; ++n)
            j.match[(int64_t)b * j.N + n] = 0;
        for (int st = 0; st < S; ++st) {
            if (j.state_pos) j.state_pos[(int64_t)b * S + st] = -1;
            if (j.state_tok) j.state_tok[(int64_t)b * S + st] = -1;
        }
    }
}

cudaError_t spot_prep_launch(const Job &j, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    pdl_config(cfg, at, dim3((j.B + 127) / 128), dim3(128), 0, s);
    return cudaLaunchKernelEx(&cfg, spot_prep_kernel, j);
}

// Any-order preparation, one thread per sequence: checks that the first u
// entries of the order are a permutation of the window indices, finds kappa
// (the leading ranks with a draft token), the verify rows needed (min(kappa
// + 1, u), which must not exceed the K verify rows given) and the rows to
// stream.  Bad inputs latch SV_ERR_DEVICE_BOUNDS and stream nothing; a
// sequence with nothing to stream gets its outputs here.
__global__ void __launch_bounds__(128) anyorder_prep_kernel(const __grid_constant__ Job j)
{
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= j.B)
        return;
    const int W = j.W;
    const int uin = __ldg(j.lens + b);
    bool bad = uin < 0 || uin > W;
    const int u = bad ? 0 : uin;
    unsigned seen = 0u;
    int kappa = 0;
    bool run = true;
    for (int r = 0; r < u; ++r) {
        const int oi = __ldg(j.order + (int64_t)b * W + r);
        if (oi < 0 || oi >= u || ((seen >> oi) & 1u)) {
            bad = true;
            break;
        }
        seen |= 1u << oi;
        run = run && __ldg(j.ids + (int64_t)b * W + oi) >= 0;
        kappa += run ? 1 : 0;
    }
    const int nreq = min(kappa + 1, u);
    bad = bad || nreq > j.K;
    if (bad)
        latch(j.err, SV_ERR_DEVICE_BOUNDS);
    j.smask[b] = bad ? 0ull : (uint64_t)nreq;
    j.svalid[b] = bad ? 0u : (unsigned)(nreq + u);
    if (bad || u == 0) {
        j.acc[b] = 0;
        j.commit_len[b] = 0;
        j.end_out[b] = __ldg(j.end_in + b);
        for (int i = 0; i < W; ++i) {
            j.commit_pos[(int64_t)b * W + i] = -1;
            j.commit_tok[(int64_t)b * W + i] = -1;
            j.next_draft[(int64_t)b * W + i] = -1;
            j.next_order[(int64_t)b * W + i] = -1;
            if (j.confidence) j.confidence[(int64_t)b * W + i] = __int_as_float(0x7FC00000);
        }
    }
}

cudaError_t anyorder_prep_launch(const Job &j, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    pdl_config(cfg, at, dim3((j.B + 127) / 128), dim3(128), 0, s);
    return cudaLaunchKernelEx(&cfg, anyorder_prep_kernel, j);
}

cudaError_t pass_launch(const Job &j, int grid, cudaStream_t s)
{
    return j.dtype == SV_BF16 ? launch_in<uint16_t>(j, grid, s) : launch_in<float>(j, grid, s);
}

}  // namespace sv
