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

struct RowMode {
    int mode;
    float c1, c2, invT;
    float thr0;       // Gumbel-max rows: the threshold the row's seed records give
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
    int pad;
    const char *row;  // the unit's logit row
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
    volatile int abort;
    // Gumbel vectors that passed level 1, per consumer warp: raw data and
    // the vector's index in the row
    uint4 gqd[kConsumerWarps][kGQ];
    uint32_t gqv[kConsumerWarps][kGQ];
    Cand2 gcand[kConsumerWarps];  // each consumer warp's Gumbel candidates of its unit
    uint64_t skip[kSkipN];   // skip thresholds of the top-id draws
    // unit slots: consumer warps write their partials and arrive on ubar; the
    // finalizer merges them and arrives on ufree
    uint64_t ubar[kUnitSlots];
    uint64_t ufree[kUnitSlots];
    WarpPart up[kUnitSlots][kConsumerWarps];
    int uunit[kUnitSlots], ub[kUnitSlots];
    unsigned uexpect[kUnitSlots];
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
    int ida;       // the draft token a light unit's row is tested on (or -1)
    uint64_t smask;   // SPOT: masked positions of the unit's state
    unsigned svalid;  // SPOT: rows the tree streams
};

// Unit order.  Rows that carry a Gumbel-max (a few times the work of a plain
// row) are streamed first, H per sequence, so that the last units of the pass
// are light ones and CTAs finish together; the other rows follow sequence by
// sequence.  A unit is one part of one row.
__device__ __forceinline__ int heavy_rows(const Job &j)
{
    return (j.kind == K_PACKED && j.Tp != 0.f) ? j.W : 0;  // the proposal rows
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
        slot = j.K + r;
    } else {
        const long long rem = (u - nh) - (long long)b * (j.rows_per_seq - H) * j.parts;
        const int r = (int)(rem / j.parts);
        part = (int)(rem - (long long)r * j.parts);
        slot = r;
    }
}

// Calls whose rows record the logit at a draft token: the target and drafter
// rows of a sampling call, the verify rows of a Packed-SS step at T > 0.
__device__ __forceinline__ bool has_drafts(const Job &j)
{
    return j.kind == K_SAMPLE || (j.kind == K_PACKED && j.Tp != 0.f);
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
    UnitPre p{0, 0, 0, -1, 0ull, 0u};
    if (u >= j.total_units)
        return p;
    const int b = unit_seq(j, u);
    const int H = heavy_rows(j);
    const long long nh = (long long)j.B * H * j.parts;
    if (has_drafts(j) && u >= nh) {
        // a light unit's slot is its rank among the light rows
        const long long rem = (u - nh) - (long long)b * (j.rows_per_seq - H) * j.parts;
        p.ida = draft_token(j, b, (int)(rem / j.parts));
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
    r.thr0 = -INFINITY;
    r.T = 1.0;
    r.key = 0;
    switch (j.kind) {
    case K_GREEDY:
        r.mode = M_ARGMAX;
        break;
    case K_SAMPLE:
        r.mode = M_LSE;
        r.c1 = slot <= j.K ? j.cp : j.cq;
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
    if (has_drafts(j) && u >= (long long)j.B * H * j.parts) {
        const int pos = draft_pos(j, i.slot);
        if (pos >= 0 && pos < n) {
            const int d = p.ida;
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
    if ((i.rm.mode & M_GUMBEL) && j.seeds) {
        const int k = gumbel_index(j, i.slot);
        const SeedRec *sr = j.seeds + ((int64_t)i.b * gumbel_rows(j) + k) * j.seed_chunks;
        for (int q = 0; q < j.seed_chunks; ++q)
            i.rm.thr0 = fmaxf(i.rm.thr0, __ldcg(&sr[q].thr));
    }
    return i;
}

// Gumbel part of a thread's state: the thresholds only (passed by value to
// the out-of-line queue screen, so that they stay in registers).  The
// candidates are kept per warp in shared memory (PassShared::gcand), written
// only by that screen, so that the stream loop does not hold them.
struct GState {
    float thr, thrS;   // level-2 and level-1 thresholds
};

// Per-thread running state of one unit.
struct TState {
    float e1, e2;      // integer reference exponents of the sums (-inf: none yet)
    float2 acc1, acc2; // sums of 2^fl(x c - e), as fp32 pairs
    float mx;          // running max
    int amax;
    GState g;
    int gqn;           // groups in this warp's queue (warp-uniform)
    float xd;          // logit at the unit's draft token (its owner thread), else NaN
};

__device__ __forceinline__ void tstate_init(TState &s)
{
    s.e1 = s.e2 = -INFINITY;
    s.acc1 = s.acc2 = make_float2(0.f, 0.f);
    s.mx = -INFINITY;
    s.amax = 0x7FFFFFFF;
    s.g.thr = s.g.thrS = -INFINITY;
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
// threshold are kept, and their lower end raises the threshold (anything
// below it - 1e-9 can neither win nor tie within 1e-9).
__device__ __forceinline__ void gumbel_level2(float x, uint32_t v, bool top, GState &s,
                                              Cand2 &c, float invT, uint64_t key)
{
    const float2 iv = logit_interval_at(x, invT, key, v, top);
    const float lo = iv.x, hi = iv.y;
    if (hi < s.thr)
        return;
    c.add(lo, hi, (int)v);
    raise_thr(s, __fsub_rd(lo, 1e-9f));
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
// ex2 per element; a pairwise tree over each vector's element pairs, and the
// vectors' sums chained in order (so that a vector's registers are free once
// it is summed).
template <typename In>
__device__ __forceinline__ float2 lse_terms(const Chunk &q, float c, float e)
{
    using VT = VecTraits<In>;
    constexpr int P = VT::P;  // element pairs per vector
    const float2 cc = make_float2(c, c), ne = make_float2(-e, -e);
    float2 part = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k) {
        float2 t[P];
#pragma unroll
        for (int i = 0; i < P; ++i) {
            const float2 y = fma2(VT::pair(q[k], i), cc, ne);
            t[i] = make_float2(ex2f(y.x), ex2f(y.y));
        }
#pragma unroll
        for (int w = 1; w < P; w <<= 1)
#pragma unroll
            for (int i = 0; i + w < P; i += 2 * w)
                t[i] = add2(t[i], t[i + w]);
        part = k == 0 ? t[0] : add2(part, t[0]);
    }
    return part;
}

// Adds the chunk to one log-sum-exp accumulator, given the chunk max cm.
// The first chunk with an element sets the reference e to ceil(cm c); a later
// chunk whose max would give a term of 2^20 or more (ceil(cm c) > e + 20)
// first moves the reference up to ceil(cm c) and rescales the accumulator
// exactly.  Every term's exponent x c - e thus stays below kLseCap + 1, and
// the test needs only the chunk max, so the warp does not wait on the sum
// before going on.
template <typename In>
__device__ __forceinline__ void lse_chunk(const Chunk &q, float c, float cm, float &e,
                                          float2 &acc)
{
    if (cm == -INFINITY)
        return;  // nothing but padding
    const float ec = ceilf(__fmul_ru(cm, c));
    if (!(ec <= e + kLseCap)) {  // the first chunk (e = -inf) or a new, larger max
        if (e > -INFINITY) {
            const float sc = pow2_int(e - ec);
            acc.x *= sc;
            acc.y *= sc;
        }
        e = ec;
    }
    acc = add2(acc, lse_terms<In>(q, c, e));
}

// Running max, and with ARG its lowest index: the first vector whose max is
// the chunk max, then the first element of it that equals it (predicated
// selects, no search loop).
template <typename In, bool ARG>
__device__ __forceinline__ float max_chunk(const Chunk &q, int vbase, TState &s)
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
    return cm;
}

// Per-id screen of the queued vectors, 32 at a time, a vector per lane: its
// top ids are skipped (the seed kernel scored every top id of the row); an
// ordinary id is bounded by the top byte of its fine bits, and survivors get
// the fp32 interval of level 2.  The lanes' candidates are merged into the
// warp's (wc, in shared memory), and every lane leaves with the warp's best
// threshold.  Whole warp.
template <typename In>
__device__ __noinline__ GState gumbel_flush(const uint4 *__restrict__ qd,
                                            const uint32_t *__restrict__ qv, int n, GState s,
                                            float invT, uint64_t key, const float *__restrict__ gt,
                                            const uint64_t *__restrict__ skip, Cand2 *wc)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    Cand2 c;
    c.init();
    __syncwarp();
    for (int i = (int)(threadIdx.x & 31); i < n; i += 32) {
        const uint4 d = qd[i];
        const uint32_t v0 = qv[i] * E;
        const uint32_t tm = top_mask(key, v0 >> 8, (int)(v0 & 255u), E, skip);
#pragma unroll 1
        for (int e = 0; e < E; ++e) {
            if ((tm >> e) & 1u)
                continue;
            const uint32_t v = v0 + e;
            const float x = VT::elem(d, e);
            const uint64_t m = fine52(key, v);
            if (fmaf(x, invT, gt[(int)(m >> 44)]) >= s.thrS)
                gumbel_level2(x, v, false, s, c, invT, key);
        }
    }
    warp_cand2(c);
    if ((threadIdx.x & 31) == 0)
        wc->merge(c);
    raise_thr(s, warp_max(s.thr));
    __syncwarp();
    return s;
}

// Level 1 on whole vectors: an ordinary id's G stays below gmax (the table's
// last entry), so a vector is queued only if its largest logit can reach the
// threshold with that bound.  The comparison is strict: a bound equal to the
// level-1 threshold stays below thr (the threshold's margin exceeds the
// bound's rounding slack), and the -inf padding of a short stage never passes,
// not even a threshold of -inf.  The chunk is tested first on its largest
// logit with one vote per warp (with the seed threshold, nearly every chunk
// stops there); otherwise gumbel_queue tests each vector, re-read from the
// stage, and queues the passing ones, compacted with a ballot, so a warp does
// not diverge per vector.  Each warp keeps its own threshold (the seed
// records give every warp the row's top-id threshold at the start).
struct GQueue {
    GState g;
    int n;  // vectors in the warp's queue (warp-uniform)
};

template <typename In>
__device__ __noinline__ GQueue gumbel_queue(const uint4 *__restrict__ st, int nv, int vbase,
                                            GQueue q, float invT, uint64_t key, float gmax,
                                            const float *__restrict__ gt,
                                            const uint64_t *__restrict__ skip, PassShared &sm)
{
    using VT = VecTraits<In>;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    uint4 *qd = sm.gqd[w];
    uint32_t *qv = sm.gqv[w];
#pragma unroll 1
    for (int k = 0; k < kVecsPerThread; ++k) {
        const int idx = t + k * kConsumers;
        const uint4 v = idx < nv ? st[idx] : VT::neg_inf_vec();
        const bool pass = fmaf(VT::hi_of(VT::pmax(v)), invT, gmax) > q.g.thrS;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, pass);
        if (bal) {
            if (pass) {
                const int r = q.n + __popc(bal & ((1u << lane) - 1u));
                qd[r] = v;
                qv[r] = (uint32_t)(vbase + idx);
            }
            q.n += __popc(bal);
            if (q.n > kGQ - 32) {
                q.g = gumbel_flush<In>(qd, qv, q.n, q.g, invT, key, gt, skip, &sm.gcand[w]);
                q.n = 0;
            }
        }
    }
    return q;
}

template <typename In>
__device__ __forceinline__ void gumbel_chunk(const uint4 *__restrict__ st, int nv, float cm,
                                             int vbase, TState &s, const RowMode &rm, float gmax,
                                             const float *__restrict__ gt,
                                             const uint64_t *__restrict__ skip, PassShared &sm)
{
    if (!__any_sync(0xFFFFFFFFu, fmaf(cm, rm.invT, gmax) > s.g.thrS))
        return;
    GQueue q{s.g, s.gqn};
    q = gumbel_queue<In>(st, nv, vbase, q, rm.invT, rm.key, gmax, gt, skip, sm);
    s.g = q.g;
    s.gqn = q.n;
}

template <typename In, int MODE>
__device__ __forceinline__ void do_chunk(const uint4 *__restrict__ st, int nv, int vbase, TState &s,
                                         const RowMode &rm, float gmax,
                                         const float *__restrict__ gt, PassShared &sm)
{
    Chunk q;
    load_chunk<In>(st, nv, q);
    float cm = -INFINITY;
    if (MODE & (M_ARGMAX | M_MAX))
        cm = max_chunk<In, (MODE & M_ARGMAX) != 0>(q, vbase, s);
    else
        cm = chunk_max<In>(q);
    if (MODE & M_LSE)
        lse_chunk<In>(q, rm.c1, cm, s.e1, s.acc1);
    if (MODE & M_LSE2)
        lse_chunk<In>(q, rm.c2, cm, s.e2, s.acc2);
    if (MODE & M_GUMBEL)
        gumbel_chunk<In>(st, nv, cm, vbase, s, rm, gmax, gt, sm.skip, sm);
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
    double cg0 = 0.0, cg3 = 1.0, cplo = 0.0, cphi = 1.0;  // its inputs, lane by lane
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
        double u = uniform_at(rng_key(j.seed, kAccept, (uint64_t)b, p0 + lane, 0), 0, j.skip);
        // Cactus: gamma* >= p gives alpha >= the lossless alpha (alo, ahi
        // above), so a sure lossless accept is a sure accept; other lanes
        // bracket gamma* over p's bracket (it grows with p), then alpha =
        // gamma* / q and the residual scale c = (1 - gamma*)/(1 - p)
        if (j.amode == SV_LENIENT_CACTUS && !(u < alo - kFlagEps)) {
            // brackets of p and q: exp_fast (within 2^-21 of exp) widened by
            // 2^-20; fp64 below -80, where fp32 would underflow
            auto lo = [](double a) { return a > -80.0 ? exp_fast(a) * (1.0 - 0x1p-20) : exp(a); };
            auto hi = [](double a) { return a > -80.0 ? exp_fast(a) * (1.0 + 0x1p-20) : exp(a); };
            const double plo = lo(lp - 1.01 * ep - 1e-13), phi = hi(lp + 1.01 * ep + 1e-13);
            const double qlo = lo(lq - 1.01 * eq - 1e-13), qhi = hi(lq + 1.01 * eq + 1e-13);
            double g0, g3;
            const bool ok = cactus_bracket_fast(plo, phi, (double)j.lam, j.cactus_emd, &g0, &g3);
            alo = ok ? fmin(1.0, g0 / qhi) : 0.0;
            ahi = ok ? fmin(1.0, g3 / qlo) : 1.0;
            cg0 = g0;
            cg3 = g3;
            cplo = plo;
            cphi = phi;
        }
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
    // the residual scale's bracket, at the rejected position only
    if (j.amode == SV_LENIENT_CACTUS && lane == f && f < n) {
        lclo = (cg3 < 1.0) ? log1p(-cg3) - log1p(-cplo) : -INFINITY;
        lchi = log1p(-cg0) - log1p(-cphi);
    }
    const double lcloh = __shfl_sync(0xFFFFFFFFu, lclo, f & 31);
    const double lchih = __shfl_sync(0xFFFFFFFFu, lchi, f & 31);
    // bonus row n (always valid): its log-sum-exp; its Gumbel-max with key
    // (SAMPLE, pos + n) is drawn by the residual pass, and only when every
    // draft is accepted
    const double Lb = __shfl_sync(0xFFFFFFFFu, rp.L1a, n);
    const float mb = __shfl_sync(0xFFFFFFFFu, rp.m, n);
    if (lane == 0) {
        if (j.lse_p) j.lse_p[(int64_t)b * (j.K + 1) + n] = (float)Lb;
        RowStat *sb = j.rs_stat + (int64_t)b * j.rows_per_seq + n;
        sb->L1 = Lb;
        sb->m = mb;
        if (rescue) {
            unsigned e = atomicAdd(j.ctl + C_RESCUE_N, 1u);
            j.rescue[e].b = b;
            j.rescue[e].kind = 0;
            j.rescue[e].h = 0;
            j.rescue[e].bonus = 0;
        } else {
            // the correction at the first rejection f < n, or the bonus
            // token when f == n: both by the residual pass
            j.acc[b] = f;
            unsigned e = atomicAdd(j.ctl + C_RESID_N, 1u);
            ResidEntry re;
            re.b = b;
            re.h = f;
            re.need_lq = 0;
            re.bonus = f == n;
            re.prow = row_ptr(j, b, f);
            re.qrow = f == n ? re.prow : row_ptr(j, b, j.K + 1 + f);
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
            j.rescue[e].bonus = 0;
        }
        return;
    }
    // The token at position f -- the correction from [p - Q]_+ after a
    // rejection, or the bonus (the Gumbel-max of row n) when every draft is
    // accepted -- is drawn by the residual pass; it is the last committed
    // token, so the stopping index does not depend on it.
    packed_commit(j, b, f, -1, false, 0);
    if (lane == 0) {
        int off = __ldg(j.prev_off + b);
        unsigned e = atomicAdd(j.ctl + C_RESID_N, 1u);
        ResidEntry re;
        re.b = b;
        re.h = f;
        re.need_lq = f < n;
        re.bonus = f == n;
        re.prow = row_ptr(j, b, f);
        re.qrow = f < n ? j.src2 + ((int64_t)b * j.W + off + f) * j.rs : re.prow;
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

// max_v softmax(x)_v = 1 / S, S = sum_v exp(x_v - max x), of one row, by the
// whole warp (16-byte loads), for the rare states whose streamed confidences
// do not separate their best position by the 1e-9 window.
//   conf_row_refined: S from CUDA's expf (documented within 2 ulp) with a
//     compensated fp32 sum per lane and an fp64 sum over the lanes: the
//     interval [*lo, *hi] of the confidence has relative half-width 5e-7.
//   conf_row64: S in fp64 (exp of the fp64 difference), for contenders that
//     the refined intervals still do not separate.
template <bool EXACT>
static __device__ __noinline__ double conf_row_sum(const Job &j, const char *row, float *mout)
{
    const int lane = threadIdx.x & 31;
    const uint4 *r4 = reinterpret_cast<const uint4 *>(row);
    const bool bf = j.dtype == SV_BF16;
    float m = -INFINITY;
    for (int k = lane; k < j.nvec; k += 32) {
        const uint4 q = __ldg(r4 + k);
        m = fmaxf(m, bf ? VecTraits<uint16_t>::hi_of(VecTraits<uint16_t>::pmax(q))
                        : VecTraits<float>::hi_of(VecTraits<float>::pmax(q)));
    }
    m = warp_max(m);
    *mout = m;
    double sd = 0.0;
    float sf = 0.f, cf = 0.f;  // compensated fp32 sum
    for (int k = lane; k < j.nvec; k += 32) {
        const uint4 q = __ldg(r4 + k);
        float f[8];
        int ne = 8;
        if (bf) {
            VecTraits<uint16_t>::unpack(q, f);
        } else {
            float g[4];
            VecTraits<float>::unpack(q, g);
            for (int e = 0; e < 4; ++e) f[e] = g[e];
            ne = 4;
        }
        for (int e = 0; e < ne; ++e) {
            if (EXACT) {
                sd += exp((double)f[e] - (double)m);
            } else {
                const float y = expf(f[e] - m) - cf;  // f - m is exact for bf16 and fp32
                const float t = sf + y;
                cf = (t - sf) - y;
                sf = t;
            }
        }
    }
    return warp_sumd(EXACT ? sd : (double)sf);
}

static __device__ __forceinline__ void conf_row_refined(const Job &j, const char *row, double *lo,
                                                        double *hi)
{
    float m;
    const double S = conf_row_sum<false>(j, row, &m);
    *lo = 1.0 / (S * (1.0 + 5e-7));
    *hi = 1.0 / (S * (1.0 - 5e-7));
}

static __device__ __forceinline__ double conf_row64(const Job &j, const char *row)
{
    float m;
    return 1.0 / conf_row_sum<true>(j, row, &m);
}

static __device__ __noinline__ void fin_spot(const Job &j, int b)
{
    const int lane = threadIdx.x & 31;
    const int S = j.N + 1, L = j.L;
    const int64_t p0 = pos0_of(j, b);
    // relative error of a confidence exp(m - L1) from the streamed sums
    const double e = 1.01 * j.eps_lse + 0x1p-21 + 1e-13;
    // sp[r], sv[r]: Phi of state lane + 32 r (position, token)
    int sp[3] = {-1, -1, -1}, sv[3] = {-1, -1, -1}, nflag = 0;
    for (int st = 0; st < S; ++st) {
        const uint64_t mk = __ldg(j.smask + (int64_t)b * S + st);
        if (mk == 0ull)
            continue;
        // lane = position: its row's confidence interval
        const bool has = lane < L && ((mk >> lane) & 1ull);
        float c = -1.f;
        double lo = -1.0, hi = -1.0;
        int am = -1;
        if (has) {
            const RowM rm = merge_row(j, b, st * L + lane, j.cr1, 1.0);
            c = exp_fast((double)rm.m - rm.L1a);
            lo = (double)c * (1.0 - e);
            hi = (double)c * (1.0 + e);
            am = rm.amax;
        }
        // the best by (confidence desc, position asc) and the largest upper
        // end among the other masked positions
        const uint32_t cm = __reduce_max_sync(0xFFFFFFFFu, f2ord(c));
        const unsigned tie = __ballot_sync(0xFFFFFFFFu, has && f2ord(c) == cm);
        int bs = __ffs(tie) - 1;
        const double blo = __shfl_sync(0xFFFFFFFFu, lo, bs);
        const float oh = (has && lane != bs) ? __double2float_ru(hi) : -1.f;
        const double ohi = (double)ord2f(__reduce_max_sync(0xFFFFFFFFu, f2ord(oh)));
        int v = __shfl_sync(0xFFFFFFFFu, am, bs);
        if (ohi >= 0.0 && __double2float_rd(blo) - ohi < kFlagEps) {
            // not separated by the streamed bounds: the contenders get the
            // refined intervals (lane = position); those still within reach
            // of the best are recomputed in fp64
            unsigned ct = __ballot_sync(0xFFFFFFFFu, has && hi >= blo - kFlagEps);
            double rlo = -1.0, rhi = -1.0;
            for (unsigned cm2 = ct; cm2; cm2 &= cm2 - 1) {
                const int s = __ffs(cm2) - 1;
                double a0, a1;
                conf_row_refined(j, row_ptr(j, b, st * L + s), &a0, &a1);
                if (lane == s) {
                    rlo = a0;
                    rhi = a1;
                }
            }
            // the best refined lower end and whether another upper end
            // comes within 1e-9 of it
            double best = -1.0;
            int s1 = -1;
            for (int o = 0; o < 32; ++o) {
                const double x = __shfl_sync(0xFFFFFFFFu, rlo, o);
                if ((ct >> o) & 1u && x > best) {
                    best = x;
                    s1 = o;
                }
            }
            const bool close = ((ct >> lane) & 1u) && lane != s1 && rhi >= best - kFlagEps;
            const unsigned cl = __ballot_sync(0xFFFFFFFFu, close);
            if (cl) {
                unsigned cx = cl | (1u << s1);
                double c1 = -1.0, c2 = -1.0;
                s1 = -1;
                while (cx) {  // ascending positions: the lowest wins exact ties
                    const int s = __ffs(cx) - 1;
                    cx &= cx - 1;
                    const double x = conf_row64(j, row_ptr(j, b, st * L + s));
                    if (x > c1) {
                        c2 = c1;
                        c1 = x;
                        s1 = s;
                    } else if (x > c2) {
                        c2 = x;
                    }
                }
                if (lane == 0 && c1 - c2 > 0.0 && c1 - c2 < kFlagEps)
                    ++nflag;
            }
            bs = s1;
            v = __shfl_sync(0xFFFFFFFFu, am, bs);
        }
        if (lane == (st & 31)) {
            sp[st >> 5] = bs;
            sv[st >> 5] = v;  // the argmax; replaced by the Gumbel-max at T > 0
        }
    }
    // T > 0: the token at s* is the coupled-noise Gumbel-max of that row
    if (j.Tp != 0.f) {
        for (int r = 0; r < 3; ++r) {
            const int st = lane + 32 * r;
            const bool has = st < S && sp[r] >= 0;
            Cand2 gc;
            gc.init();
            if (has)
                gc = merge_row(j, b, st * L + sp[r], j.cr1, 1.0).gc;
            const GRes g = resolve_lanes(j, row_ptr(j, b, has ? st * L + sp[r] : 0),
                                         rng_key(j.seed, kTree, (uint64_t)b,
                                                 p0 + (has ? sp[r] : 0), 0),
                                         (double)j.Tp, j.invTp, gc, has);
            if (has) {
                sv[r] = g.v;
                nflag += g.flag;
            }
        }
    }
    for (int r = 0; r < 3; ++r) {
        const int st = lane + 32 * r;
        if (st < S) {
            if (j.state_pos) j.state_pos[(int64_t)b * S + st] = sp[r];
            if (j.state_tok) j.state_tok[(int64_t)b * S + st] = sv[r];
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
// order and also window index r.  The scores are returned for the caller's
// order policy, which ranks the next window (App. C "Procedure").
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
    // temperature 1
    int z = -1;
    double sc = -1.0;
    if (lane < u) {
        const RowM rm = merge_row(j, b, j.K + lane, j.cr1, 1.0);
        z = rm.amax;
        sc = (double)exp_fast((double)rm.m - rm.L1a);
    }
    const int wpos = lane < u ? __ldg(wp + lane) : 0x7FFFFFFF;
    const bool ret = lane < u && !((accd >> lane) & 1u) && wpos <= E;
    if (lane < W) {
        j.next_draft[(int64_t)b * W + lane] = ret ? z : -1;
        if (j.confidence)
            j.confidence[(int64_t)b * W + lane] =
                lane < u ? (float)sc : __int_as_float(0x7FC00000);
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
    Cand2 g;
    g.init();
    if (gum) {
        __syncwarp();
        g = sm.gcand[w];
    }
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

// Streams one unit whose first stage is ready in `stage`: every stage of the
// unit with the row mode fixed at compile time, then the unit's partial.
// Returns false if a wait timed out or the producer aborted.
template <typename In, int MODE>
__device__ __forceinline__ bool unit_loop(const Job &j, PassShared &sm, unsigned char *stages,
                                          const float *gt, int &stage, uint32_t &phase,
                                          const RowMode &rm)
{
    const int lane = threadIdx.x & 31;
    const StageMeta &m0 = sm.meta[stage];
    const UnitHead uh{m0.unit, m0.lu, m0.b, m0.expect, m0.xid};
    TState s;
    tstate_init(s);
    // a Gumbel-max row starts from the threshold of its top ids, scored
    // before the stream (the screen below skips them)
    const float gmax = (MODE & M_GUMBEL) ? g_ordinary_max(gt) : 0.f;
    if (MODE & M_GUMBEL) {
        raise_thr(s.g, rm.thr0);
        if (lane == 0)
            sm.gcand[threadIdx.x >> 5].init();
    }
    for (;;) {
        const StageMeta &mt = sm.meta[stage];
        const int nv = mt.nv, vbase = mt.vbase, last = mt.last;
        const uint4 *st = reinterpret_cast<const uint4 *>(stages + (size_t)stage * kStageBytes);
        do_chunk<In, MODE>(st, nv, vbase, s, rm, gmax, gt, sm);
        if (uh.xid >= 0) {
            // the thread that holds the draft token's vector records its logit
            constexpr int E = VecTraits<In>::N;
            const int iv = uh.xid / E - vbase;
            if (iv >= 0 && iv < nv && (int)threadIdx.x == iv % kConsumers)
                s.xd = VecTraits<In>::elem(st[iv], uh.xid % E);
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
        s.g = gumbel_flush<In>(sm.gqd[w], sm.gqv[w], s.gqn, s.g, rm.invT, rm.key, gt, sm.skip,
                               &sm.gcand[w]);
        s.gqn = 0;
    }
    finish_unit(j, uh, s, rm, sm);
    return true;
}

// Only the row modes of entry-point kind KIND are instantiated.
template <typename In, int KIND>
__device__ __forceinline__ bool unit_dispatch(const Job &j, PassShared &sm, unsigned char *stages,
                                              const float *gt, int &stage, uint32_t &phase,
                                              const RowMode &rm)
{
    const int m = rm.mode;
    if constexpr (KIND == K_GREEDY) {
        return unit_loop<In, M_ARGMAX>(j, sm, stages, gt, stage, phase, rm);
    } else if constexpr (KIND == K_SAMPLE) {
        return unit_loop<In, M_LSE>(j, sm, stages, gt, stage, phase, rm);
    } else if constexpr (KIND == K_TREE) {
        if (m & M_GUMBEL)
            return unit_loop<In, M_GUMBEL>(j, sm, stages, gt, stage, phase, rm);
        return unit_loop<In, M_ARGMAX>(j, sm, stages, gt, stage, phase, rm);
    } else if constexpr (KIND == K_ANYORDER) {
        if (m & M_LSE)
            return unit_loop<In, M_ARGMAX | M_LSE>(j, sm, stages, gt, stage, phase, rm);
        return unit_loop<In, M_ARGMAX>(j, sm, stages, gt, stage, phase, rm);
    } else if constexpr (KIND == K_SPOT) {
        if (m & M_GUMBEL)
            return unit_loop<In, M_GUMBEL | M_LSE | M_MAX>(j, sm, stages, gt, stage, phase, rm);
        return unit_loop<In, M_ARGMAX | M_LSE>(j, sm, stages, gt, stage, phase, rm);
    } else {
        switch (m) {
        case M_ARGMAX: return unit_loop<In, M_ARGMAX>(j, sm, stages, gt, stage, phase, rm);
        case M_LSE: return unit_loop<In, M_LSE>(j, sm, stages, gt, stage, phase, rm);
        case M_ARGMAX | M_LSE:
            return unit_loop<In, M_ARGMAX | M_LSE>(j, sm, stages, gt, stage, phase, rm);
        case M_GUMBEL | M_LSE | M_MAX:
            return unit_loop<In, M_GUMBEL | M_LSE | M_MAX>(j, sm, stages, gt, stage, phase, rm);
        default:
            return unit_loop<In, M_GUMBEL | M_LSE | M_LSE2 | M_MAX>(j, sm, stages, gt, stage,
                                                                     phase, rm);
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
        for (int q = 0; q < kUnitSlots; ++q) {
            mbar_init(&sm.ubar[q], kConsumerWarps);
            mbar_init(&sm.ufree[q], 1);
        }
        for (int q = 0; q < kPlanQ; ++q) {
            mbar_init(&sm.plan_full[q], 1);
            mbar_init(&sm.plan_empty[q], 1);
        }
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
        // Lane 0 streams the planned units in order.
        if (t == kConsumers) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t pend = 0, pend_par = 0;  // stages with a copy not yet re-acquired
            int lu = 0;                       // local unit number
            bool ok = true;
            for (long long pi = 0;; ++pi) {
                const int q = (int)(pi % kPlanQ);
                if (!mbar_wait(&sm.plan_full[q], (uint32_t)((pi / kPlanQ) & 1))) {
                    ok = false;
                    break;
                }
                const PlanEntry &ce = sm.plan[q];
                if (ce.kind < 0)
                    break;
                const int step = kStageVecs;
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
                    mt.rm = ce.rm;
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
        for (;;) {
            if (!mbar_wait(&sm.full[stage], phase)) {
                latch(j.err, SV_ERR_TIMEOUT);
                break;
            }
            if (sm.meta[stage].unit < 0 || sm.abort)
                break;
            const RowMode rm = sm.meta[stage].rm;
            if (!unit_dispatch<In, KIND>(j, sm, stages, gt, stage, phase, rm))
                break;
        }
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

// ---------------------------------------------------------------------------
// Seed kernel.  Before the stream, every top id (an id whose uniform lies in
// the top 1/256, about one per block of 256 ids) of every Gumbel-max row of
// the call is found by its skip draws, its logit is loaded, and it is scored
// in an fp32 interval.  The blocks of all Gumbel-max rows, laid end to end,
// are split into equal spans, one per warp (one resident wave of warps);
// a span covers pieces of one or more rows.  A piece's record, the best
// lower end - 1e-9 (a threshold no winner can fall below) and the piece's
// candidates, goes to the row's record numbered by the span boundaries that
// lie inside the row before the piece; the warp that ends a row also writes
// its unused records as empty.
//
// The warp first lists a piece's top ids in shared memory: each lane walks
// one block a draw at a time and, when its block ends, takes the next block
// of the piece, so that the lanes stay busy although blocks hold different
// numbers of top ids; new ids are appended with a ballot, and each listed
// id's logit is copied to shared memory asynchronously while the draws go
// on.  The list is then scored with every lane converged, two ids a lane:
// first the best lower bound of the batch (logit and a table of G lower
// bounds by the top byte of the fine bits) raises the threshold; then an id
// is bounded by its logit and the matching upper bound, and only ids whose
// bound reaches the threshold get the fp32 interval.  Warps never wait for
// one another; the streaming pass starts every Gumbel-max unit from its
// row's threshold and skips top ids, and the decision step merges the seed
// records into the row's candidates.
// ---------------------------------------------------------------------------
constexpr int kSeedThreads = 256;
constexpr int kSeedList = 64;  // listed top ids a warp scores at once (two a lane)

// Queues the copy of id v's logit into *xw: the 4-byte word that holds it
// (a bf16 pair, or the fp32 value).  The pair's other element lies in the row
// unless v is the row's last element with an even index; that one is loaded
// directly.
template <typename In>
__device__ __forceinline__ void seed_fetch(const char *row, uint32_t v, uint32_t V, uint32_t *xw)
{
    if (sizeof(In) == 4) {
        cp_async4(xw, row + (size_t)v * 4);
    } else if ((v | 1u) < V) {
        cp_async4(xw, row + (size_t)(v & ~1u) * 2);
    } else {
        *xw = (uint32_t)__ldg((const unsigned short *)row + v) << ((v & 1u) * 16);
    }
}

template <typename In>
__device__ __forceinline__ float seed_logit(uint32_t w, uint32_t v)
{
    if (sizeof(In) == 4)
        return __uint_as_float(w);
    return __uint_as_float((v & 1u) ? (w & 0xFFFF0000u) : (w << 16));
}

// One id of the list (fine bits m): screened against the lane's threshold
// with the top-id upper bounds, else scored.
__device__ __forceinline__ void seed_one(uint32_t v, float x, uint64_t m, const RowMode &rm,
                                         const float *gtop, Cand2 &c, float &thr, float &thrS)
{
    if (!(fmaf(x, rm.invT, gtop[(int)(m >> 44)]) > thrS))
        return;  // cannot reach the threshold
    const float2 iv = logit_interval_m(x, rm.invT, m, true);
    c.add(iv.x, iv.y, (int)v);
    const float t = __fsub_rd(iv.x, 1e-9f);
    if (t > thr) {
        thr = t;
        thrS = level1_thr(t);
    }
}

__device__ __forceinline__ void seed_raise(float t, float &thr, float &thrS)
{
    if (t > thr) {
        thr = t;
        thrS = level1_thr(t);
    }
}

template <typename In>
__device__ __forceinline__ void seed_score(const uint32_t *ids, const uint32_t *xw, int n,
                                           const RowMode &rm, const float *gtop, Cand2 &c,
                                           float &thr, float &thrS)
{
    const int lane = threadIdx.x & 31;
    const bool h0 = lane < n, h1 = lane + 32 < n;
    float x0 = 0.f, x1 = 0.f, lo = -INFINITY;
    uint64_t m0 = 0, m1 = 0;
    if (h0) {
        x0 = seed_logit<In>(xw[lane], ids[lane]);
        m0 = fine52(rm.key, ids[lane]);
        lo = logit_lower_bound(x0, rm.invT, gtop[kGTab + (int)(m0 >> 44)]);
    }
    if (h1) {
        x1 = seed_logit<In>(xw[lane + 32], ids[lane + 32]);
        m1 = fine52(rm.key, ids[lane + 32]);
        lo = fmaxf(lo, logit_lower_bound(x1, rm.invT, gtop[kGTab + (int)(m1 >> 44)]));
    }
    // the batch's best lower bound: the id it belongs to still passes the
    // screen below and is scored, so the threshold stays below a candidate
    seed_raise(__fsub_rd(warp_max(lo), 1e-9f), thr, thrS);
    if (h0)
        seed_one(ids[lane], x0, m0, rm, gtop, c, thr, thrS);
    if (h1)
        seed_one(ids[lane + 32], x1, m1, rm, gtop, c, thr, thrS);
    // every lane leaves with the warp's best threshold
    seed_raise(warp_max(thr), thr, thrS);
}

template <typename In>
__global__ void __launch_bounds__(kSeedThreads) seed_kernel(const __grid_constant__ Job j)
{
    __shared__ uint64_t skip[kSkipN];
    __shared__ float gtop[2 * kGTab];
    __shared__ uint32_t idl[kSeedThreads / 32][kSeedList];
    __shared__ uint32_t xwl[kSeedThreads / 32][kSeedList];
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i < kSkipN; i += blockDim.x)
        skip[i] = __ldg(j.skip + i);
    for (int i = threadIdx.x; i < 2 * kGTab; i += blockDim.x)
        gtop[i] = __ldg(j.gtop + i);
    __syncthreads();
    const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
    const unsigned lt = (1u << lane) - 1u;
    constexpr int kWarps = kSeedThreads / 32;
    const int H = gumbel_rows(j);
    const uint32_t nblk = ((uint32_t)j.V + 255u) >> 8;
    const long long span = j.seed_span;
    const long long total = (long long)j.B * H * nblk;
    const long long w0 = ((long long)blockIdx.x * kWarps + wl) * span;
    const long long wend = min(w0 + span, total);
    uint32_t *ids = idl[wl];
    uint32_t *xw = xwl[wl];
    // pieces of the span, one row each (warp-uniform)
    for (long long s = w0; s < wend;) {
        const long long grow = s / nblk;
        const long long rstart = grow * nblk;
        const uint32_t b0 = (uint32_t)(s - rstart);
        const uint32_t bend = (uint32_t)min((long long)nblk, wend - rstart);
        // record number: span boundaries inside the row up to the piece
        const int rec = b0 == 0u ? 0 : (int)(s / span - rstart / span);
        const int b = (int)(grow / H), k = (int)(grow % H);
        const int n = clamp_len(j, b);
        const int slot = gumbel_slot(j, k);
        bool valid = true;
        int np = 0;
        if (j.kind == K_SPOT)
            valid = ((__ldg(j.smask + (int64_t)b * (j.N + 1) + slot / j.L) >> (slot % j.L)) &
                     1ull) != 0;
        if (j.kind == K_TREE)
            np = __ldg(j.node_pos + (int64_t)b * j.N + slot);
        SeedRec r;
        r.thr = r.hi1 = r.lo1 = r.hi2 = r.lo2 = r.hi3 = -INFINITY;
        r.v1 = r.v2 = -1;
        if (valid) {  // warp-uniform
            const RowMode rm = row_mode(j, b, slot, n, pos0_of(j, b), np);
            const char *row = slot_row(j, b, slot);
            Cand2 c;
            c.init();
            float thr = -INFINITY, thrS = -INFINITY;
            uint32_t nextb = b0 + 32u;  // next block to hand out (warp-uniform)
            uint32_t beta = b0 + (uint32_t)lane;
            bool act = beta < bend;
            int pos = -1, i = 0, cnt = 0;
            // Each draw moves its lane's offset up by at least one, so a block
            // ends within 257 draws and the loop within 257 * span trips.
            while (__any_sync(0xFFFFFFFFu, act)) {
                bool got = false, done = false;
                uint32_t v = 0u;
                if (act) {
                    pos = next_top(rm.key, beta, i++, pos, skip);
                    v = beta * 256u + (uint32_t)pos;
                    got = pos <= 255 && v < (uint32_t)j.V;
                    done = !got;
                }
                const unsigned gm = __ballot_sync(0xFFFFFFFFu, got);
                if (got) {
                    const int q = cnt + __popc(gm & lt);
                    ids[q] = v;
                    seed_fetch<In>(row, v, (uint32_t)j.V, &xw[q]);
                }
                cnt += __popc(gm);
                const unsigned dm = __ballot_sync(0xFFFFFFFFu, done);
                if (done) {
                    beta = nextb + (uint32_t)__popc(dm & lt);
                    act = beta < bend;
                    pos = -1;
                    i = 0;
                }
                nextb += (uint32_t)__popc(dm);
                if (cnt > kSeedList - 32) {  // room for one more trip's ids
                    cp_async_wait_all();
                    __syncwarp();
                    seed_score<In>(ids, xw, cnt, rm, gtop, c, thr, thrS);
                    __syncwarp();
                    cnt = 0;
                }
            }
            cp_async_wait_all();
            __syncwarp();
            if (cnt > 0)
                seed_score<In>(ids, xw, cnt, rm, gtop, c, thr, thrS);
            __syncwarp();
            warp_cand2(c);
            r.thr = warp_max(thr);
            r.hi1 = c.hi1;
            r.lo1 = c.lo1;
            r.hi2 = c.hi2;
            r.lo2 = c.lo2;
            r.hi3 = c.hi3;
            r.v1 = c.v1;
            r.v2 = c.v2;
        }
        SeedRec *rr = j.seeds + grow * j.seed_chunks;
        if (lane == 0)
            rr[rec] = r;
        if (bend == nblk) {
            // the row ends in this span: its later records stay empty
            SeedRec e;
            e.thr = e.hi1 = e.lo1 = e.hi2 = e.lo2 = e.hi3 = -INFINITY;
            e.v1 = e.v2 = -1;
            for (int q = rec + 1 + lane; q < j.seed_chunks; q += 32)
                rr[q] = e;
        }
        s = rstart + bend;
    }
}

// Resident seed CTAs per SM (the smaller of the two instances).
cudaError_t seed_setup(int *blocks_per_sm)
{
    int a = 0, b = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, seed_kernel<uint16_t>,
                                                                  kSeedThreads, 0);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, seed_kernel<float>, kSeedThreads, 0);
    *blocks_per_sm = a < b ? a : b;
    return e;
}

cudaError_t seed_launch(const Job &j, int grid, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    pdl_config(cfg, at, dim3(grid), dim3(kSeedThreads), 0, s);
    return j.dtype == SV_BF16 ? cudaLaunchKernelEx(&cfg, seed_kernel<uint16_t>, j)
                              : cudaLaunchKernelEx(&cfg, seed_kernel<float>, j);
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
