// sv_pass.cu -- the streaming kernel of libsv.
//
// One persistent CTA per SM streams logit rows from HBM exactly once.  A
// producer warp takes work units (a contiguous part of one row) from a global
// counter and moves them into an 8-stage shared-memory ring with bulk copies
// (cp.async.bulk, completion on an mbarrier); eight consumer warps compute
// the row statistics the verify rules need:
//   - max / lowest-index argmax                 (greedy rules, [PackedSS] eq. 1)
//   - sum 2^((x - m) c) for log-sum-exp at T    (p, q of [PackedSS] §2.2, [SPOT] eq. 2)
//   - Gumbel-max with exact fp64 candidates     ([SPOT] eq. 4, eqs. 5-7)
// The CTA that completes the last unit of a sequence runs that sequence's
// decision step (prefix scan, stopping index, tree path) in one warp.
#include <math.h>

#include "sv_common.cuh"

namespace sv {

struct StageMeta {
    int unit;   // -1: end of work
    int nv;     // 16-byte vectors in this stage
    int vbase;  // row vector index of the stage's first vector
    int first;  // first stage of its unit
    int last;   // last stage of its unit
    int pad[3];
};

struct PassShared {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    StageMeta meta[kStages];
    uint32_t thr[2];
    float rf[kConsumerWarps][4];
    int ri[kConsumerWarps][2];
    float rg[kConsumerWarps][5];
    int rgi[kConsumerWarps][2];
    volatile int abort;
};

struct RowMode {
    int mode;
    float c1, c2, invT;
    double T;
    uint64_t key;
};

__device__ RowMode row_mode(const Job &j, int b, int slot)
{
    RowMode r;
    r.mode = 0;
    r.c1 = r.c2 = r.invT = 0.f;
    r.T = 1.0;
    r.key = 0;
    int64_t p0 = pos0_of(j, b);
    switch (j.kind) {
    case K_GREEDY:
        r.mode = M_ARGMAX;
        break;
    case K_SAMPLE: {
        int n = clamp_len(j, b);
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
    }
    case K_TREE:
        if (j.Tp == 0.f) {
            r.mode = M_ARGMAX;
        } else {
            r.mode = M_GUMBEL;
            r.invT = j.invTp;
            r.T = j.Tp;
            int np = __ldg(j.node_pos + (int64_t)b * j.N + slot);
            r.key = rng_key(j.seed, kTree, (uint64_t)b, p0 + np, 0);
        }
        break;
    default: {  // Packed-SS
        int n = clamp_len(j, b);
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
            int jj = slot - j.K;
            if (j.Tp == 0.f) {
                r.mode = M_ARGMAX | M_LSE;  // confidence needs the T = 1 normaliser
                r.c1 = j.c1;
            } else {
                r.mode = M_GUMBEL | M_LSE;
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
    }
    return r;
}

// Per-thread running state of one unit.
struct TState {
    float mx, mn;
    int amax;
    float mref;      // reference logit of the sums (a logit this thread has seen)
    float mc1, mc2;  // fl(mref * c1), fl(mref * c2)
    float acc1, acc2;
    Cand2 c;         // Gumbel candidates
    float lomax;     // best lower end seen
    float thr, thrS; // level-2 and level-1 thresholds
    float pub;       // threshold last published to the CTA
    int seedv;
};

__device__ __forceinline__ void tstate_init(TState &s)
{
    s.mx = -INFINITY;
    s.mn = INFINITY;
    s.amax = 0x7FFFFFFF;
    s.mref = -INFINITY;
    s.mc1 = s.mc2 = 0.f;
    s.acc1 = s.acc2 = 0.f;
    s.c.init();
    s.lomax = -INFINITY;
    s.thr = s.thrS = s.pub = -INFINITY;
    s.seedv = -1;
}

__device__ __forceinline__ void raise_thr(TState &s, float t)
{
    if (t > s.thr) {
        s.thr = t;
        s.thrS = level1_thr(t);
    }
}

// Level 2: fp32 interval of x/T + G; candidates whose upper end reaches the
// threshold are kept, and the best lower end raises the threshold (anything
// below it - 1e-9 can neither win nor tie within 1e-9).
__device__ __forceinline__ void gumbel_level2(float x, uint32_t v, uint32_t b0, TState &s,
                                              const RowMode &rm)
{
    const float2 iv = logit_interval_at(x, rm.invT, rm.key, v, b0);
    const float lo = iv.x, hi = iv.y;
    if (hi < s.thr)
        return;
    s.c.add(lo, hi, (int)v);
    if (lo > s.lomax) {
        s.lomax = lo;
        raise_thr(s, __fsub_rd(lo, 1e-9f));
    }
}

template <typename In, int MODE>
__device__ __forceinline__ void do_chunk(const uint4 *__restrict__ st, int nv, int vbase, TState &s,
                                         const RowMode &rm, const float *__restrict__ gt)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    const int t = threadIdx.x;
    uint4 q[kVecsPerThread];
    bool ok[kVecsPerThread];
#pragma unroll
    for (int k = 0; k < kVecsPerThread; ++k) {
        int idx = t + k * kConsumers;
        ok[k] = idx < nv;
        q[k] = ok[k] ? st[idx] : make_uint4(0, 0, 0, 0);
    }
    if (MODE & (M_ARGMAX | M_LSE)) {
        // chunk max / min on packed values (bf16x2 or fp32), as a short tree
        uint32_t pm = VT::kNegInf, pn = VT::kPosInf;
#pragma unroll
        for (int k = 0; k < kVecsPerThread; ++k)
            if (ok[k]) {
                pm = VT::bmax(pm, VT::pmax(q[k]));
                if (MODE & M_LSE)
                    pn = VT::bmin(pn, VT::pmin(q[k]));
            }
        const float cm = VT::hi_of(pm);
        if ((MODE & M_ARGMAX) && cm > s.mx) {
            bool found = false;
#pragma unroll
            for (int k = 0; k < kVecsPerThread; ++k) {
                float f[E];
                VT::unpack(q[k], f);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    if (!found && ok[k] && f[e] == cm) {
                        found = true;
                        s.amax = (vbase + t + k * kConsumers) * E + e;
                    }
            }
        }
        s.mx = fmaxf(s.mx, cm);
        if ((MODE & M_LSE) && cm > -INFINITY) {
            s.mn = fminf(s.mn, VT::lo_of(pn));
            if (s.mref == -INFINITY) {
                s.mref = cm;
                s.mc1 = __fmul_rn(cm, rm.c1);
                if (MODE & M_LSE2)
                    s.mc2 = __fmul_rn(cm, rm.c2);
            } else {
                float cmax = (MODE & M_LSE2) ? fmaxf(rm.c1, rm.c2) : rm.c1;
                if ((cm - s.mref) * cmax > 64.f) {  // keep every term below 2^64
                    float n1 = __fmul_rn(cm, rm.c1);
                    s.acc1 *= ex2f(s.mc1 - n1);
                    s.mc1 = n1;
                    if (MODE & M_LSE2) {
                        float n2 = __fmul_rn(cm, rm.c2);
                        s.acc2 *= ex2f(s.mc2 - n2);
                        s.mc2 = n2;
                    }
                    s.mref = cm;
                }
            }
            // one FFMA and one ex2 per term; stage partials summed as a tree
            float part1[kVecsPerThread], part2[kVecsPerThread];
#pragma unroll
            for (int k = 0; k < kVecsPerThread; ++k) {
                part1[k] = 0.f;
                part2[k] = 0.f;
                if (ok[k]) {
                    float f[E], e1[E];
                    VT::unpack(q[k], f);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        e1[e] = ex2f(fmaf(f[e], rm.c1, -s.mc1));
#pragma unroll
                    for (int w = E / 2; w >= 1; w >>= 1)
#pragma unroll
                        for (int e = 0; e < w; ++e)
                            e1[e] += e1[e + w];
                    part1[k] = e1[0];
                    if (MODE & M_LSE2) {
                        float e2[E];
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            e2[e] = ex2f(fmaf(f[e], rm.c2, -s.mc2));
#pragma unroll
                        for (int w = E / 2; w >= 1; w >>= 1)
#pragma unroll
                            for (int e = 0; e < w; ++e)
                                e2[e] += e2[e + w];
                        part2[k] = e2[0];
                    }
                }
            }
#pragma unroll
            for (int w = kVecsPerThread / 2; w >= 1; w >>= 1)
#pragma unroll
                for (int k = 0; k < w; ++k) {
                    part1[k] += part1[k + w];
                    part2[k] += part2[k + w];
                }
            s.acc1 += part1[0];
            if (MODE & M_LSE2)
                s.acc2 += part2[0];
        }
    }
    if (MODE & M_GUMBEL) {
        // level 1 on groups of 4 ids: one hash word; skip the group unless a
        // byte is 0xFF (unbounded bucket) or its largest logit can reach the
        // threshold with the largest finite bucket bound.
        const uint32_t klo = (uint32_t)rm.key;
        const float gmax = g8max(gt);
#pragma unroll
        for (int k = 0; k < kVecsPerThread; ++k)
            if (ok[k]) {
                const uint32_t v0 = (uint32_t)(vbase + t + k * kConsumers) * E;
#pragma unroll
                for (int g = 0; g < E / 4; ++g) {
                    const uint32_t wa = word_a(klo, (v0 >> 2) + g);
                    const bool top = ((~wa - 0x01010101u) & wa & 0x80808080u) != 0u;
                    const float gx = VT::group_max(q[k], g);
                    if (top || fmaf(gx, rm.invT, gmax) >= s.thrS) {
                        // rare: per-id screen, deliberately not unrolled
#pragma unroll 1
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t v = v0 + 4 * g + e;
                            const uint32_t b0 = (wa >> (8 * e)) & 0xFFu;
                            const float x = VT::elem(q[k], 4 * g + e);
                            if ((int)v != s.seedv &&
                                fmaf(x, rm.invT, gup_of(gt, rm.key, v, b0)) >= s.thrS)
                                gumbel_level2(x, v, b0, s, rm);
                        }
                    }
                }
            }
    }
}

// First stage of a Gumbel unit: each warp scores in fp32 the element with the
// largest table bound it holds, and the CTA starts from the best lower end of
// these (a rigorous lower bound of the unit's maximum).
template <typename In>
__device__ __forceinline__ void gumbel_seed(const uint4 *__restrict__ st, int nv, int vbase,
                                            TState &s, const RowMode &rm,
                                            const float *__restrict__ gt, PassShared &sm,
                                            int slot)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    const int t = threadIdx.x;
    const uint32_t klo = (uint32_t)rm.key;
    float bub = -INFINITY, bx = 0.f;
    int bv = -1;
    uint32_t bb0 = 0;
#pragma unroll 1
    for (int k = 0; k < kVecsPerThread; ++k) {
        int idx = t + k * kConsumers;
        if (idx < nv) {
            const uint4 q = st[idx];
            uint32_t v0 = (uint32_t)(vbase + idx) * E;
#pragma unroll 1
            for (int i = 0; i < E; ++i) {
                uint32_t v = v0 + i;
                uint32_t b0 = (word_a(klo, v >> 2) >> (8 * (i & 3))) & 0xFFu;
                float x = VT::elem(q, i);
                float ub = fmaf(x, rm.invT, gup_of(gt, rm.key, v, b0));
                if (ub > bub) {
                    bub = ub;
                    bv = (int)v;
                    bx = x;
                    bb0 = b0;
                }
            }
        }
    }
    float wv = bub;
    int wi = bv;
    warp_argmax(wv, wi);
    if (bv >= 0 && bv == wi) {
        s.seedv = bv;
        const float2 iv = logit_interval_at(bx, rm.invT, rm.key, (uint32_t)bv, bb0);
        const float lo = iv.x, hi = iv.y;
        s.c.add(lo, hi, bv);
        s.lomax = lo;
        raise_thr(s, __fsub_rd(lo, 1e-9f));
        atomicMax(&sm.thr[slot], f2ord(s.thr));
    }
    named_sync(1, kConsumers);
    raise_thr(s, ord2f(*(volatile uint32_t *)&sm.thr[slot]));
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

__device__ void fin_greedy(const Job &j, int b)
{
    const int lane = threadIdx.x & 31;
    int n = clamp_len(j, b);
    if (lane == 0) check_len(j, b);
    bool match = false;
    if (lane < n) {
        RowM r = merge_row(j, b, lane, 0.f, 0.f);
        int d = __ldg(j.ids + (int64_t)b * j.K + lane);
        match = (d == r.amax);
    }
    unsigned mm = __ballot_sync(0xFFFFFFFFu, match);
    int h = (~mm == 0u) ? 32 : __ffs(~mm) - 1;
    h = min(h, n);
    if (lane == 0) {
        RowM r = merge_row(j, b, h, 0.f, 0.f);
        j.acc[b] = h;
        j.next[b] = r.amax;
    }
}

__device__ void fin_sample(const Job &j, int b)
{
    const int lane = threadIdx.x & 31;
    int n = clamp_len(j, b);
    if (lane == 0) check_len(j, b);
    const int64_t p0 = pos0_of(j, b);
    bool acc = false, und = false;
    double Lp = 0, Lq = 0, ep = 0, eq = 0;
    if (lane < n) {
        RowM rp = merge_row(j, b, lane, j.cp, 0.f);
        RowM rq = merge_row(j, b, j.K + 1 + lane, j.cq, 0.f);
        Lp = kLn2 * rp.L2b1;
        Lq = kLn2 * rq.L2b1;
        ep = row_eps(rp, j.cp);
        eq = row_eps(rq, j.cq);
        int d = __ldg(j.ids + (int64_t)b * j.K + lane);
        double lp = -INFINITY, lq = 0.0;
        if (d < 0 || d >= j.V) {
            latch(j.err, SV_ERR_DEVICE_BOUNDS);
        } else {
            float xd = load_logit(j, row_ptr(j, b, lane), d);
            float yd = load_logit(j, row_ptr(j, b, j.K + 1 + lane), d);
            lp = (double)xd / (double)j.Tp - Lp;
            lq = (double)yd / (double)j.Tq - Lq;
        }
        double r = exp(lp - lq);
        double rel = 1.01 * (ep + eq) + 1e-15;
        double alo = alpha_of(j.amode, r * (1.0 - rel), j.lam);
        double ahi = alpha_of(j.amode, r * (1.0 + rel), j.lam);
        double u = uniform_at(rng_key(j.seed, kAccept, (uint64_t)b, p0 + lane, 0), 0);
        acc = u < alo - kFlagEps;
        bool rej = u >= ahi + kFlagEps;
        und = !(acc || rej) || j.force_rescue;
        if (j.force_rescue)
            acc = false;
        if (j.p_at) j.p_at[(int64_t)b * j.K + lane] = (float)exp(lp);
        if (j.q_at) j.q_at[(int64_t)b * j.K + lane] = (float)exp(lq);
        if (j.lse_p) j.lse_p[(int64_t)b * (j.K + 1) + lane] = (float)Lp;
        if (j.lse_q) j.lse_q[(int64_t)b * j.K + lane] = (float)Lq;
        RowStat *sp = j.rs_stat + (int64_t)b * j.rows_per_seq + lane;
        sp->L1 = Lp;
        sp->L2 = rp.L2b1;
        sp->m = rp.m;
        sp->eps = (float)ep;
        RowStat *sq = j.rs_stat + (int64_t)b * j.rows_per_seq + j.K + 1 + lane;
        sq->L1 = Lq;
        sq->L2 = rq.L2b1;
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
    // bonus row (always valid): its Gumbel-max with key (SAMPLE, pos + n)
    RowM rb = merge_row(j, b, n, j.cp, 0.f);
    const char *rown = row_ptr(j, b, n);
    GRes gb = resolve_lanes(j, rown, rng_key(j.seed, kSample, (uint64_t)b, p0 + n, 0),
                            (double)j.Tp, j.invTp, rb.gc, lane == 0);
    if (lane == 0) {
        double Lb = kLn2 * rb.L2b1;
        if (j.lse_p) j.lse_p[(int64_t)b * (j.K + 1) + n] = (float)Lb;
        RowStat *sb = j.rs_stat + (int64_t)b * j.rows_per_seq + n;
        sb->L1 = Lb;
        sb->m = rb.m;
        sb->gidx = gb.v;
        sb->gflag = gb.flag;
        if (rescue) {
            unsigned e = atomicAdd(j.ctl + C_RESCUE_N, 1u);
            j.rescue[e].b = b;
            j.rescue[e].kind = 0;
            j.rescue[e].h = 0;
        } else if (f == n) {
            j.acc[b] = n;
            j.next[b] = gb.v;
            if (j.flags) j.flags[b] = gb.flag;
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
            j.resid[e] = re;
        }
    }
}

__device__ void fin_tree(const Job &j, int b)
{
    const int lane = threadIdx.x & 31;
    const int64_t p0 = pos0_of(j, b);
    unsigned mlo = 0, mhi = 0;
    int nflag = 0;
    for (int half = 0; half < 2; ++half) {
        int n = lane + 32 * half;
        bool has = n < j.N;
        RowM r = merge_row(j, b, has ? n : 0, 0.f, 0.f);
        int win;
        if (j.Tp == 0.f) {
            win = r.amax;
        } else {
            int np = has ? __ldg(j.node_pos + (int64_t)b * j.N + n) : 0;
            GRes g = resolve_lanes(j, row_ptr(j, b, has ? n : 0),
                                   rng_key(j.seed, kTree, (uint64_t)b, p0 + np, 0),
                                   (double)j.Tp, j.invTp, r.gc, has);
            win = g.v;
            if (has)
                nflag += g.flag;
        }
        bool m = has && (win == __ldg(j.node_tok + (int64_t)b * j.N + n));
        if (has && j.match) j.match[(int64_t)b * j.N + n] = m ? 1 : 0;
        unsigned bal = __ballot_sync(0xFFFFFFFFu, m);
        if (half == 0) mlo = bal; else mhi = bal;
    }
    for (int o = 16; o; o >>= 1)
        nflag += __shfl_xor_sync(0xFFFFFFFFu, nflag, o);
    if (lane == 0) {
        uint64_t ok = 0;
        uint8_t depth[kMaxN];
        int best = -1, bestd = 0;
        for (int n = 0; n < j.N; ++n) {
            int par = __ldg(j.parent + (int64_t)b * j.N + n);
            int np = __ldg(j.node_pos + (int64_t)b * j.N + n);
            if (par < -1 || par >= n || np < 0) {
                latch(j.err, SV_ERR_DEVICE_BOUNDS);
                depth[n] = 0;
                continue;
            }
            bool m = (n < 32) ? ((mlo >> n) & 1u) : ((mhi >> (n - 32)) & 1u);
            bool okn = m && (par < 0 || ((ok >> par) & 1ull));
            depth[n] = (uint8_t)(par < 0 ? 1 : depth[par] + 1);
            if (okn) {
                ok |= 1ull << n;
                if (depth[n] > bestd) {
                    bestd = depth[n];
                    best = n;
                }
            }
        }
        j.path_len[b] = bestd;
        j.commit_count[b] = bestd + 1;
        for (int k = 0; k < j.max_depth; ++k)
            j.path_nodes[(int64_t)b * j.max_depth + k] = -1;
        for (int n = best, d = bestd; n >= 0; n = __ldg(j.parent + (int64_t)b * j.N + n), --d)
            if (d - 1 < j.max_depth)
                j.path_nodes[(int64_t)b * j.max_depth + d - 1] = n;
        if (j.flags) j.flags[b] = nflag;
    }
}

__device__ void fin_packed(const Job &j, int b)
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
        RowM r = merge_row(j, b, slot, greedy ? j.c1 : j.cp, j.c1);
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
            conf = exp2((double)__fmul_rn(r.m, j.c1) - r.L2b1);
        } else {
            t.z = g.v;
            t.gflag = g.flag;
            double LT = kLn2 * r.L2b1;
            float yz = load_logit(j, row_ptr(j, b, slot), t.z);
            t.q = (float)exp((double)yz / (double)j.Tp - LT);
            conf = (j.Tp == 1.f) ? exp2((double)__fmul_rn(r.m, j.cp) - r.L2b1)
                                 : exp2((double)__fmul_rn(r.m, j.c1) - r.L2b2);
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
            RowM r = merge_row(j, b, lane, 0.f, 0.f);
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
        RowM rp = merge_row(j, b, lane, j.cp, 0.f);
        Lp = kLn2 * rp.L2b1;
        ep = row_eps(rp, j.cp);
        int d = __ldg(j.ids + (int64_t)b * Km1 + lane);
        double lp = -INFINITY;
        if (d < 0 || d >= j.V)
            latch(j.err, SV_ERR_DEVICE_BOUNDS);
        else
            lp = (double)load_logit(j, row_ptr(j, b, lane), d) / (double)j.Tp - Lp;
        double lq = log((double)__ldg(j.prev_q + (int64_t)b * Km1 + lane));
        double r = exp(lp - lq);
        double rel = 1.01 * ep + 1e-15;
        double alo = fmin(1.0, r * (1.0 - rel)), ahi = fmin(1.0, r * (1.0 + rel));
        double u = uniform_at(rng_key(j.seed, kAccept, (uint64_t)b, p0 + lane, 0), 0);
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
        RowM rb = merge_row(j, b, n, j.cp, 0.f);
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
        j.resid[e] = re;
    }
}

// ---------------------------------------------------------------------------
// The streaming kernel.
// ---------------------------------------------------------------------------
template <typename In, int MODE>
__device__ __forceinline__ void run_chunk(const uint4 *st, const StageMeta &mt, TState &s,
                                          const RowMode &rm, const float *gt, PassShared &sm,
                                          int tslot)
{
    if ((MODE & M_GUMBEL) && mt.first)
        gumbel_seed<In>(st, mt.nv, mt.vbase, s, rm, gt, sm, tslot);
    do_chunk<In, MODE>(st, mt.nv, mt.vbase, s, rm, gt);
}

template <typename In>
__device__ __forceinline__ void dispatch_chunk(const uint4 *st, const StageMeta &mt, TState &s,
                                               const RowMode &rm, const float *gt,
                                               PassShared &sm, int tslot)
{
    switch (rm.mode) {
    case M_ARGMAX: run_chunk<In, M_ARGMAX>(st, mt, s, rm, gt, sm, tslot); break;
    case M_LSE: run_chunk<In, M_LSE>(st, mt, s, rm, gt, sm, tslot); break;
    case M_LSE | M_GUMBEL: run_chunk<In, M_LSE | M_GUMBEL>(st, mt, s, rm, gt, sm, tslot); break;
    case M_GUMBEL: run_chunk<In, M_GUMBEL>(st, mt, s, rm, gt, sm, tslot); break;
    case M_ARGMAX | M_LSE: run_chunk<In, M_ARGMAX | M_LSE>(st, mt, s, rm, gt, sm, tslot); break;
    case M_GUMBEL | M_LSE | M_LSE2:
        run_chunk<In, M_GUMBEL | M_LSE | M_LSE2>(st, mt, s, rm, gt, sm, tslot);
        break;
    default: break;
    }
}

// End of a unit: reduce the consumers' state into one RowPart record, and run
// the decision step of the sequence if this was its last unit.
__device__ void finish_unit(const Job &j, int unit, TState &s, const RowMode &rm,
                            PassShared &sm, int tslot)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const bool gum = (rm.mode & M_GUMBEL) != 0;
    float mx = s.mx;
    int am = s.amax;
    warp_argmax(mx, am);
    float mn = warp_min(s.mn);
    Cand2 g = s.c;
    if (gum)
        warp_cand2(g);
    if (lane == 0) {
        sm.rf[w][0] = mx;
        sm.rf[w][1] = mn;
        sm.ri[w][0] = am;
        sm.rg[w][0] = g.hi1;
        sm.rg[w][1] = g.lo1;
        sm.rg[w][2] = g.hi2;
        sm.rg[w][3] = g.lo2;
        sm.rg[w][4] = g.hi3;
        sm.rgi[w][0] = g.v1;
        sm.rgi[w][1] = g.v2;
    }
    named_sync(1, kConsumers);
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < kConsumerWarps; ++q)
        M = fmaxf(M, sm.rf[q][0]);
    float t1 = 0.f, t2 = 0.f;
    if ((rm.mode & M_LSE) && s.mref > -INFINITY) {
        // terms were 2^(x c - mc); the unit record is relative to fl(M c)
        t1 = s.acc1 * ex2f(s.mc1 - __fmul_rn(M, rm.c1));
        if (rm.mode & M_LSE2)
            t2 = s.acc2 * ex2f(s.mc2 - __fmul_rn(M, rm.c2));
    }
    float w1 = warp_sum(t1), w2 = warp_sum(t2);
    float wmn = 0.f, wmx = 0.f;
    int wam = 0;
    Cand2 wg;
    wg.init();
    if (t == 0) {
        wmx = -INFINITY;
        wmn = INFINITY;
        wam = 0x7FFFFFFF;
        for (int q = 0; q < kConsumerWarps; ++q) {
            float v = sm.rf[q][0];
            int i = sm.ri[q][0];
            if (v > wmx || (v == wmx && (unsigned)i < (unsigned)wam)) {
                wmx = v;
                wam = i;
            }
            wmn = fminf(wmn, sm.rf[q][1]);
            if (gum) {
                Cand2 o;
                o.hi1 = sm.rg[q][0];
                o.lo1 = sm.rg[q][1];
                o.hi2 = sm.rg[q][2];
                o.lo2 = sm.rg[q][3];
                o.hi3 = sm.rg[q][4];
                o.v1 = sm.rgi[q][0];
                o.v2 = sm.rgi[q][1];
                wg.merge(o);
            }
        }
        sm.thr[tslot ^ 1] = f2ord(-INFINITY);  // next unit's threshold slot
    }
    if (lane == 0) {
        sm.rf[w][2] = w1;
        sm.rf[w][3] = w2;
    }
    named_sync(1, kConsumers);
    if (w == 0) {
        int last = 0, b = 0;
        if (lane == 0) {
            float S1 = 0.f, S2 = 0.f;
            for (int q = 0; q < kConsumerWarps; ++q) {
                S1 += sm.rf[q][2];
                S2 += sm.rf[q][3];
            }
            RowPart r;
            r.m = wmx;
            r.mn = wmn;
            r.s1 = S1;
            r.s2 = S2;
            r.amax = wam;
            r.ghi1 = wg.hi1;
            r.glo1 = wg.lo1;
            r.ghi2 = wg.hi2;
            r.glo2 = wg.lo2;
            r.ghi3 = wg.hi3;
            r.gv1 = wg.v1;
            r.gv2 = wg.v2;
            r.pad[0] = r.pad[1] = r.pad[2] = r.pad[3] = 0;
            j.rp[unit] = r;
            long long per_seq = (long long)j.rows_per_seq * j.parts;
            b = (int)(unit / per_seq);
            unsigned expect = (unsigned)(valid_slots(j, b) * j.parts);
            __threadfence();
            unsigned old = atomicAdd(j.seq_done + b, 1u);
            last = (old + 1u == expect);
            if (last)
                __threadfence();
        }
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        b = __shfl_sync(0xFFFFFFFFu, b, 0);
        if (last) {
            switch (j.kind) {
            case K_GREEDY: fin_greedy(j, b); break;
            case K_SAMPLE: fin_sample(j, b); break;
            case K_TREE: fin_tree(j, b); break;
            default: fin_packed(j, b); break;
            }
        }
    }
}

template <typename In>
__global__ void __launch_bounds__(kPassThreads, SV_MIN_BLOCKS) pass_kernel(const Job j)
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
        sm.thr[0] = f2ord(-INFINITY);
        sm.thr[1] = f2ord(-INFINITY);
        sm.abort = 0;
        mbar_fence_init();
    }
    for (int i = t; i < kGTab; i += blockDim.x)
        gt[i] = __ldg(j.gtab + i);
    __syncthreads();

    const long long per_seq = (long long)j.rows_per_seq * j.parts;
    if (t >= kConsumers) {
        // ---------------- producer warp ----------------
        if (t == kConsumers) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t pend = 0, pend_par = 0;  // stages with a copy not yet re-acquired
            bool ok = true;
            for (;;) {
                long long u = (long long)atomicAdd(j.ctl + C_UNIT, 1u);
                if (u >= j.total_units)
                    break;
                int b = (int)(u / per_seq);
                int rem = (int)(u - (long long)b * per_seq);
                int slot = rem / j.parts, part = rem - slot * j.parts;
                if (!slot_valid(j, b, slot))
                    continue;
                const char *row = slot_row(j, b, slot);
                int vs = part * j.part_vecs;
                int ve = min(j.nvec, vs + j.part_vecs);
                for (int v = vs; v < ve; v += kStageVecs) {
                    int nv = min(kStageVecs, ve - v);
                    if (!mbar_wait(&sm.empty[stage], phase ^ 1u)) {
                        ok = false;
                        break;
                    }
                    pend &= ~(1u << stage);  // the consumers released it: its copy landed
                    StageMeta &mt = sm.meta[stage];
                    mt.unit = (int)u;
                    mt.nv = nv;
                    mt.vbase = v;
                    mt.first = (v == vs);
                    mt.last = (v + kStageVecs >= ve);
                    mbar_arrive_tx(&sm.full[stage], (uint32_t)nv * 16u);
                    bulk_g2s(stages + (size_t)stage * kStageBytes, row + (int64_t)v * 16,
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
        int tslot = 0;
        TState s;
        RowMode rm;
        rm.mode = 0;
        tstate_init(s);
        for (;;) {
            if (!mbar_wait(&sm.full[stage], phase)) {
                latch(j.err, SV_ERR_TIMEOUT);
                break;
            }
            StageMeta mt = sm.meta[stage];
            if (mt.unit < 0 || sm.abort)
                break;
            if (mt.first) {
                int b = (int)(mt.unit / per_seq);
                int rem = (int)(mt.unit - (long long)b * per_seq);
                rm = row_mode(j, b, rem / j.parts);
                tstate_init(s);
            }
            if (rm.mode & M_GUMBEL)
                raise_thr(s, ord2f(*(volatile uint32_t *)&sm.thr[tslot]));
            const uint4 *st = reinterpret_cast<const uint4 *>(stages + (size_t)stage * kStageBytes);
            if (j.dtype == SV_BF16)
                dispatch_chunk<uint16_t>(st, mt, s, rm, gt, sm, tslot);
            else
                dispatch_chunk<float>(st, mt, s, rm, gt, sm, tslot);
            if ((rm.mode & M_GUMBEL) && s.thr > s.pub) {
                atomicMax(&sm.thr[tslot], f2ord(s.thr));
                s.pub = s.thr;
            }
            __syncwarp();
            if ((t & 31) == 0)
                mbar_arrive(&sm.empty[stage]);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
            if (mt.last) {
                finish_unit(j, mt.unit, s, rm, sm, tslot);
                tslot ^= 1;
            }
        }
    }
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

// Host-side launchers (the kernels are templates of this translation unit).
cudaError_t pass_setup(int *blocks_per_sm)
{
    const int smem = (int)pass_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(pass_kernel<uint16_t>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(pass_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, pass_kernel<uint16_t>,
                                                          kPassThreads, smem);
    return e;
}

cudaError_t pass_launch(const Job &j, int grid, cudaStream_t s)
{
    if (j.dtype == SV_BF16)
        pass_kernel<uint16_t><<<grid, kPassThreads, pass_smem_bytes(), s>>>(j);
    else
        pass_kernel<float><<<grid, kPassThreads, pass_smem_bytes(), s>>>(j);
    return cudaGetLastError();
}

}  // namespace sv
