// sv_resid.cuh -- the scores of the residual draw and their bounds.
//
// At the first rejection, the correction is the Gumbel-max of log w_v + G(v)
// with w = [p - q]_+ ([SPOT] App. B eq. 14; [PackedSS] Alg. 2 line 7).  With
// a = x/Tp, b = y/Tq and Delta = Lq - Lp,
//   log w_v = a_v - Lp + log(1 - exp(b_v - a_v - Delta))   (when b - a < Delta);
// dropping the common -Lp, every score is bracketed for Delta in [dlo, dhi]
// (the log-sum-exps carry the fp32 error bound of the streaming pass, or the
// fp64 rounding on the fp64 path).  The scan uses the three-level filter of
// sv_gumbel.cuh: the table bound ignores log(1 - .) <= 0, survivors get fp32
// intervals, and the two best candidates are certified or re-scored in fp64.
// A bonus draw (every draft accepted) is the same scan with the score
// a_v + G(v) alone (no q row; the common -Lp dropped).
#pragma once

#include "sv_common.cuh"

namespace sv {

__device__ __forceinline__ double log1mexp(double a)  // log(1 - e^a), a < 0
{
    return (a > -0.6931471805599453) ? log(-expm1(a)) : log1p(-exp(a));
}

struct RCtx {
    const char *prow, *qrow;
    double Tp, Tq, dlo, dhi;
    float invTp, invTq, dlo32, dhi32;  // [dlo32, dhi32] contains [dlo, dhi]
    uint64_t key;
    bool bonus;  // the bonus draw: score x/Tp + G, the q row unused
};

// fp64 interval of the residual score of id v (Delta bracket only); false
// when w_v = 0 for every Delta in the bracket.
__device__ __forceinline__ bool resid_interval64(const RCtx &c, float x, float y, uint64_t m,
                                                 bool top, double &lo, double &hi)
{
    double z = (double)x / c.Tp, w = (double)y / c.Tq;
    if (c.bonus) {
        lo = hi = z + gumbel64(m, top);
        return true;
    }
    double ah = w - z - c.dhi;
    if (!(ah < 0.0))
        return false;
    double al = w - z - c.dlo;
    double G = gumbel64(m, top);
    hi = z + log1mexp(ah) + G;
    lo = (al < 0.0) ? z + log1mexp(al) + G : -INFINITY;
    return true;
}

// log(1 - e^d), d < 0, in fp32 with a bound on its error: e = e^d carries
// the ex2 error and the rounding of d log2(e); t = 1 - e is then off by at
// most e (2^-21 + |d| 2^-22) + 2^-24 t, and lg2 adds 2^-22.
__device__ __forceinline__ float log1mexp32(float d, float &err)
{
    const float e = ex2f(d * 1.44269504088896f);
    const float t = 1.f - e;
    const float r = 0.69314718055995f * lg2a(t);
    // lg2.approx: error 2^-22 relative to max(1, |result|)
    err = (e * (0x1p-21f + fabsf(d) * 0x1p-22f)) / t + (1.f + fabsf(r)) * 0x1p-21f;
    return r;
}

// fp32 interval of the residual score; false when w_v = 0 for sure.
__device__ __forceinline__ bool resid_interval32(const RCtx &c, float x, float y, uint64_t m,
                                                 bool top, float &lo, float &hi)
{
    if (c.bonus) {
        const float2 iv = logit_interval_m(x, c.invTp, m, top);
        lo = iv.x;
        hi = iv.y;
        return true;
    }
    const float z = x * c.invTp, w = y * c.invTq;
    const float dz = w - z;
    const float edz = (fabsf(z) + fabsf(w)) * 0x1p-21f;
    const float dmin = (dz - c.dhi32) - edz - fabsf(dz - c.dhi32) * 0x1p-22f;  // smallest d
    const float dmax = (dz - c.dlo32) + edz + fabsf(dz - c.dlo32) * 0x1p-22f;  // largest d
    if (dmin >= 0.f)
        return false;
    const float g = gumbel32(m, top);
    float e1, lwh;
    const float lw1 = log1mexp32(dmin, e1);
    if (1.f - ex2f(dmin * 1.44269504088896f) > 0x1p-18f && e1 < 1.f)
        lwh = lw1 + e1;
    else {  // 1 - e^d <= -d
        lwh = 0.69314718055995f * lg2a(-dmin);
        lwh += (1.f + fabsf(lwh)) * 0x1p-20f;
    }
    float lwl = -INFINITY;
    if (dmax < 0.f && 1.f - ex2f(dmax * 1.44269504088896f) > 0x1p-18f) {
        float e2;
        const float lw2 = log1mexp32(dmax, e2);
        if (e2 < 1.f)
            lwl = lw2 - e2;
    }
    const float sh = z + lwh + g, sl = z + lwl + g;
    const float slack = (fabsf(z) + fabsf(sh)) * 0x1p-21f + kG32Err;
    hi = sh + slack;
    lo = sl - ((fabsf(z) + fabsf(sl)) * 0x1p-21f + kG32Err);
    return true;
}

// fp32 test that w_v = 0 for every Delta in the bracket.
__device__ __forceinline__ bool surely_zero(const RCtx &c, float x, float y)
{
    if (c.bonus)
        return false;
    float a = x * c.invTp, b = y * c.invTq;
    float d = (b - a) - c.dhi32;
    return d > (fabsf(a) + fabsf(b) + fabsf(c.dhi32) + 1.f) * 0x1p-20f;
}

struct Track32 {
    Cand2 c;
    float lomax, thr, thrS;
    __device__ __forceinline__ void init()
    {
        c.init();
        lomax = thr = thrS = -INFINITY;
    }
    __device__ __forceinline__ void raise(float t)
    {
        if (t > thr) {
            thr = t;
            thrS = level1_thr(t);
        }
    }
    __device__ __forceinline__ void add(const RCtx &ctx, float x, float y, uint32_t v, uint64_t m,
                                        bool top)
    {
        if (surely_zero(ctx, x, y)) return;
        float lo, hi;
        if (!resid_interval32(ctx, x, y, m, top, lo, hi) || hi < thr) return;
        c.add(lo, hi, (int)v);
        if (lo > lomax) {
            lomax = lo;
            raise(__fsub_rd(lo, 1e-9f));
        }
    }
};
// Per-id screen of one vector whose bound reached the threshold: top ids are
// skipped (the seed phase scored every top id of the scanned range); an ordinary id
// is bounded by the top byte of its fine bits.
template <typename In, typename Tr>
__device__ __forceinline__ void resid_vector(const RCtx &c, const uint4 &qx, const uint4 &qy,
                                             int k, const float *gt, const uint64_t *skip, Tr &tr)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    const uint32_t v0 = (uint32_t)k * E;
    const uint32_t tm = top_mask(c.key, v0 >> 8, (int)(v0 & 255u), E, skip);
#pragma unroll 1
    for (int i = 0; i < E; ++i) {
        if ((tm >> i) & 1u)
            continue;
        const uint32_t v = v0 + i;
        const float xi = VT::elem(qx, i);
        const uint64_t m = fine52(c.key, v);
        if (fmaf(xi, c.invTp, gt[(int)(m >> 44)]) < tr.thrS)
            continue;
        tr.add(c, xi, VT::elem(qy, i), v, m, false);
    }
}

__device__ __forceinline__ void fill_ctx(const Job &j, RCtx &ctx, const char *prow, const char *qrow,
                                         double D, double eD)
{
    ctx.prow = prow;
    ctx.qrow = qrow;
    ctx.Tp = j.Tp;
    ctx.Tq = (j.kind == K_PACKED) ? j.Tp : j.Tq;
    ctx.dlo = D - eD;
    ctx.dhi = D + eD;
    ctx.invTp = j.invTp;
    ctx.invTq = (float)(1.0 / ctx.Tq);
    ctx.dlo32 = __double2float_rd(ctx.dlo);
    ctx.dhi32 = __double2float_ru(ctx.dhi);
    ctx.bonus = false;
}

// Scores every top id of ids [lo, hi) of the pair into tr.  Thread tid of
// nthr takes blocks of 256 ids in turn, two at a time: it lists their top ids
// (a couple of skip draws per block), then loads all their logits, then
// scores them, so that the loads of a thread are in flight together.  Ids
// beyond the list of a crowded pair of blocks (rare) are scored one by one.
template <typename In, typename Tr>
__device__ __forceinline__ void seed_top_ids(const RCtx &c, uint32_t lo, uint32_t hi,
                                             const uint64_t *skip, int tid, int nthr, Tr &tr)
{
    using VT = VecTraits<In>;
    constexpr int kList = 12;
    if (hi <= lo)
        return;
    const uint32_t b1 = (hi - 1) >> 8;
    for (uint32_t beta = (lo >> 8) + (uint32_t)tid; beta <= b1; beta += 2u * (uint32_t)nthr) {
        uint32_t id[kList];
        int n = 0;
        for (int h = 0; h < 2; ++h) {
            const uint32_t bb = beta + (uint32_t)(h * nthr);
            if (bb > b1)
                break;
            int pos = -1;
            for (int i = 0; i < kSkipN; ++i) {
                pos = next_top(c.key, bb, i, pos, skip);
                const uint32_t v = bb * 256u + (uint32_t)pos;
                if (pos > 255 || v >= hi)
                    break;
                if (v < lo)
                    continue;
                if (n < kList)
                    id[n++] = v;
                else
                    tr.add(c, VT::load1(c.prow, (int)v), VT::load1(c.qrow, (int)v), v,
                           fine52(c.key, v), true);
            }
        }
        float x[kList], y[kList];
        for (int k = 0; k < n; ++k) {
            x[k] = VT::load1(c.prow, (int)id[k]);
            y[k] = VT::load1(c.qrow, (int)id[k]);
        }
        for (int k = 0; k < n; ++k)
            tr.add(c, x[k], y[k], id[k], fine52(c.key, id[k]), true);
    }
}

// Context of the residual draw of entry re.
// The weights [c p - q]_+ are those of [p - q]_+ with Lp lowered by log c,
// so the bracket of Delta = Lq - Lp widens by the bracket of log c.
__device__ __forceinline__ void resid_ctx(const Job &j, const ResidEntry &re, RCtx &ctx)
{
    const double D = re.Lq - re.Lp;
    const double eD = 1.001 * (re.epsp + re.epsq) + 1e-14 * (fabs(re.Lp) + fabs(re.Lq));
    fill_ctx(j, ctx, re.prow, re.qrow, D, eD);
    ctx.dlo += re.lclo;
    ctx.dhi += re.lchi;
    ctx.dlo32 = __double2float_rd(ctx.dlo);
    ctx.dhi32 = __double2float_ru(ctx.dhi);
    ctx.key = rng_key(j.seed, kSample, (uint64_t)re.b, pos0_of(j, re.b) + re.h, 0);
    ctx.bonus = re.bonus != 0;
}

// The correction of entry re from the merged candidates of its whole row
// pair: certified in fp32, else the two contenders re-scored in fp64, else
// the sequence goes to the fp64 path.  One thread.
__device__ __forceinline__ void resid_resolve(const Job &j, const ResidEntry &re, const RCtx &ctx,
                                              const Cand2 &all, const uint64_t *skip)
{
    int win = -1;
    if (gumbel_certified(all)) {
        win = all.v1;
    } else if (all.v1 >= 0) {
        double l1 = -INFINITY, h1 = -INFINITY, l2 = -INFINITY, h2 = -INFINITY;
        float x1 = load_logit(j, re.prow, all.v1), y1 = load_logit(j, re.qrow, all.v1);
        resid_interval64(ctx, x1, y1, fine52(ctx.key, all.v1), is_top(ctx.key, all.v1, skip),
                         l1, h1);
        if (all.v2 >= 0) {
            float x2 = load_logit(j, re.prow, all.v2), y2 = load_logit(j, re.qrow, all.v2);
            resid_interval64(ctx, x2, y2, fine52(ctx.key, all.v2),
                             is_top(ctx.key, all.v2, skip), l2, h2);
        }
        const double others = (double)all.hi3;
        if (l1 > fmax(h2, others) + kFlagEps) win = all.v1;
        else if (l2 > fmax(h1, others) + kFlagEps) win = all.v2;
    }
    if (win >= 0 && !j.force_rescue) {
        if (j.kind == K_SAMPLE) {
            j.next[re.b] = win;
            if (j.flags) j.flags[re.b] = 0;
        } else if (re.h < j.commit_len[re.b]) {
            j.committed[(int64_t)re.b * j.K + re.h] = win;
        }
    } else {
        unsigned k = atomicAdd(j.ctl + C_RESCUE_N, 1u);
        RescueEntry x;
        x.b = re.b;
        x.kind = 1;
        x.h = re.h;
        x.resid = 1;
        x.Lp = 0;
        x.Lq = 0;
        x.flags = 0;
        x.bonus = re.bonus;
        x.pad[0] = x.pad[1] = 0;
        j.rescue[k] = x;
    }
}

}  // namespace sv
