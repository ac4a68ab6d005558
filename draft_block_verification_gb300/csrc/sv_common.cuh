// sv_common.cuh -- decision-step helpers shared by the streaming kernel and
// the post-pass kernels (residual draw, total variation, fp64 path).
#pragma once

#include <math.h>

#include "sv_gumbel.cuh"
#include "sv_job.cuh"

namespace sv {

__device__ __forceinline__ int clamp_len(const Job &j, int b)
{
    int n = seq_len(j, b);
    int hi = (j.kind == K_PACKED) ? j.K - 1 : j.K;
    return min(max(n, 0), hi);
}

// ---------------------------------------------------------------------------
// Row merging for the decision step.
// ---------------------------------------------------------------------------
struct RowM {
    float m;            // row max (modes that track it)
    float xd;           // logit at the row's draft token (NaN if not recorded)
    int amax;
    double L2c1, L2c2;  // log2 sum_v 2^(x_v c) with the fp32 factors c1, c2
    double L1a, L1b;    // natural log-sum-exps of x / T for the same two sums
    Cand2 gc;           // Gumbel candidates of the row
};

constexpr double kLn2 = 0.6931471805599453;
constexpr double kLog2e = 1.4426950408889634;

__device__ __forceinline__ RowPart load_part(const RowPart *p)
{
    RowPart r;
    const uint4 *s = reinterpret_cast<const uint4 *>(p);
    uint4 *d = reinterpret_cast<uint4 *>(&r);
#pragma unroll
    for (int i = 0; i < (int)(sizeof(RowPart) / 16); ++i)
        d[i] = __ldcg(s + i);
    return r;
}

// log2 S for S >= 0 with absolute error below 2^-22: S = m 2^k exactly with
// m in [1/2, 1), and log2 m in fp32 (|log2 m| <= 1; log2f is within 1 ulp,
// the rounding of m adds under 2^-23.5).  The fp64 library log2 would cost
// hundreds of cycles per call on a part with a slow fp64 pipe.
__device__ __forceinline__ double log2_fast(double S)
{
    int k;
    const double m = frexp(S, &k);
    return (double)k + (double)log2f((float)m);
}

// e^d in fp32 with relative error below 2^-21 for |d| < 87: d = h + l with
// h = fl32(d), e^d = expf(h) (within 2 ulp) times 1 + l (|l| < 2^-24 |d|,
// e^l - 1 - l below l^2).  Overflows to inf above, flushes to 0 below.
__device__ __forceinline__ float exp_fast(double d)
{
    const float h = (float)d;
    const float l = (float)(d - (double)h);
    return expf(h) * (1.f + l);
}

// Merge the unit records of one row.  Record u holds s_u = sum 2^fl(x c - e_u)
// with an integer e_u; with E = max_u e_u the row sum is
// S = sum_u s_u 2^(e_u - E) (exact scalings), log2 sum 2^(x c) = E + log2 S,
// and the natural log-sum-exp of x/T is ln2 (E c*/c + log2 S) (the exponent
// shift x (c - c*) that is common to all terms taken out).  r1, r2 are the
// ratios c*/c of the two sums (computed on the host in fp64); log2 S carries
// the absolute error of log2_fast.
static __device__ RowM merge_row(const Job &j, int b, int slot, double r1, double r2)
{
    const int nrec = j.parts;
    const RowPart *p = j.rp + ((int64_t)b * j.rows_per_seq + slot) * nrec;
    RowM r;
    r.m = -INFINITY;
    r.xd = __int_as_float(0x7FC00000);
    r.amax = 0x7FFFFFFF;
    r.gc.init();
    // one pass over the records (each read once); a larger exponent moves the
    // running sum by an exact power of two
    float E1 = -INFINITY, E2 = -INFINITY;
    double S1 = 0.0, S2 = 0.0;
    for (int q = 0; q < nrec; ++q) {
        RowPart x = load_part(p + q);
        if (x.m > r.m || (x.m == r.m && x.amax < r.amax)) {
            r.m = x.m;
            r.amax = x.amax;
        }
        r.xd = fmaxf(r.xd, x.xd);
        if (x.s1 > 0.f) {
            if (x.e1 > E1) {
                S1 = (E1 > -INFINITY ? ldexp(S1, (int)(E1 - x.e1)) : 0.0) + (double)x.s1;
                E1 = x.e1;
            } else {
                S1 += ldexp((double)x.s1, (int)(x.e1 - E1));
            }
        }
        if (x.s2 > 0.f) {
            if (x.e2 > E2) {
                S2 = (E2 > -INFINITY ? ldexp(S2, (int)(E2 - x.e2)) : 0.0) + (double)x.s2;
                E2 = x.e2;
            } else {
                S2 += ldexp((double)x.s2, (int)(x.e2 - E2));
            }
        }
        Cand2 c;
        c.hi1 = x.ghi1;
        c.lo1 = x.glo1;
        c.hi2 = x.ghi2;
        c.lo2 = x.glo2;
        c.hi3 = x.ghi3;
        c.v1 = x.gv1;
        c.v2 = x.gv2;
        r.gc.merge(c);
    }
    // a Gumbel-max row's top ids were scored before the stream (seed
    // records, one per chunk of the row); the stream skipped them
    if (j.seeds) {
        const int k = gumbel_index(j, slot);
        if (k >= 0) {
            const SeedRec *sr =
                j.seeds + ((int64_t)b * gumbel_rows(j) + k) * j.seed_chunks;
            for (int q = 0; q < j.seed_chunks; ++q) {
                const float4 a = __ldcg(reinterpret_cast<const float4 *>(sr + q));
                const float4 c4 = __ldcg(reinterpret_cast<const float4 *>(sr + q) + 1);
                Cand2 c;
                c.hi1 = a.y;
                c.lo1 = a.z;
                c.hi2 = a.w;
                c.lo2 = c4.x;
                c.hi3 = c4.y;
                c.v1 = __float_as_int(c4.z);
                c.v2 = __float_as_int(c4.w);
                r.gc.merge(c);
            }
        }
    }
    const double l1 = log2_fast(S1), l2 = log2_fast(S2);
    r.L2c1 = (double)E1 + l1;
    r.L2c2 = (double)E2 + l2;
    r.L1a = kLn2 * ((double)E1 * r1 + l1);
    r.L1b = kLn2 * ((double)E2 * r2 + l2);
    return r;
}

__device__ __forceinline__ const char *row_ptr(const Job &j, int b, int slot)
{
    return slot_row(j, b, slot);
}

__device__ __forceinline__ float load_logit(const Job &j, const char *row, int v)
{
    return j.dtype == SV_BF16 ? VecTraits<uint16_t>::load1(row, v) : VecTraits<float>::load1(row, v);
}

__device__ __forceinline__ double alpha_of(int mode, double r, double lam)
{
    double a = (mode == SV_LENIENT_RATIO) ? lam * r
             : (mode == SV_LENIENT_LINEAR) ? (1.0 - lam) * r + lam
                                           : r;
    return a < 1.0 ? a : 1.0;
}

// ---------------------------------------------------------------------------
// Modified Cactus lenience ([TwoTrade] App. E).  The drafted token y with
// target probability p gets gamma*: the largest gamma in [p, 1] with
//   Phi(gamma) = gamma log(gamma/p) + (1-gamma) log((1-gamma)/(1-p)) <= delta
// (eq. 17); every other token is scaled by c = (1-gamma*)/(1-p).  Phi rises
// from 0 at p to log(1/p) at 1, so gamma* = 1 when delta >= log(1/p).
// ---------------------------------------------------------------------------
// Phi(g) - delta in fp64, with both logs taken as log1p of small quotients
// (g near p when delta is small); *scale receives the size of its terms.
__device__ __forceinline__ double cactus_f(double g, double p, double delta, double *d1,
                                           double *scale)
{
    const double a = log1p((g - p) / p);          // log(g / p)
    const double b = log1p((p - g) / (1.0 - p));  // log((1 - g) / (1 - p))
    *d1 = a - b;                                  // Phi'(g)
    *scale = fabs(g * a) + fabs((1.0 - g) * b) + delta;
    return g * a + (1.0 - g) * b - delta;
}

// gamma* by Newton's method (the page's solver), started at the page's
// second-order solution p + sqrt(2 delta p (1-p)) and kept inside the
// bracket of the root by bisection steps.  Returns a verified bracket
// [*glo, *ghi] of gamma*: the Newton point widened by 1e-10 relative on each
// side, each side checked to lie on its side of the root with a margin of
// 64 roundings of Phi's terms.  false when the check fails (the caller then
// treats the decision as undecided).  fp64; a few hundred cycles per step on
// this part's fp64 pipe, run for the few draft positions of one sequence.
static __device__ __noinline__ bool cactus_bracket(double p, double delta, double *glo, double *ghi)
{
    if (!(p > 0.0)) {
        *glo = *ghi = 0.0;
        return true;
    }
    if (p >= 1.0 || delta >= -log(p)) {  // Phi(1) = log(1/p)
        *glo = *ghi = 1.0;
        return p >= 1.0 || delta > -log(p) * (1.0 + 1e-15);
    }
    if (!(delta > 0.0)) {
        *glo = *ghi = p;
        return true;
    }
    double lo = p, hi = 1.0;
    double g = p + sqrt(2.0 * delta * p * (1.0 - p));
    if (!(g > lo && g < hi))
        g = 0.5 * (lo + hi);
    for (int it = 0; it < 64; ++it) {
        double d1, sc;
        const double f = cactus_f(g, p, delta, &d1, &sc);
        if (f > 0.0)
            hi = g;
        else
            lo = g;
        double gn = g - f / d1;
        if (!(gn > lo && gn < hi))
            gn = 0.5 * (lo + hi);
        if (gn == g || hi - lo <= 4e-16 * hi)
            break;
        g = gn;
    }
    const double a = fmax(p, g * (1.0 - 1e-10)), b = fmin(1.0, g * (1.0 + 1e-10));
    double d1, sa, sb;
    const double fa = cactus_f(a, p, delta, &d1, &sa);
    bool ok = a == p || fa < -64.0 * 0x1p-53 * sa;
    if (b < 1.0) {
        const double fb = cactus_f(b, p, delta, &d1, &sb);
        ok = ok && fb > 64.0 * 0x1p-53 * sb;
    }
    *glo = a;
    *ghi = b;
    return ok;
}

// Newton's method for gamma* in fp32 (the same steps and logs as
// cactus_bracket), for the fast path's bracket below.
__device__ __forceinline__ float cactus_newton32(float p, float delta)
{
    float lo = p, hi = 1.f;
    float g = p + sqrtf(2.f * delta * p * (1.f - p));
    if (!(g > lo && g < hi))
        g = 0.5f * (lo + hi);
    for (int it = 0; it < 24; ++it) {
        const float a = log1pf((g - p) / p), b = log1pf((p - g) / (1.f - p));
        const float f = g * a + (1.f - g) * b - delta;
        if (f > 0.f)
            hi = g;
        else
            lo = g;
        float gn = g - f / (a - b);
        if (!(gn > lo && gn < hi))
            gn = 0.5f * (lo + hi);
        if (gn == g)
            break;
        g = gn;
    }
    return g;
}

// Bracket [*glo, *ghi] of gamma*(p) for every p in [plo, phi] (gamma* grows
// with p): the fp32 Newton points at plo and phi, widened by 2^-14
// relative, each checked in fp64 to lie on its side of its root (margin of
// 64 roundings of Phi's terms).  Two fp64 evaluations of Phi in all; falls
// back to the fp64 Newton of cactus_bracket when a check fails, or when p
// reaches emd = exp(-delta) (1 - 1e-12), below which gamma* < 1 (Phi(1) =
// log(1/p) > delta).  false when no bracket could be certified.
static __device__ __noinline__ bool cactus_bracket_fast(double plo, double phi, double delta,
                                                 double emd, double *glo, double *ghi)
{
    double d1, sc;
    bool ok_lo, ok_hi;
    if (!(plo > 0.0) || !(delta > 0.0) || plo >= emd) {
        double a;
        ok_lo = cactus_bracket(plo, delta, glo, &a);
    } else {
        *glo = fmax(plo, (double)cactus_newton32((float)plo, (float)delta) * (1.0 - 0x1p-14));
        const double f = cactus_f(*glo, plo, delta, &d1, &sc);
        ok_lo = *glo == plo || f < -64.0 * 0x1p-53 * sc;
        if (!ok_lo) {
            double a;
            ok_lo = cactus_bracket(plo, delta, glo, &a);
        }
    }
    if (phi >= 1.0 || !(delta > 0.0) || phi >= emd) {
        double a;
        ok_hi = cactus_bracket(phi, delta, &a, ghi);
    } else {
        *ghi = fmin(1.0, (double)cactus_newton32((float)fmin(phi, 1.0), (float)delta) *
                             (1.0 + 0x1p-14));
        ok_hi = *ghi >= 1.0;
        if (!ok_hi) {
            const double f = cactus_f(*ghi, phi, delta, &d1, &sc);
            ok_hi = f > 64.0 * 0x1p-53 * sc;
        }
        if (!ok_hi) {
            double a;
            ok_hi = cactus_bracket(phi, delta, &a, ghi);
        }
    }
    return ok_lo && ok_hi;
}

// Acceptance probability min{1, gamma* / q} in fp64 from log p(d), log q(d)
// (the fp64 path); gamma* is the middle of its bracket.
__device__ __forceinline__ double cactus_alpha64(double lp, double lq, double delta)
{
    const double p = exp(lp);
    double glo, ghi;
    cactus_bracket(p, delta, &glo, &ghi);
    const double g = 0.5 * (glo + ghi);
    const double a = exp((g == p ? lp : log(g)) - lq);
    return a < 1.0 ? a : 1.0;
}

// log c = log((1 - gamma*)/(1 - p)) for the residual in fp64 (the fp64 path).
__device__ __forceinline__ double cactus_log_scale64(double lp, double delta)
{
    const double p = exp(lp);
    double glo, ghi;
    cactus_bracket(p, delta, &glo, &ghi);
    const double g = 0.5 * (glo + ghi);
    if (g == p)
        return 0.0;
    return log1p(-g) - log1p(-p);
}

// Acceptance probability of any rule in fp64 (the fp64 path).
__device__ __forceinline__ double alpha_exact(int mode, double lp, double lq, double lam)
{
    if (mode == SV_LENIENT_CACTUS)
        return cactus_alpha64(lp, lq, lam);
    return alpha_of(mode, exp(lp - lq), lam);
}

// ---------------------------------------------------------------------------
// Level 3 of the Gumbel-max filter for a logit row (score x/T + G).
// ---------------------------------------------------------------------------
struct GRes {
    int v;     // winner
    int flag;  // best and second-best fp64 scores closer than 1e-9
};

__device__ __forceinline__ double exact_logit_score(const Job &j, const char *row, uint64_t key,
                                                    double T, int v)
{
    float x = load_logit(j, row, v);
    return (double)x / T + gumbel64(fine52(key, (uint32_t)v), is_top(key, (uint32_t)v, j.skip));
}

// The best candidate's lower end beats every other upper end by > 1e-9.
__device__ __forceinline__ bool gumbel_certified(const Cand2 &c)
{
    float other = fmaxf(c.hi2, c.hi3);
    return c.v1 >= 0 && ((double)c.lo1 - (double)other > kFlagEps);
}

// Warp-level (all 32 lanes, uniform arguments).  Certified candidates return
// at once; otherwise the two kept candidates are scored in fp64, and if some
// other element's upper end still reaches within 1e-9 of the best (rare) the
// whole row is rescanned with fp64 scores for everything its table bound
// admits.
static __device__ __noinline__ GRes resolve_logit_row(const Job &j, const char *row, uint64_t key, double T,
                                         float invT, const Cand2 &c)
{
    if (gumbel_certified(c))
        return GRes{c.v1, 0};
    double s1 = (c.v1 >= 0) ? exact_logit_score(j, row, key, T, c.v1) : -INFINITY;
    double s2 = (c.v2 >= 0) ? exact_logit_score(j, row, key, T, c.v2) : -INFINITY;
    bool first = c.v2 < 0 || s1 > s2 || (s1 == s2 && c.v1 < c.v2);
    double best = first ? s1 : s2, second = first ? s2 : s1;
    if ((double)c.hi3 < best - kFlagEps)
        return GRes{first ? c.v1 : c.v2, (best - second < kFlagEps) ? 1 : 0};
    const int lane = threadIdx.x & 31;
    const float thr = level1_thr(__double2float_rd(best - 2.0 * kFlagEps));
    Top2 t;
    t.init();
    for (int v = lane; v < j.V; v += 32) {
        const float x = load_logit(j, row, v);
        const uint64_t m = fine52(key, (uint32_t)v);
        const bool top = is_top(key, (uint32_t)v, j.skip);
        if (!top && fmaf(x, invT, __ldg(j.gtab + (int)(m >> 44))) < thr)
            continue;
        t.add((double)x / T + gumbel64(m, top), v);
    }
    warp_top2(t);
    return GRes{t.i1, (t.s1 - t.s2 < kFlagEps) ? 1 : 0};
}

// Warp-level: each lane holds the candidates of one logit row (need = false
// when it holds none); rows that are not certified are resolved one at a time
// by the whole warp.  Returns the lane's winner and near-tie flag.
static __device__ __noinline__ GRes resolve_lanes(const Job &j, const char *row, uint64_t key, double T,
                                     float invT, const Cand2 &c, bool need)
{
    const int lane = threadIdx.x & 31;
    GRes out{c.v1, 0};
    unsigned m = __ballot_sync(0xFFFFFFFFu, need && !gumbel_certified(c));
    while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const char *r2 = (const char *)__shfl_sync(0xFFFFFFFFu, (unsigned long long)row, src);
        uint64_t k2 = __shfl_sync(0xFFFFFFFFu, (unsigned long long)key, src);
        double T2 = __shfl_sync(0xFFFFFFFFu, T, src);
        float i2 = __shfl_sync(0xFFFFFFFFu, invT, src);
        Cand2 c2;
        c2.hi1 = __shfl_sync(0xFFFFFFFFu, c.hi1, src);
        c2.lo1 = __shfl_sync(0xFFFFFFFFu, c.lo1, src);
        c2.hi2 = __shfl_sync(0xFFFFFFFFu, c.hi2, src);
        c2.lo2 = __shfl_sync(0xFFFFFFFFu, c.lo2, src);
        c2.hi3 = __shfl_sync(0xFFFFFFFFu, c.hi3, src);
        c2.v1 = __shfl_sync(0xFFFFFFFFu, c.v1, src);
        c2.v2 = __shfl_sync(0xFFFFFFFFu, c.v2, src);
        GRes r = resolve_logit_row(j, r2, k2, T2, i2, c2);
        if (lane == src)
            out = r;
    }
    return out;
}

// Writes the stopping index, the committed tokens, the next draft and the
// flags of a Packed-SS sequence once h is decided ([PackedSS] Alg. 1 lines
// 6-10, Alg. 2 lines 8-13).  The correction c may still be unknown (c_known
// false): it is then written later at committed[b, h] by the residual kernel;
// an EOS at index h can only give a = h + 1, so a never depends on c.
// Shared with the fp64 path.  Called by one full warp.
static __device__ void packed_commit(const Job &j, int b, int h, int c, bool c_known, int flags_base)
{
    const int lane = threadIdx.x & 31;
    const int Km1 = j.K - 1;
    int d = (lane < h) ? __ldg(j.ids + (int64_t)b * Km1 + lane) : -1;
    bool eos = (j.eos >= 0) && (lane < h) && (d == j.eos);
    unsigned em = __ballot_sync(0xFFFFFFFFu, eos);
    int a = h + 1;
    if (j.remaining)
        a = min(a, max(__ldg(j.remaining + b), 0));
    if (em)
        a = min(a, __ffs(em));  // first EOS at 1-indexed position i
    if (c_known && j.eos >= 0 && c == j.eos)
        a = min(a, h + 1);
    if (lane < j.K) {
        int tok = -1;
        if (lane < a)
            tok = (lane < h) ? d : (c_known ? c : -1);
        j.committed[(int64_t)b * j.K + lane] = tok;
    }
    int nl = max(0, j.W - a);
    int gf = 0;
    if (lane < j.W) {
        const float nan = __int_as_float(0x7FC00000);
        int src = a + lane;
        DraftTmp t = (lane < nl) ? j.dtmp[(int64_t)b * j.W + src] : DraftTmp{-1, 0, nan, 0.f};
        j.next_draft[(int64_t)b * j.W + lane] = t.z;
        if (j.next_q) j.next_q[(int64_t)b * j.W + lane] = (lane < nl) ? t.q : nan;
        gf = (lane < nl) ? t.gflag : 0;
    }
    for (int o = 16; o; o >>= 1)
        gf += __shfl_xor_sync(0xFFFFFFFFu, gf, o);
    if (lane == 0) {
        j.acc[b] = h;
        j.commit_len[b] = a;
        j.next_len[b] = nl;
        if (j.flags) j.flags[b] = flags_base + gf;
    }
}

// Launch configuration that allows programmatic dependent launch: the
// kernel may be scheduled while the previous kernel of the stream finishes
// (it calls pdl_wait before it touches global memory).
inline void pdl_config(cudaLaunchConfig_t &cfg, cudaLaunchAttribute (&at)[1], dim3 grid,
                       dim3 block, size_t smem, cudaStream_t s)
{
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
}

}  // namespace sv
