// sv_gumbel.cuh -- the uniforms of a row and Gumbel-max over a vocabulary row.
//
// Uniforms.  All randomness of a row is read from the SplitMix64 stream
// seeded with the row key k (stream_at(k, n) = output n + 1).  The ids are
// split into blocks of 256.  Which ids of a block fall into the top 1/256 of
// the unit interval ("top" ids) is drawn as i.i.d. Bernoulli(1/256) trials by
// geometric skipping: draw i of block b is M = stream_at(k, b * 2^16 + i); its
// gap is the number of g in 1..256 with M < C_g, C_g = ceil(2^64 (255/256)^g)
// (so P(gap >= g) = (255/256)^g to within 2^-64); the first top offset is
// gap_0, each next one the previous plus 1 + gap_i.  The 52 fine bits of id v
// are m = stream_at(k, 2^40 + v) >> 12, w = (2m + 1) / 2^53, and
// u = w * 255/256 for an ordinary id, 1 - u = (1 - w) / 256 for a top id.
//
// Gumbel-max.  The sample is argmax_v s_v, s_v = z_v + G(v) (z = x/T for a
// logit row, or the residual log-weight of [SPOT] App. B eq. 14), with
// G = -log(-log u) ([SPOT] eq. 4, the Gumbel-argmax identity eqs. 5-7).  The
// layout makes a row cheap to screen:
//   top ids (about one per block) are found from a couple of draws per block
//   and scored first, which gives a threshold close to the row's maximum;
//   an ordinary id has G < G(255/256) = 5.5414..., so a vector of ids whose
//   largest score bound stays below the threshold is skipped at once; ids of
//   the few vectors that pass are bounded by the top byte of their fine bits
//   (a 256-entry table), and survivors get G in fp32 with a proved interval;
//   the two candidates with the largest upper ends are certified (lower end
//   of the best > upper end of every other + 1e-9), or evaluated in fp64.
#pragma once

#include "sv_dev.cuh"

namespace sv {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr int kGTab = 256;   // G bounds of an ordinary id by the top byte of its fine bits
constexpr int kSkipN = 257;  // skip thresholds C_1..C_256 (entry 0 unused)
// |G32 - G| bound for the fp32 evaluation below (about 8x the analysis: the
// two lg2.approx calls and the argument rounding give under 2^-20; a GPU
// self-test measures it).
constexpr float kG32Err = 0x1p-17f;

__host__ __device__ __forceinline__ uint64_t stream_at(uint64_t key, uint64_t n)
{
    return splitmix_out(key + n * kGamma);
}

// The 52 fine bits of id v.
__device__ __forceinline__ uint64_t fine52(uint64_t key, uint32_t v)
{
    return stream_at(key, (1ull << 40) + v) >> 12;
}

// Gap of a skip draw: the largest g in 0..256 with M < C_g (C decreasing,
// C_0 taken as 2^64), i.e. g = floor(t), t = log(u) / log(255/256), u = M /
// 2^64, capped at 256.  t is estimated from log2 of u rounded to 24 bits.
// For u >= 0.36 (t <= 257) the estimate is within 1e-4 of t: the rounding of
// u moves log2 u by at most 2^-25 / (0.36 ln 2) < 1.2e-7, lg2.approx errs by
// at most 2^-22.6 < 1.7e-7, and the product and its constant add under
// 4.2e-5.  So an estimate more than kGapEps = 2^-9 away from every integer
// (and from 256) has the exact floor; the rest, about 0.4 % of draws, are
// corrected against the exact thresholds.
constexpr float kGapEps = 0x1p-9f;

__device__ __forceinline__ int skip_gap(uint64_t M, const uint64_t *__restrict__ C)
{
    float u = __uint2float_rn((uint32_t)(M >> 40)) * 0x1p-24f + 0x1p-25f;
    float l2;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(u));
    // 1 / log2(255/256) = -177.0989; u < 1 so the estimate is >= 0
    const float t = l2 * -177.09888f;
    if (t >= 256.f + kGapEps)
        return 256;
    const float fl = floorf(t), fr = t - fl;
    if (fr >= kGapEps && fr <= 1.f - kGapEps && t < 256.f)
        return (int)fl;
    int g = (int)fminf(t, 256.f);
    g = max(0, min(g, 256));
    while (g < 256 && M < C[g + 1])
        ++g;
    while (g > 0 && M >= C[g])
        --g;
    return g;
}

// Offset of the next top id of block beta after draw i (pos: the previous
// offset, -1 before the first draw).
__device__ __forceinline__ int next_top(uint64_t key, uint32_t beta, int i, int pos,
                                        const uint64_t *__restrict__ C)
{
    return pos + 1 + skip_gap(stream_at(key, ((uint64_t)beta << 16) | (uint32_t)i), C);
}

// Top ids among offsets o0 .. o0 + n - 1 of block beta, as a bit mask (n <= 32).
__device__ __forceinline__ uint32_t top_mask(uint64_t key, uint32_t beta, int o0, int n,
                                             const uint64_t *__restrict__ C)
{
    uint32_t msk = 0;
    int pos = -1;
    for (int i = 0; i < 257; ++i) {  // offsets grow by at least one per draw
        pos = next_top(key, beta, i, pos, C);
        if (pos >= o0 + n)
            break;
        if (pos >= o0)
            msk |= 1u << (pos - o0);
    }
    return msk;
}

__device__ __forceinline__ bool is_top(uint64_t key, uint32_t v, const uint64_t *__restrict__ C)
{
    return top_mask(key, v >> 8, (int)(v & 255u), 1, C) != 0u;
}

// u and 1 - u as integers over 2^61 (both exact).
__device__ __forceinline__ void u_parts(uint64_t m, bool top, uint64_t &un, uint64_t &dn)
{
    if (top) {
        dn = (1ull << 53) - 2 * m - 1;
        un = (1ull << 61) - dn;
    } else {
        un = 255ull * (2 * m + 1);
        dn = (1ull << 61) - un;
    }
}

// The uniform and the Gumbel value in fp64 (the same expressions as the
// definition, so the values are reproducible bit for bit).
__device__ __forceinline__ double uniform64(uint64_t m, bool top)
{
    const double w = (double)(2 * m + 1) * 0x1p-53;
    return top ? 1.0 - (1.0 - w) / 256.0 : w * (255.0 / 256.0);
}
__device__ __forceinline__ double gumbel64(uint64_t m, bool top)
{
    const double w = (double)(2 * m + 1) * 0x1p-53;
    if (top)
        return -log(-log1p(-((1.0 - w) / 256.0)));
    return -log(-log(w * (255.0 / 256.0)));
}
__device__ __forceinline__ double uniform_at(uint64_t key, uint32_t v,
                                             const uint64_t *__restrict__ C)
{
    return uniform64(fine52(key, v), is_top(key, v, C));
}

__device__ __forceinline__ float lg2a(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// G = -ln(E), E = -ln(u), in fp32.  For u < 3/4, E comes from lg2 of u (u is
// exact to 2^-24).  For u >= 3/4, d = 1 - u is exact as an integer over 2^61
// and E = -ln(1 - d) = 2 atanh(d / (2 - d)) by its odd series in
// s = d/(2-d) <= 1/7, truncated after s^9 (relative error < 4e-10).
__device__ __forceinline__ float gumbel32(uint64_t m, bool top)
{
    const float ln2 = 0.693147180559945f;
    uint64_t un, dn;
    u_parts(m, top, un, dn);
    float E;
    if (un < (3ull << 59)) {
        float u = __ull2float_rn(un) * 0x1p-61f;
        E = -ln2 * lg2a(u);
    } else {
        float d = __ull2float_rn(dn) * 0x1p-61f;
        float s = __fdiv_rn(d, 2.f - d);
        float s2 = s * s;
        float p = fmaf(s2, 1.f / 9.f, 1.f / 7.f);
        p = fmaf(s2, p, 1.f / 5.f);
        p = fmaf(s2, p, 1.f / 3.f);
        p = fmaf(s2, p, 1.f);
        E = 2.f * s * p;
    }
    return -ln2 * lg2a(E);
}

// Bound of G over every ordinary id (the table's last entry).
__device__ __forceinline__ float g_ordinary_max(const float *tab) { return tab[kGTab - 1]; }

// Threshold used against level-1 (table) bounds: an fp32 bound ub of an
// exact score satisfies exact <= ub + (|ub| + 40) 2^-21, so an element whose
// ub is at most thr - (|thr| + 41) 2^-21 stays at least about 2^-21 below thr
// and cannot reach it.  The threshold is rounded down at each step, so the
// fp32 value never exceeds that real bound.
__device__ __forceinline__ float level1_thr(float thr)
{
    return __fsub_rd(thr, __fmul_ru(__fadd_ru(fabsf(thr), 41.f), 0x1p-21f));
}

// Candidates with the two largest upper ends, and the largest upper end of
// every other candidate seen (hi3).
struct Cand2 {
    float hi1, lo1, hi2, lo2, hi3;
    int v1, v2;
    __device__ __forceinline__ void init()
    {
        hi1 = lo1 = hi2 = lo2 = hi3 = -INFINITY;
        v1 = v2 = -1;
    }
    __device__ __forceinline__ void add(float lo, float hi, int v)
    {
        if (v1 < 0 || hi > hi1 || (hi == hi1 && v < v1)) {
            if (v2 >= 0) hi3 = fmaxf(hi3, hi2);
            hi2 = hi1;
            lo2 = lo1;
            v2 = v1;
            hi1 = hi;
            lo1 = lo;
            v1 = v;
        } else if (v2 < 0 || hi > hi2 || (hi == hi2 && v < v2)) {
            if (v2 >= 0) hi3 = fmaxf(hi3, hi2);
            hi2 = hi;
            lo2 = lo;
            v2 = v;
        } else {
            hi3 = fmaxf(hi3, hi);
        }
    }
    __device__ __forceinline__ void merge(const Cand2 &o)
    {
        if (o.v1 >= 0) add(o.lo1, o.hi1, o.v1);
        if (o.v2 >= 0) add(o.lo2, o.hi2, o.v2);
        hi3 = fmaxf(hi3, o.hi3);
    }
    // Best lower end among the two kept candidates.
    __device__ __forceinline__ float lomax() const { return fmaxf(lo1, lo2); }
};

// The warp's best candidate by (upper end desc, id asc) when each lane
// offers (hi, v, lo), v = -1 for none: two 32-bit warp reductions and a
// ballot.  hi, v and lo become the winner's in every lane; returns the
// winning lane, or -1 when no lane offers a candidate.
__device__ __forceinline__ int warp_best(float &hi, int &v, float &lo)
{
    const uint32_t h = f2ord(hi);
    const uint32_t hm = __reduce_max_sync(0xFFFFFFFFu, h);
    const bool top = h == hm && v >= 0;
    const int vm = __reduce_min_sync(0xFFFFFFFFu, top ? v : 0x7FFFFFFF);
    const unsigned wins = __ballot_sync(0xFFFFFFFFu, top && v == vm);
    if (wins == 0u) {
        hi = ord2f(hm);
        v = -1;
        lo = -INFINITY;
        return -1;
    }
    const int wl = __ffs(wins) - 1;
    hi = __shfl_sync(0xFFFFFFFFu, hi, wl);
    v = __shfl_sync(0xFFFFFFFFu, v, wl);
    lo = __shfl_sync(0xFFFFFFFFu, lo, wl);
    return wl;
}

// The warp's merged candidates in every lane: its top two by (upper end
// desc, id asc) and the largest upper end of every other candidate.  Each
// lane holds its own top two and hi3, with distinct ids across lanes.  Every
// lane of the warp calls it.
__device__ __forceinline__ void warp_cand2(Cand2 &c)
{
    const int lane = threadIdx.x & 31;
    float h1 = c.hi1, l1 = c.lo1;
    int v1 = c.v1;
    const int w1 = warp_best(h1, v1, l1);
    // each lane's best remaining candidate
    float h2 = lane == w1 ? c.hi2 : c.hi1, l2 = lane == w1 ? c.lo2 : c.lo1;
    int v2 = lane == w1 ? c.v2 : c.v1;
    const int w2 = warp_best(h2, v2, l2);
    // the largest upper end left in each lane once the two kept are out
    float rest = c.v1 >= 0 ? c.hi1 : -INFINITY;
    if (lane == w1 && lane == w2)
        rest = c.v2 >= 0 ? c.hi3 : -INFINITY;
    else if (lane == w1 || lane == w2)
        rest = fmaxf(c.v2 >= 0 ? c.hi2 : -INFINITY, c.hi3);
    const uint32_t r = __reduce_max_sync(0xFFFFFFFFu, f2ord(rest));
    c.hi1 = h1;
    c.lo1 = l1;
    c.v1 = v1;
    c.hi2 = h2;
    c.lo2 = l2;
    c.v2 = v2;
    c.hi3 = fmaxf(ord2f(r), -INFINITY);
}

// fp32 interval (lo, hi) of the Gumbel-perturbed logit x/T + G for id v with
// fine bits m (top: whether v is a top id).
__device__ __forceinline__ float2 logit_interval_m(float x, float invT, uint64_t m, bool top)
{
    float z = x * invT;
    float g = gumbel32(m, top);
    float s = z + g;
    float e = (fabsf(z) + fabsf(s)) * 0x1p-21f + kG32Err;
    return make_float2(s - e, s + e);
}

// A lower bound of x/T + G for an id whose G is at least glo (a table value
// rounded down, so exact as a bound): the rounding of x/T and of the sum is
// covered by the same slack as the interval's lower end above.
__device__ __forceinline__ float logit_lower_bound(float x, float invT, float glo)
{
    const float z = x * invT;
    const float s = z + glo;
    return s - ((fabsf(z) + fabsf(s)) * 0x1p-21f + kG32Err);
}

// The same for id v.  Out of line: it runs for a few ids per row.
static __device__ __noinline__ float2 logit_interval_at(float x, float invT, uint64_t key, uint32_t v,
                                                        bool top)
{
    float z = x * invT;
    float g = gumbel32(fine52(key, v), top);
    float s = z + g;
    float e = (fabsf(z) + fabsf(s)) * 0x1p-21f + kG32Err;
    return make_float2(s - e, s + e);
}

}  // namespace sv
