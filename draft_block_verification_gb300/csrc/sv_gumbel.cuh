// sv_gumbel.cuh -- Gumbel-max over a vocabulary row with a three-level filter.
//
// The sample is argmax_v s_v, s_v = z_v + G(key, v) (z = x/T for a logit row,
// or the residual log-weight of [SPOT] App. B eq. 14), with G = -log(-log u)
// ([SPOT] eq. 4, the Gumbel-argmax identity eqs. 5-7).  u's 52 random bits are
// laid out so that a whole row can be screened cheaply:
//   level 1: one 32-bit hash per 4 ids gives each id the top 8 bits of u,
//            bounding G by a 256-entry table; a group of 4 is skipped unless
//            one of its bytes is 0xFF or its largest logit can still reach
//            the running threshold;
//   level 2: survivors get G in fp32 with a proved interval, and s_v an
//            interval [lo, hi];
//   level 3: the two candidates with the largest upper ends are certified
//            (lower end of the best > upper end of every other + 1e-9), or
//            evaluated in fp64 when their intervals overlap.
#pragma once

#include "sv_dev.cuh"

namespace sv {

constexpr int kG8 = 256;            // coarse table: G at the top of each 8-bit bucket
constexpr int kGTab = 2 * kG8;      // + the 256 sub-buckets of the top bucket
// |G32 - G| bound for the fp32 evaluation below (about 8x the analysis: the
// two lg2.approx calls and the argument rounding give under 2^-20; a GPU
// self-test measures it).
constexpr float kG32Err = 0x1p-17f;

__device__ __forceinline__ uint32_t word_a(uint32_t klo, uint32_t j)
{
    return murmur_fmix(klo ^ (j * 0x9E3779B9u));
}
__device__ __forceinline__ uint32_t word_b(uint32_t khi, uint32_t j)
{
    return murmur_fmix(khi ^ (j * 0x85EBCA77u));
}

// 52 random bits of id v whose top byte b0 is known.
__device__ __forceinline__ uint64_t bits52_of(uint64_t key, uint32_t v, uint32_t b0)
{
    uint32_t b1 = (word_b((uint32_t)(key >> 32), v >> 2) >> (8u * (v & 3u))) & 0xFFu;
    uint64_t low = splitmix_out(key ^ ((uint64_t)v * 0xD1B54A32D192ED03ull)) >> 28;
    return ((uint64_t)b0 << 44) | ((uint64_t)b1 << 36) | low;
}
__device__ __forceinline__ uint64_t bits52_full(uint64_t key, uint32_t v)
{
    uint32_t b0 = (word_a((uint32_t)key, v >> 2) >> (8u * (v & 3u))) & 0xFFu;
    return bits52_of(key, v, b0);
}
__device__ __forceinline__ double u_of(uint64_t m)
{
    return (double)(2 * m + 1) * 0x1p-53;
}
__device__ __forceinline__ double uniform_at(uint64_t key, uint32_t v)
{
    return u_of(bits52_full(key, v));
}

// Level-1 bound of G for id v: byte b0 of word a; if b0 == 255, the next
// byte (word b) selects a sub-bucket.  The table is rounded up.
__device__ __forceinline__ float gup_of(const float *tab, uint64_t key, uint32_t v, uint32_t b0)
{
    if (b0 != 255u)
        return tab[b0];
    uint32_t b1 = (word_b((uint32_t)(key >> 32), v >> 2) >> (8u * (v & 3u))) & 0xFFu;
    return tab[kG8 + b1];
}

__device__ __forceinline__ float lg2a(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// G = -ln(E), E = -ln(u), u = (2m+1) 2^-53, in fp32.  For u < 3/4, E comes
// from lg2 of u (u is exact to 2^-24).  For u >= 3/4, 1 - u is exact as the
// integer 2^53 - 2m - 1 and E = -ln(1 - d) = 2 atanh(d / (2 - d)) by its odd
// series in s = d/(2-d) <= 1/7, truncated after s^9 (relative error < 4e-10).
__device__ __forceinline__ float gumbel32(uint64_t m)
{
    const float ln2 = 0.693147180559945f;
    float E;
    if (m < (3ull << 50)) {
        float u = __ull2float_rn(2 * m + 1) * 0x1p-53f;
        E = -ln2 * lg2a(u);
    } else {
        float d = __ull2float_rn((1ull << 53) - 2 * m - 1) * 0x1p-53f;
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

// Largest finite entry of the coarse table (b0 = 254), for the group test.
__device__ __forceinline__ float g8max(const float *tab) { return tab[kG8 - 2]; }

// Threshold used against level-1 (table) bounds: an fp32 bound ub of an
// exact score satisfies exact <= ub + (|ub| + 40) 2^-21, so comparing ub with
// thr - (|thr| + 41) 2^-21 never drops an element that can reach thr.
__device__ __forceinline__ float level1_thr(float thr)
{
    return thr - (fabsf(thr) + 41.f) * 0x1p-21f;
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

__device__ __forceinline__ void warp_cand2(Cand2 &c)
{
    for (int o = 16; o; o >>= 1) {
        Cand2 p;
        p.hi1 = __shfl_xor_sync(0xFFFFFFFFu, c.hi1, o);
        p.lo1 = __shfl_xor_sync(0xFFFFFFFFu, c.lo1, o);
        p.hi2 = __shfl_xor_sync(0xFFFFFFFFu, c.hi2, o);
        p.lo2 = __shfl_xor_sync(0xFFFFFFFFu, c.lo2, o);
        p.hi3 = __shfl_xor_sync(0xFFFFFFFFu, c.hi3, o);
        p.v1 = __shfl_xor_sync(0xFFFFFFFFu, c.v1, o);
        p.v2 = __shfl_xor_sync(0xFFFFFFFFu, c.v2, o);
        c.merge(p);
    }
}

// fp32 interval (lo, hi) of the Gumbel-perturbed logit x/T + G for id v with
// top byte b0.  Out of line: it runs for a few ids per row, and inlining it
// into the unrolled streaming loops would flood the instruction cache.
static __device__ __noinline__ float2 logit_interval_at(float x, float invT, uint64_t key, uint32_t v,
                                                        uint32_t b0)
{
    float z = x * invT;
    float g = gumbel32(bits52_of(key, v, b0));
    float s = z + g;
    float e = (fabsf(z) + fabsf(s)) * 0x1p-21f + kG32Err;
    return make_float2(s - e, s + e);
}

}  // namespace sv
