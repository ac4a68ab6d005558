// sv_dev.cuh -- device-side building blocks of libsv: the counter-based random
// numbers, error latching, mbarrier / bulk-copy wrappers, per-row partial
// records and warp reductions.
//
// Sources (short names used in comments):
//   [PackedSS] "One Call Ahead: Packed Self-Speculative Decoding with Diffusion Drafting"
//   [SPOT]     "On the SPOT: Enhancing Speculative Decoding for Diffusion Language Models
//               via Commit-Order Prediction"
//   [TwoTrade] "Speculative Diffusion is a Tale of Two Tradeoffs"
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sv.h"

namespace sv {

// ---------------------------------------------------------------------------
// Launch geometry of the streaming kernel: one CTA per SM with 16 consumer
// warps, each thread taking 4 16-byte vectors of a 32 KB stage, and a ring of
// 4 stages (128 KB in flight per SM).  Chosen by measurement on GB300 among
// 8-17 consumer warps, 16-36 KB stages and 4-7 stages: more consumer warps
// hide the per-element dependency chains, which dominate the rows that carry
// a Gumbel-max (16 warps against 12: tree T = 1 and Packed-SS T = 1 steps 8%
// and 13% faster, the lossless step 1% faster, Packed-SS T = 0 4% slower).
// 19 warps round up to 20 in the register file, so a thread gets 96
// registers.
// ---------------------------------------------------------------------------
#ifndef SV_CONSUMER_WARPS
#define SV_CONSUMER_WARPS 16
#endif
#ifndef SV_STAGES
#define SV_STAGES 4
#endif
#ifndef SV_STAGE_BYTES
#define SV_STAGE_BYTES 32768
#endif
#ifndef SV_SPIN_SLEEP_NS
#define SV_SPIN_SLEEP_NS 64
#endif
#ifndef SV_MIN_BLOCKS
#define SV_MIN_BLOCKS 1
#endif
constexpr int kConsumerWarps = SV_CONSUMER_WARPS;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kPassThreads = kConsumers + 96;     // + producer, finalizer and planner warps
constexpr int kStageBytes = SV_STAGE_BYTES;       // one bulk copy
constexpr int kStageVecs = kStageBytes / 16;      // 16-byte vectors per stage
constexpr int kVecsPerThread = kStageVecs / kConsumers;
constexpr int kStages = SV_STAGES;
static_assert(kVecsPerThread * kConsumers == kStageVecs, "stage must split evenly");
constexpr int ceil_log2(int n) { return n <= 1 ? 0 : 1 + ceil_log2((n + 1) / 2); }
// Longest fp32 summation path of a unit's log-sum-exp partial, one addition
// per stage aside: the pairwise tree of a vector's element pairs (up to 4),
// the chain over the chunk's vectors, the x + y of the packed pair, the warp
// sum and the sequential sum over the consumer warps.
constexpr int kLseSumDepth = 2 + (kVecsPerThread - 1) + 1 + 5 + (kConsumerWarps - 1);
constexpr int kMaxK = 32;
constexpr int kMaxN = 64;
constexpr double kFlagEps = 1e-9;                 // near-threshold window

// Random-number streams.
enum : uint32_t { kAccept = 1, kSample = 2, kDraft = 3, kTree = 4 };

// Row work modes (bit set).  M_MAX keeps the row max without its index.
enum : int { M_ARGMAX = 1, M_LSE = 2, M_LSE2 = 4, M_GUMBEL = 8, M_MAX = 16 };

// Entry-point kinds.
enum : int { K_GREEDY = 0, K_SAMPLE = 1, K_TREE = 2, K_PACKED = 3, K_SPOT = 4, K_ANYORDER = 5 };
constexpr int kMaxL = 32;  // SPOT: positions per block state (one lane each)

// ---------------------------------------------------------------------------
// Counter-based random numbers, written from the published definition of
// SplitMix64 (Steele, Lea & Flood): its output function, and its stream
// (output n + 1 of the generator seeded with s is the output function of
// s + n * 0x9E3779B97F4A7C15).
//   key(seed, stream, seq, pos, iter): fold each field into a running 64-bit
//     state through the output function.
//   The uniforms of a row are read from the stream seeded with the row key
//   (the layout is described in sv_gumbel.cuh).
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ uint64_t splitmix_out(uint64_t state)
{
    uint64_t z = state + 0x9E3779B97F4A7C15ull;
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z;
}

__host__ __device__ __forceinline__ uint64_t rng_key(uint64_t seed, uint32_t stream, uint64_t seq,
                                                     int64_t pos, uint64_t iter)
{
    uint64_t s = splitmix_out(seed);
    s = splitmix_out(s ^ (uint64_t)stream);
    s = splitmix_out(s ^ seq);
    s = splitmix_out(s ^ (uint64_t)pos);
    return splitmix_out(s ^ iter);
}

// ---------------------------------------------------------------------------
// Error latch: the first non-OK status wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void latch(int *err, int code)
{
    atomicCAS(err, 0, code);
}

// Spin limits (iterations); every wait in libsv is bounded.
constexpr uint32_t kSpinLimit = 1u << 24;

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy wrappers (sm_90+ PTX).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Non-blocking test of a phase.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait of at most `limit` tries; returns false when the limit
// expired.
__device__ __forceinline__ bool mbar_wait_n(uint64_t *bar, uint32_t parity, uint32_t limit)
{
    for (uint32_t i = 0; i < limit; ++i) {
        if (mbar_try(bar, parity))
            return true;
        if (SV_SPIN_SLEEP_NS > 0 && i > 64)
            __nanosleep(SV_SPIN_SLEEP_NS);
    }
    return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    return mbar_wait_n(bar, parity, kSpinLimit);
}

// Bounded wait for a global word to leave the value `old` (the form of the
// grid barrier of the fp64 path), giving up after `limit` tries or when *ab
// is set; returns false when it gave up.
__device__ __forceinline__ bool spin_until_change(const volatile unsigned *word, unsigned old,
                                                  const volatile unsigned *ab, uint32_t limit)
{
    for (uint32_t it = 0; *word == old; ++it) {
        if ((ab && *ab) || it >= limit)
            return false;
        __nanosleep(256);
    }
    return true;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Asynchronous 4-byte copy from global to shared memory (both addresses
// 4-byte aligned), completed by cp_async_wait_all.
__device__ __forceinline__ void cp_async4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Programmatic dependent launch (sm_90+).  pdl_wait blocks until the kernel
// that precedes this one in the stream has completed and its writes are
// visible (a no-op for a kernel launched without the attribute); every
// kernel of the library calls it before it touches global memory.
// pdl_trigger lets the next kernel of the stream be scheduled early: its
// CTAs take SM resources as this kernel's CTAs exit and then wait in
// pdl_wait, which hides the launch gap.  A kernel triggers only once all its
// CTAs are running, so the next kernel can never take resources that this
// kernel's own CTAs still need.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}


// Fast 2^x (MUFU); relative error within 2^-21 over the range used here, which
// the error bounds below assume and a GPU test measures.
__device__ __forceinline__ float ex2f(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic: one instruction per pair).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
        " mov.b64 c, {%6, %7};\n fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 d;
    asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
        " add.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// 2^d for an integer-valued d <= 0, exactly (0 below the normal range).
__device__ __forceinline__ float pow2_int(float d)
{
    return d < -126.f ? 0.f : __int_as_float((127 + (int)d) << 23);
}

// ---------------------------------------------------------------------------
// Ordered encoding of floats for unsigned atomicMax.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f2ord(float f)
{
    uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord2f(uint32_t o)
{
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// ---------------------------------------------------------------------------
// Partial statistics of one unit (a contiguous part of one logit row).
// Log-sum-exps are kept as s = sum 2^fl(x c - e) with an integer-valued
// reference exponent e, so that moving a sum to another reference is an exact
// power-of-two scaling.
// ---------------------------------------------------------------------------
struct __align__(16) RowPart {
    float m;        // max logit of the part (modes that track it; else -inf)
    float e1, e2;   // reference exponents of s1, s2 (-inf: empty sum)
    float s1, s2;   // sum 2^fl(x c1 - e1), sum 2^fl(x c2 - e2)
    int amax;       // lowest id attaining m (argmax mode)
    // Gumbel candidates (see Cand2 in sv_gumbel.cuh)
    float ghi1, glo1, ghi2, glo2, ghi3;
    int gv1, gv2;
    float xd;       // logit at the row's draft token, if the unit holds it (else NaN)
    int pad[2];
};

// Merged per-row statistics kept for the later kernels.
struct __align__(16) RowStat {
    double L1;    // natural log-sum-exp of x / T (the row's temperature)
    double L2;    // log2 sum 2^(x c) with the fp32 factor c = fl32(log2(e) / T)
    float m;      // row max
    float eps;    // bound on the relative error of exp(L1) (fp32 path)
    int gidx;     // Gumbel-max winner
    int gflag;    // its near-tie flag
};

// Top-2 bookkeeping of exact Gumbel scores; ties go to the lower id.
struct Top2 {
    double s1, s2;
    int i1;
    __device__ __forceinline__ void init()
    {
        s1 = -INFINITY;
        s2 = -INFINITY;
        i1 = -1;
    }
    __device__ __forceinline__ void add(double s, int i)
    {
        if (s > s1 || (s == s1 && i1 >= 0 && i < i1) || i1 < 0) {
            if (i1 >= 0)
                s2 = fmax(s2, s1);
            s1 = s;
            i1 = i;
        } else {
            s2 = fmax(s2, s);
        }
    }
    __device__ __forceinline__ void merge(double os1, int oi1, double os2)
    {
        if (oi1 >= 0)
            add(os1, oi1);
        s2 = fmax(s2, os2);
    }
};

__device__ __forceinline__ void warp_top2(Top2 &t)
{
    for (int o = 16; o; o >>= 1) {
        double a = __shfl_xor_sync(0xFFFFFFFFu, t.s1, o);
        double c = __shfl_xor_sync(0xFFFFFFFFu, t.s2, o);
        int i = __shfl_xor_sync(0xFFFFFFFFu, t.i1, o);
        t.merge(a, i, c);
    }
}

// (value desc, index asc) argmax reduction over a warp.
__device__ __forceinline__ void warp_argmax(float &v, int &i)
{
    for (int o = 16; o; o >>= 1) {
        float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
        if (ov > v || (ov == v && (unsigned)oi < (unsigned)i)) {
            v = ov;
            i = oi;
        }
    }
}

__device__ __forceinline__ float warp_max(float v)
{
    for (int o = 16; o; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_min(float v)
{
    for (int o = 16; o; o >>= 1)
        v = fminf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v)
{
    for (int o = 16; o; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sumd(double v)
{
    for (int o = 16; o; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Element access of a 16-byte vector.
template <typename In>
struct VecTraits;
template <>
struct VecTraits<uint16_t> {  // bf16 bit patterns
    static constexpr int N = 8;
    static constexpr int P = 4;  // element pairs per vector (one 32-bit word each)
    __device__ __forceinline__ static float2 pair(const uint4 &q, int i)
    {
        const uint32_t w = i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w;
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
    __device__ __forceinline__ static uint4 neg_inf_vec()
    {
        return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
    __device__ __forceinline__ static void unpack(const uint4 &q, float (&f)[8])
    {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = __uint_as_float(w[j] << 16);
            f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static float load1(const void *row, int v)
    {
        uint16_t b = __ldg((const unsigned short *)row + v);
        return __uint_as_float((uint32_t)b << 16);
    }
    // Packed (bf16x2) max and min over the 8 elements; invalid vectors give
    // -inf / +inf.
    __device__ __forceinline__ static uint32_t pmax(const uint4 &q)
    {
        return bmax(bmax(q.x, q.y), bmax(q.z, q.w));
    }
    __device__ __forceinline__ static uint32_t pmin(const uint4 &q)
    {
        return bmin(bmin(q.x, q.y), bmin(q.z, q.w));
    }
    __device__ __forceinline__ static uint32_t bmax(uint32_t a, uint32_t b)
    {
        __nv_bfloat162 r = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&a),
                                   *reinterpret_cast<const __nv_bfloat162 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
    __device__ __forceinline__ static uint32_t bmin(uint32_t a, uint32_t b)
    {
        __nv_bfloat162 r = __hmin2(*reinterpret_cast<const __nv_bfloat162 *>(&a),
                                   *reinterpret_cast<const __nv_bfloat162 *>(&b));
        return *reinterpret_cast<uint32_t *>(&r);
    }
    static constexpr uint32_t kNegInf = 0xFF80FF80u, kPosInf = 0x7F807F80u;
    // element i (run-time index) of the vector, without local memory
    __device__ __forceinline__ static float elem(const uint4 &q, int i)
    {
        uint32_t w = (i < 2) ? q.x : (i < 4) ? q.y : (i < 6) ? q.z : q.w;
        return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
    // the raw data of group g (elements 4g .. 4g+3) in the first half of a vector
    __device__ __forceinline__ static uint4 group_data(const uint4 &q, int g)
    {
        return g == 0 ? make_uint4(q.x, q.y, 0u, 0u) : make_uint4(q.z, q.w, 0u, 0u);
    }
    // element e (run-time index) of group data
    __device__ __forceinline__ static float gelem(const uint4 &d, int e)
    {
        const uint32_t w = (e < 2) ? d.x : d.y;
        return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
    // largest of the 4 elements of group g (elements 4g .. 4g+3)
    __device__ __forceinline__ static float group_max(const uint4 &q, int g)
    {
        uint32_t p = g == 0 ? bmax(q.x, q.y) : bmax(q.z, q.w);
        return fmaxf(__uint_as_float(p << 16), __uint_as_float(p & 0xFFFF0000u));
    }
    __device__ __forceinline__ static float hi_of(uint32_t p)
    {
        return fmaxf(__uint_as_float(p << 16), __uint_as_float(p & 0xFFFF0000u));
    }
    __device__ __forceinline__ static float lo_of(uint32_t p)
    {
        return fminf(__uint_as_float(p << 16), __uint_as_float(p & 0xFFFF0000u));
    }
};
template <>
struct VecTraits<float> {
    static constexpr int N = 4;
    static constexpr int P = 2;
    __device__ __forceinline__ static float2 pair(const uint4 &q, int i)
    {
        return i == 0 ? make_float2(__uint_as_float(q.x), __uint_as_float(q.y))
                      : make_float2(__uint_as_float(q.z), __uint_as_float(q.w));
    }
    __device__ __forceinline__ static uint4 neg_inf_vec()
    {
        return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
    }
    __device__ __forceinline__ static void unpack(const uint4 &q, float (&f)[4])
    {
        f[0] = __uint_as_float(q.x);
        f[1] = __uint_as_float(q.y);
        f[2] = __uint_as_float(q.z);
        f[3] = __uint_as_float(q.w);
    }
    __device__ __forceinline__ static float load1(const void *row, int v)
    {
        return __ldg((const float *)row + v);
    }
    __device__ __forceinline__ static uint32_t pmax(const uint4 &q)
    {
        return __float_as_uint(fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                                     fmaxf(__uint_as_float(q.z), __uint_as_float(q.w))));
    }
    __device__ __forceinline__ static uint32_t pmin(const uint4 &q)
    {
        return __float_as_uint(fminf(fminf(__uint_as_float(q.x), __uint_as_float(q.y)),
                                     fminf(__uint_as_float(q.z), __uint_as_float(q.w))));
    }
    __device__ __forceinline__ static uint32_t bmax(uint32_t a, uint32_t b)
    {
        return __float_as_uint(fmaxf(__uint_as_float(a), __uint_as_float(b)));
    }
    __device__ __forceinline__ static uint32_t bmin(uint32_t a, uint32_t b)
    {
        return __float_as_uint(fminf(__uint_as_float(a), __uint_as_float(b)));
    }
    static constexpr uint32_t kNegInf = 0xFF800000u, kPosInf = 0x7F800000u;
    __device__ __forceinline__ static float group_max(const uint4 &q, int)
    {
        return __uint_as_float(pmax(q));
    }
    __device__ __forceinline__ static float elem(const uint4 &q, int i)
    {
        return __uint_as_float((i == 0) ? q.x : (i == 1) ? q.y : (i == 2) ? q.z : q.w);
    }
    __device__ __forceinline__ static uint4 group_data(const uint4 &q, int) { return q; }
    __device__ __forceinline__ static float gelem(const uint4 &d, int e) { return elem(d, e); }
    __device__ __forceinline__ static float hi_of(uint32_t p) { return __uint_as_float(p); }
    __device__ __forceinline__ static float lo_of(uint32_t p) { return __uint_as_float(p); }
};

// Relative error bounds of exp(L) for a row log-sum-exp L computed in fp32.
//
// Streaming kernel.  Terms are t = 2^fl(x c - e), one FFMA and one ex2 each,
// with an integer reference e; a chunk whose max would give a term of 2^20
// or more first moves the reference up, so every exponent a = x c - e stays
// below kLseCap + 1.
// Moves between references are exact powers of two.  With c = fl32(c*),
// c* = log2(e)/T, the row's value is reported as E c*/c + log2 S (E the
// reference of S), which leaves per term an exponent error of at most
// 2^-24 |a| from the FFMA and 2^-24 |a| from c.  The row max has a >= -1, so
// S >= 1/2, and with n terms:
//   terms with a >= -24:       2^-21 (ex2) + 2 ln2 2^-24 max(kLseCap + 1, 24)
//   terms with -48 <= a < -24: total weight <= n 2^-24, each off by at most
//                              2^-21 + 2 ln2 2^-24 48
//   terms with a < -48:        total weight <= n 2^-48
// plus 2^-24 per fp32 addition on the longest summation path (depth), and
// one 2^-21 of slack.
constexpr float kLseCap = 20.f;
__host__ __device__ __forceinline__ double lse_rel_bound_stream(double n, double depth)
{
    const double u = 0x1p-24, ln2 = 0.6931471805599453;
    const double near = 0x1p-21 + 2.0 * ln2 * u * 24.0;  // kLseCap + 1 <= 24
    const double mid = 0x1p-21 + 2.0 * ln2 * u * 48.0;
    return 2.0 * 0x1p-21 + near + 2.0 * n * u * mid + 2.0 * n * 0x1p-48 + 1.01 * depth * u;
}
// Row passes that subtract first (terms 2^((x - m_ref) c)): exponent rounding
// of 3 ulps of |t| <= R.
__host__ __device__ __forceinline__ double lse_rel_bound(double range_c)
{
    return 3.0 * 0x1p-21 + 3.0 * 0.6931471805599453 * 0x1p-24 * range_c + 64.0 * 0x1p-24;
}

}  // namespace sv
