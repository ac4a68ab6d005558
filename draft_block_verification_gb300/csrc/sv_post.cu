// sv_post.cu -- the kernels that run after the streaming pass:
//   tv_kernel     total variation 1 - sum_v min(p_v, q_v) of every (p, q) row
//                 pair ([TwoTrade] eq. 1), a second pass over both rows;
//   resid_kernel  the correction drawn from the residual [p - q]_+ at the
//                 first rejection ([PackedSS] Alg. 2 line 7; [SPOT] App. B
//                 eq. 14), a second pass over one row pair per sequence;
//   rescue_kernel the fp64 path for the rare sequences whose fp32 decisions
//                 fell inside their error bound.
#include <math.h>
#include <stddef.h>

#include "sv_resid.cuh"

namespace sv {

constexpr int kPostThreads = 256;
constexpr int kPostWarps = kPostThreads / 32;
constexpr int kResidChunks = 8;     // chunks per residual row pair on the fp64 path
constexpr int kRescueChunks = 16;   // chunks per row on the fp64 path
constexpr int kMaxPairs = 32;
constexpr int kLoadsAhead = 4;      // vectors per row each thread loads before using them

struct PostShared {
    float f[kPostWarps][4];
    double d[kPostWarps][4];
    int i[kPostWarps][2];
    uint32_t thr;
    unsigned item;
    int flag;
};

// ---------------------------------------------------------------------------
// Block reductions (all threads of the block call them).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_max(float v, PostShared &sm)
{
    v = warp_max(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sm.f[threadIdx.x >> 5][0] = v;
    __syncthreads();
    float r = -INFINITY;
    for (int w = 0; w < kPostWarps; ++w) r = fmaxf(r, sm.f[w][0]);
    return r;
}
__device__ __forceinline__ float block_min(float v, PostShared &sm)
{
    v = warp_min(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sm.f[threadIdx.x >> 5][1] = v;
    __syncthreads();
    float r = INFINITY;
    for (int w = 0; w < kPostWarps; ++w) r = fminf(r, sm.f[w][1]);
    return r;
}
__device__ __forceinline__ float block_sum(float v, PostShared &sm)
{
    v = warp_sum(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sm.f[threadIdx.x >> 5][2] = v;
    __syncthreads();
    float r = 0.f;
    for (int w = 0; w < kPostWarps; ++w) r += sm.f[w][2];
    return r;
}
__device__ __forceinline__ double block_sumd(double v, PostShared &sm)
{
    v = warp_sumd(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sm.d[threadIdx.x >> 5][0] = v;
    __syncthreads();
    double r = 0.0;
    for (int w = 0; w < kPostWarps; ++w) r += sm.d[w][0];
    return r;
}

// Streaming 16-byte load.  Volatile so that the compiler keeps a batch of
// them ahead of their uses (memory-level parallelism) instead of sinking each
// load to its first use.
template <typename In>
__device__ __forceinline__ uint4 ldv(const char *row, int k)
{
    uint4 r;
    asm volatile("ld.global.cs.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(reinterpret_cast<const uint4 *>(row) + k));
    return r;
}

__device__ __forceinline__ int chunk_lo(int nvec, int c, int nc) { return (int)((int64_t)nvec * c / nc); }

// ---------------------------------------------------------------------------
// fp32 log-sum-exp partial of vectors [vb, ve) of one row (same arithmetic and
// error model as the streaming kernel): returns max, min and
// sum 2^((x - max) c).
// ---------------------------------------------------------------------------
template <typename In>
__device__ void lse_chunk32(const char *row, int vb, int ve, float c, PostShared &sm, float &M,
                            float &S, float &mn)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    float mref = -INFINITY, acc = 0.f, mx = -INFINITY, lo = INFINITY;
    for (int k0 = vb + threadIdx.x; k0 < ve; k0 += kLoadsAhead * blockDim.x) {
      uint4 qv[kLoadsAhead];
#pragma unroll
      for (int u = 0; u < kLoadsAhead; ++u) {
        const int k = k0 + u * blockDim.x;
        qv[u] = k < ve ? ldv<In>(row, k) : VT::neg_inf_vec();
      }
#pragma unroll
      for (int u = 0; u < kLoadsAhead; ++u) {
        if (k0 + u * (int)blockDim.x >= ve)
            break;
        float f[E];
        VT::unpack(qv[u], f);
        float cm = -INFINITY;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            cm = fmaxf(cm, f[e]);
            lo = fminf(lo, f[e]);
        }
        mx = fmaxf(mx, cm);
        if (mref == -INFINITY) {
            mref = cm;
        } else if ((cm - mref) * c > 64.f) {
            acc *= ex2f((mref - cm) * c);
            mref = cm;
        }
        float t[E];
#pragma unroll
        for (int e = 0; e < E; ++e) t[e] = ex2f((f[e] - mref) * c);
#pragma unroll
        for (int w = E / 2; w >= 1; w >>= 1)
#pragma unroll
            for (int e = 0; e < w; ++e) t[e] += t[e + w];
        acc += t[0];
      }
    }
    M = block_max(mx, sm);
    mn = block_min(lo, sm);
    float mine = (mref > -INFINITY) ? acc * ex2f((mref - M) * c) : 0.f;
    S = block_sum(mine, sm);
}

// ---------------------------------------------------------------------------
// Total variation.
// ---------------------------------------------------------------------------
template <typename In>
__global__ void __launch_bounds__(kPostThreads) tv_kernel(const __grid_constant__ Job j)
{
    __shared__ PostShared sm;
    pdl_wait();
    pdl_trigger();
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    const int TC = j.tv_chunks;
    const unsigned items = (unsigned)j.B * j.K * TC;
    for (;;) {
        if (threadIdx.x == 0) sm.item = atomicAdd(j.ctl + C_TWORK, 1u);
        __syncthreads();
        unsigned it = sm.item;
        __syncthreads();
        if (it >= items) break;
        int pair = it / TC, c = it - pair * TC;
        int b = pair / j.K, i = pair - b * j.K;
        if (i >= clamp_len(j, b)) continue;
        const RowStat sp = j.rs_stat[(int64_t)b * j.rows_per_seq + i];
        const RowStat sq = j.rs_stat[(int64_t)b * j.rows_per_seq + j.K + 1 + i];
        const float lgp = (float)sp.L2, lgq = (float)sq.L2;
        const char *prow = slot_row(j, b, i), *qrow = slot_row(j, b, j.K + 1 + i);
        int vb = chunk_lo(j.nvec, c, TC), ve = chunk_lo(j.nvec, c + 1, TC);
        float acc = 0.f;
        // several vectors of both rows in flight per thread before any use
        for (int k0 = vb + threadIdx.x; k0 < ve; k0 += kLoadsAhead * blockDim.x) {
            uint4 px[kLoadsAhead], qy[kLoadsAhead];
#pragma unroll
            for (int u = 0; u < kLoadsAhead; ++u) {
                const int k = k0 + u * blockDim.x;
                px[u] = k < ve ? ldv<In>(prow, k) : VT::neg_inf_vec();
                qy[u] = k < ve ? ldv<In>(qrow, k) : VT::neg_inf_vec();
            }
#pragma unroll
            for (int u = 0; u < kLoadsAhead; ++u) {
                float x[E], y[E];
                VT::unpack(px[u], x);
                VT::unpack(qy[u], y);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    float fa = fmaf(x[e], j.cp, -lgp);  // log2 p_v
                    float fb = fmaf(y[e], j.cq, -lgq);  // log2 q_v
                    acc += ex2f(fminf(fa, fb));         // -inf padding adds 0
                }
            }
        }
        float s = block_sum(acc, sm);
        if (threadIdx.x == 0) {
            j.tvpart[(int64_t)pair * TC + c] = s;
            __threadfence();
            unsigned old = atomicAdd(j.tvdone + pair, 1u);
            if (old + 1u == (unsigned)TC) {
                __threadfence();
                double S = 0.0;
                for (int q = 0; q < TC; ++q) S += (double)__ldcg(j.tvpart + (int64_t)pair * TC + q);
                j.tv[(int64_t)b * j.K + i] = (float)(1.0 - S);
                j.tvdone[pair] = 0u;
            }
        }
    }
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(j.ctl + C_TEXIT, 1u) + 1u == gridDim.x) {
            j.ctl[C_TWORK] = 0u;
            j.ctl[C_TEXIT] = 0u;
            __threadfence();
        }
    }
}

// ---------------------------------------------------------------------------
// Residual draws (the scores and their intervals are in sv_resid.cuh): one
// row pair per sequence that rejected.  The fast path (resid_kernel, below)
// gives each pair one CTA; the fp64 path scans a pair in chunks on different
// CTAs (resid_scan with the fp64 tracker) and merges them after a grid
// barrier.  Packed-SS calls first need the stored proposal row's
// log-sum-exp.
// ---------------------------------------------------------------------------
struct RBest {  // fp64-interval tracker of the fp64 path
    double lo, hi, hio;
    int i;
    __device__ __forceinline__ void init()
    {
        lo = -INFINITY;
        hi = -INFINITY;
        hio = -INFINITY;
        i = -1;
    }
    __device__ __forceinline__ void add(double l, double h, int v)
    {
        if (i < 0 || l > lo || (l == lo && v < i)) {
            if (i >= 0) hio = fmax(hio, hi);
            lo = l;
            hi = h;
            i = v;
        } else {
            hio = fmax(hio, h);
        }
    }
    __device__ __forceinline__ void merge(const RBest &o)
    {
        hio = fmax(hio, o.hio);
        if (o.i >= 0) add(o.lo, o.hi, o.i);
    }
};

// fp64-interval candidate tracker of the fp64 path.
struct Track64 {
    RBest r;
    float lomax, thr, thrS;
    __device__ __forceinline__ void init()
    {
        r.init();
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
        double lo, hi;
        if (!resid_interval64(ctx, x, y, m, top, lo, hi)) return;
        r.add(lo, hi, (int)v);
        if (lo > -INFINITY && (float)lo > lomax) {
            lomax = __double2float_rd(lo);
            raise(__double2float_rd(lo - kFlagEps - (fabs(lo) + 41.0) * 0x1p-21));
        }
    }
};

__device__ __forceinline__ void block_rbest(RBest &r, PostShared &sm, RBest &out)
{
    for (int o = 16; o; o >>= 1) {
        RBest q;
        q.lo = __shfl_xor_sync(0xFFFFFFFFu, r.lo, o);
        q.hi = __shfl_xor_sync(0xFFFFFFFFu, r.hi, o);
        q.hio = __shfl_xor_sync(0xFFFFFFFFu, r.hio, o);
        q.i = __shfl_xor_sync(0xFFFFFFFFu, r.i, o);
        r.merge(q);
    }
    __syncthreads();
    int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        sm.d[w][0] = r.lo;
        sm.d[w][1] = r.hi;
        sm.d[w][2] = r.hio;
        sm.i[w][0] = r.i;
    }
    __syncthreads();
    out.init();
    for (int q = 0; q < kPostWarps; ++q) {
        RBest t;
        t.lo = sm.d[q][0];
        t.hi = sm.d[q][1];
        t.hio = sm.d[q][2];
        t.i = sm.i[q][0];
        out.merge(t);
    }
}


// Seed of a scan over vectors [vb, ve): the CTA scores every top id of the
// range (a couple of skip draws per block of 256 ids) and shares the best
// lower end as the threshold.
template <typename In, typename Tr>
__device__ __forceinline__ void resid_seed(const RCtx &c, int vb, int ve, const uint64_t *skip,
                                           PostShared &sm, Tr &tr)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    if (threadIdx.x == 0) sm.thr = f2ord(-INFINITY);
    __syncthreads();
    seed_top_ids<In>(c, (uint32_t)vb * E, (uint32_t)ve * E, skip, (int)threadIdx.x,
                     (int)blockDim.x, tr);
    atomicMax(&sm.thr, f2ord(tr.thr));
    __syncthreads();
    tr.raise(ord2f(sm.thr));
}

// Scan vectors [vb, ve) of the pair (the fp64 path's chunks).  Seed: the CTA
// scores every top id of the chunk first (a couple of skip draws per block of
// 256 ids), which sets a threshold close to the chunk's best; then each
// vector whose largest logit can reach it with the ordinary-id bound is
// screened per id.  (Scores drop the common -Lp, and log w <= x/T - Lp, so
// x/T + G bounds a score.)
template <typename In, typename Tr>
__device__ void resid_scan(const RCtx &c, int vb, int ve, const float *gt, const uint64_t *skip,
                           PostShared &sm, Tr &tr)
{
    using VT = VecTraits<In>;
    tr.init();
    resid_seed<In>(c, vb, ve, skip, sm, tr);
    const float gmax = gt[kGTab - 1];
    float pub = tr.thr;
    for (int k0 = vb + threadIdx.x; k0 < ve; k0 += kLoadsAhead * blockDim.x) {
        uint4 px[kLoadsAhead];
#pragma unroll
        for (int u = 0; u < kLoadsAhead; ++u) {
            const int k = k0 + u * blockDim.x;
            px[u] = k < ve ? ldv<In>(c.prow, k) : VT::neg_inf_vec();
        }
        tr.raise(ord2f(*(volatile uint32_t *)&sm.thr));
#pragma unroll
        for (int u = 0; u < kLoadsAhead; ++u) {
            const int k = k0 + u * blockDim.x;
            if (k >= ve)
                break;
            if (fmaf(VT::hi_of(VT::pmax(px[u])), c.invTp, gmax) >= tr.thrS)
                resid_vector<In>(c, px[u], ldv<In>(c.qrow, k), k, gt, skip, tr);
        }
        if (tr.thr > pub) {
            atomicMax(&sm.thr, f2ord(tr.thr));
            pub = tr.thr;
        }
    }
}

// ---------------------------------------------------------------------------
// The residual pass: one CTA of NT threads per residual entry scans the
// entry's whole row pair, so no CTA waits for another: the row's top ids set
// one threshold for the whole row, and the candidates are merged inside the
// CTA.  NT = 1024 (one CTA per SM) when there are at most as many sequences as
// SMs, else 512 (two CTAs per SM), so that up to twice as many sequences are
// drawn in one wave.
// ---------------------------------------------------------------------------
constexpr int kRQ = 64;        // vectors per warp queued for the per-id screen
constexpr int kScanAhead = 8;  // vectors per thread loaded together
constexpr int kSeedPer = 2;    // listed top ids each thread scores from registers

template <int NT>
struct ResidShared {
    static constexpr int W = NT / 32;
    int qv[W][kRQ];                // queued vectors (row vector index) per warp
    uint32_t ids[kSeedPer * NT];   // top ids of the row
    int nids;
    uint32_t thr;                  // the CTA's Gumbel threshold (ordered float)
    float f[W][5];                 // block reductions
    int iv[W][2];
    double Lq, epsq;               // Packed-SS: the proposal row's log-sum-exp
};

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// fp32 log-sum-exp of a whole row with the CTA (the arithmetic and error
// model of lse_chunk32): max, min and sum 2^((x - max) c).
template <typename In, int NT>
__device__ void resid_lse32(const char *row, int nvec, float c, ResidShared<NT> &rs, float &M,
                            float &S, float &mn)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    float mref = -INFINITY, acc = 0.f, mx = -INFINITY, lo = INFINITY;
    for (int base = 0; base < nvec; base += kScanAhead * NT) {
        uint4 qv[kScanAhead];
#pragma unroll
        for (int u = 0; u < kScanAhead; ++u) {
            const int k = base + t + u * NT;
            qv[u] = k < nvec ? ldv<In>(row, k) : VT::neg_inf_vec();
        }
#pragma unroll
        for (int u = 0; u < kScanAhead; ++u) {
            float f[E];
            VT::unpack(qv[u], f);
            float cm = -INFINITY, cl = INFINITY;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                cm = fmaxf(cm, f[e]);
                cl = fminf(cl, f[e]);
            }
            if (cm == -INFINITY)
                continue;  // past the end of the row
            lo = fminf(lo, cl);
            mx = fmaxf(mx, cm);
            if (mref == -INFINITY) {
                mref = cm;
            } else if ((cm - mref) * c > 64.f) {
                acc *= ex2f((mref - cm) * c);
                mref = cm;
            }
            float tt[E];
#pragma unroll
            for (int e = 0; e < E; ++e) tt[e] = ex2f((f[e] - mref) * c);
#pragma unroll
            for (int h = E / 2; h >= 1; h >>= 1)
#pragma unroll
                for (int e = 0; e < h; ++e) tt[e] += tt[e + h];
            acc += tt[0];
        }
    }
    const float wm = warp_max(mx), wl = warp_min(lo);
    if (lane == 0) {
        rs.f[w][0] = wm;
        rs.f[w][1] = wl;
    }
    __syncthreads();
    float bm = -INFINITY, bl = INFINITY;
    for (int q = 0; q < (NT / 32); ++q) {
        bm = fmaxf(bm, rs.f[q][0]);
        bl = fminf(bl, rs.f[q][1]);
    }
    const float mine = (mref > -INFINITY) ? acc * ex2f((mref - bm) * c) : 0.f;
    const float ws = warp_sum(mine);
    __syncthreads();
    if (lane == 0) rs.f[w][2] = ws;
    __syncthreads();
    float bs = 0.f;
    for (int q = 0; q < (NT / 32); ++q) bs += rs.f[q][2];
    M = bm;
    S = bs;
    mn = bl;
}

// Scores every top id of ids [0, V) into tr.  First the CTA lists them in
// shared memory (threads take blocks of 256 ids in turn: a couple of skip
// draws each); then each thread loads the logits of its share of the list at
// once, into registers, and scores them, so a thread waits for one round of
// loads.  Ids past the list's capacity (far beyond the expected V/256) are
// scored where they are found.
template <typename In, int NT>
__device__ __forceinline__ void seed_row(const RCtx &c, uint32_t V, const uint64_t *skip,
                                         ResidShared<NT> &rs, Track32 &tr)
{
    using VT = VecTraits<In>;
    const int t = threadIdx.x;
    const uint32_t nb = (V + 255u) >> 8;
    for (uint32_t beta = (uint32_t)t; beta < nb; beta += NT) {
        int pos = -1;
        for (int i = 0; i < kSkipN; ++i) {
            pos = next_top(c.key, beta, i, pos, skip);
            const uint32_t v = beta * 256u + (uint32_t)pos;
            if (pos > 255 || v >= V)
                break;
            const int slot = atomicAdd(&rs.nids, 1);
            if (slot < (kSeedPer * NT))
                rs.ids[slot] = v;
            else
                tr.add(c, VT::load1(c.prow, (int)v), VT::load1(c.qrow, (int)v), v,
                       fine52(c.key, v), true);
        }
    }
    __syncthreads();
    const int n = min(rs.nids, (kSeedPer * NT));
    uint32_t id[kSeedPer];
    float x[kSeedPer], y[kSeedPer];
#pragma unroll
    for (int r = 0; r < kSeedPer; ++r) {
        const int i = t + r * NT;
        id[r] = i < n ? rs.ids[i] : 0xFFFFFFFFu;
        x[r] = y[r] = 0.f;
        if (i < n) {
            x[r] = VT::load1(c.prow, (int)id[r]);
            y[r] = VT::load1(c.qrow, (int)id[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < kSeedPer; ++r)
        if (id[r] != 0xFFFFFFFFu)
            tr.add(c, x[r], y[r], id[r], fine52(c.key, id[r]), true);
}

// Per-id screen of a warp's queued vectors, one vector per lane.
template <typename In, int NT>
__device__ __forceinline__ void resid_flush(const RCtx &c, const ResidShared<NT> &rs, int n,
                                            const float *gt, const uint64_t *skip, Track32 &tr)
{
    const int w = threadIdx.x >> 5;
    __syncwarp();
    for (int i = (int)(threadIdx.x & 31); i < n; i += 32) {
        const int k = rs.qv[w][i];
        resid_vector<In>(c, ldv<In>(c.prow, k), ldv<In>(c.qrow, k), k, gt, skip, tr);
    }
    __syncwarp();
}

// The warp's best threshold into the CTA's word, when it beats what the
// warp published before.
template <int NT>
__device__ __forceinline__ void publish_thr(const Track32 &tr, ResidShared<NT> &rs, uint32_t &pub)
{
    const uint32_t w = __reduce_max_sync(0xFFFFFFFFu, f2ord(tr.thr));
    if (w > pub) {
        if ((threadIdx.x & 31) == 0) atomicMax(&rs.thr, w);
        pub = w;
    }
}

// Gumbel-max over the residual scores of the whole row pair (the row was
// prefetched into L2 by the caller while the CTA scores the row's top ids).
// A vector whose largest logit can reach the threshold with the ordinary-id
// bound is queued (compacted with a ballot) and the queue is screened per id
// with a vector per lane, so a warp does not diverge per vector.
template <typename In, int NT>
__device__ void resid_scan_row(const RCtx &c, int nvec, uint32_t V, const float *gt,
                               const uint64_t *skip, ResidShared<NT> &rs, Track32 &tr)
{
    using VT = VecTraits<In>;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    tr.init();
    seed_row<In, NT>(c, V, skip, rs, tr);
    uint32_t pub = 0u;
    publish_thr(tr, rs, pub);
    __syncthreads();
    const float gmax = gt[kGTab - 1];
    int qn = 0;
    for (int base = 0; base < nvec; base += kScanAhead * NT) {
        uint4 px[kScanAhead];
#pragma unroll
        for (int u = 0; u < kScanAhead; ++u) {
            const int k = base + t + u * NT;
            px[u] = k < nvec ? ldv<In>(c.prow, k) : VT::neg_inf_vec();
        }
        tr.raise(ord2f(*(volatile uint32_t *)&rs.thr));
#pragma unroll
        for (int u = 0; u < kScanAhead; ++u) {
            const int k = base + t + u * NT;
            // (k < nvec: past the row's end there is no vector, and with no
            // threshold yet a -inf bound would still compare >= -inf)
            const bool pass =
                k < nvec && fmaf(VT::hi_of(VT::pmax(px[u])), c.invTp, gmax) >= tr.thrS;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, pass);
            if (bal) {
                if (pass) rs.qv[w][qn + __popc(bal & ((1u << lane) - 1u))] = k;
                qn += __popc(bal);
                if (qn > kRQ - 32) {
                    resid_flush<In, NT>(c, rs, qn, gt, skip, tr);
                    qn = 0;
                    tr.raise(ord2f(*(volatile uint32_t *)&rs.thr));
                }
            }
        }
        publish_thr(tr, rs, pub);
    }
    if (qn) resid_flush<In, NT>(c, rs, qn, gt, skip, tr);
}

// The CTA's merged candidates, in thread 0's `out`.
template <int NT>
__device__ __forceinline__ void resid_cand2(Cand2 &c, ResidShared<NT> &rs, Cand2 &out)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    warp_cand2(c);
    if (lane == 0) {
        rs.f[w][0] = c.hi1;
        rs.f[w][1] = c.lo1;
        rs.f[w][2] = c.hi2;
        rs.f[w][3] = c.lo2;
        rs.f[w][4] = c.hi3;
        rs.iv[w][0] = c.v1;
        rs.iv[w][1] = c.v2;
    }
    __syncthreads();
    out.init();
    if (w == 0) {
        if (lane < (NT / 32)) {
            out.hi1 = rs.f[lane][0];
            out.lo1 = rs.f[lane][1];
            out.hi2 = rs.f[lane][2];
            out.lo2 = rs.f[lane][3];
            out.hi3 = rs.f[lane][4];
            out.v1 = rs.iv[lane][0];
            out.v2 = rs.iv[lane][1];
        }
        warp_cand2(out);
    }
}

template <typename In, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) resid_kernel(const __grid_constant__ Job j)
{
    __shared__ ResidShared<NT> rs;
    __shared__ float gt[kGTab];
    __shared__ uint64_t skip[kSkipN];  // skip thresholds of the top-id draws
    const int t = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    const unsigned nE = *(volatile unsigned *)(j.ctl + C_RESID_N);
    if (blockIdx.x < nE) {
        for (int i = t; i < kGTab; i += NT)
            gt[i] = __ldg(j.gtab + i);
        for (int i = t; i < kSkipN; i += NT)
            skip[i] = __ldg(j.skip + i);
    }
    for (unsigned e = blockIdx.x; e < nE; e += gridDim.x) {
        ResidEntry re = j.resid[e];
        if (t == 0) {
            // the p row streams whole; the q row is read only where a
            // candidate needs it (or whole, for a Packed-SS log-sum-exp)
            prefetch_l2(re.prow, (uint32_t)j.nvec * 16u);
            if (re.need_lq) prefetch_l2(re.qrow, (uint32_t)j.nvec * 16u);
            rs.nids = 0;
            rs.thr = f2ord(-INFINITY);
        }
        __syncthreads();
        if (re.need_lq) {
            // Packed-SS: the stored proposal row's log-sum-exp.
            float M, S, mn;
            resid_lse32<In, NT>(re.qrow, j.nvec, j.cp, rs, M, S, mn);
            if (t == 0) {
                rs.Lq = (double)M / (double)j.Tp + log((double)S);
                rs.epsq = lse_rel_bound(((double)M - (double)mn) * (double)j.cp);
            }
            __syncthreads();
            re.Lq = rs.Lq;
            re.epsq = rs.epsq;
        }
        RCtx ctx;
        resid_ctx(j, re, ctx);
        Track32 tr;
        resid_scan_row<In, NT>(ctx, j.nvec, (uint32_t)j.V, gt, skip, rs, tr);
        Cand2 all;
        resid_cand2(tr.c, rs, all);
        if (t == 0) resid_resolve(j, re, ctx, all, skip);
        __syncthreads();  // rs is reused by the next entry
    }
    if (t == 0) {
        __threadfence();
        if (atomicAdd(j.ctl + C_REXIT, 1u) + 1u == gridDim.x) {
            j.ctl[C_REXIT] = 0u;
            j.ctl[C_RESID_N] = 0u;
            __threadfence();
        }
    }
}

// ---------------------------------------------------------------------------
// fp64 path.  A cooperative launch (every CTA resident) with bounded grid
// barriers between its phases:
//   1. fp64 log-sum-exp of every row pair the listed sequences need;
//   2. exact acceptance decisions, flags, and the position h of the
//      correction (one warp per sequence);
//   3. the residual draw at h with exact log-sum-exps;
//   4. outputs.
// ---------------------------------------------------------------------------
__device__ bool grid_sync(const Job &j)
{
    __syncthreads();
    int ok = 1;
    if (threadIdx.x == 0) {
        volatile unsigned *gen = j.ctl + C_GGEN;
        volatile unsigned *ab = j.ctl + C_ABORT;
        unsigned g = *gen;
        __threadfence();
        if (atomicAdd(j.ctl + C_GBAR, 1u) + 1u == gridDim.x) {
            j.ctl[C_GBAR] = 0u;
            __threadfence();
            atomicAdd(j.ctl + C_GGEN, 1u);
        } else if (!spin_until_change(gen, g, ab, kSpinLimit)) {
            latch(j.err, SV_ERR_TIMEOUT);
            atomicExch(j.ctl + C_ABORT, 1u);
            ok = 0;
        }
        __threadfence();
    }
    return __syncthreads_and(ok) != 0;
}

__device__ __forceinline__ double *lse64_rec(const Job &j, int e, int i, int r, int c)
{
    double *base = j.rpart + (int64_t)j.B * kResidChunks * 8;
    return base + ((((int64_t)e * kMaxPairs + i) * 2 + r) * kRescueChunks + c) * 2;
}
__device__ __forceinline__ double *res64_rec(const Job &j, int e, int c)
{
    double *base = j.rpart + (int64_t)j.B * kResidChunks * 8 +
                   (int64_t)j.B * kMaxPairs * 2 * kRescueChunks * 2;
    return base + ((int64_t)e * kResidChunks + c) * 4;
}

__device__ __forceinline__ const char *pair_row(const Job &j, int b, int i, int r)
{
    if (r == 0) return slot_row(j, b, i);
    if (j.kind == K_SAMPLE) return slot_row(j, b, j.K + 1 + i);
    int off = __ldg(j.prev_off + b);
    return j.src2 + ((int64_t)b * j.W + off + i) * j.rs;
}

// exact log-sum-exp of x / T over vectors [vb, ve): (max, sum exp((x - max)/T))
template <typename In>
__device__ void lse_chunk64(const char *row, int vb, int ve, double T, PostShared &sm, double &M,
                            double &S)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    float mx = -INFINITY;
    for (int k = vb + threadIdx.x; k < ve; k += blockDim.x) {
        float f[E];
        VT::unpack(ldv<In>(row, k), f);
#pragma unroll
        for (int e = 0; e < E; ++e) mx = fmaxf(mx, f[e]);
    }
    float m = block_max(mx, sm);
    double md = (double)m / T, s = 0.0;
    for (int k = vb + threadIdx.x; k < ve; k += blockDim.x) {
        float f[E];
        VT::unpack(ldv<In>(row, k), f);
#pragma unroll
        for (int e = 0; e < E; ++e) s += exp((double)f[e] / T - md);
    }
    M = md;
    S = block_sumd(s, sm);
}

__device__ double merge64(const Job &j, int e, int i, int r)
{
    double M = -INFINITY;
    for (int c = 0; c < kRescueChunks; ++c) M = fmax(M, __ldcg(lse64_rec(j, e, i, r, c)));
    double S = 0.0;
    for (int c = 0; c < kRescueChunks; ++c) {
        double *q = lse64_rec(j, e, i, r, c);
        S += __ldcg(q + 1) * exp(__ldcg(q) - M);
    }
    return M + log(S);
}

template <typename In>
__global__ void __launch_bounds__(kPostThreads) rescue_kernel(const __grid_constant__ Job j)
{
    __shared__ PostShared sm;
    __shared__ float gt[kGTab];
    // No pdl_trigger: the grid barriers below need every CTA of this grid
    // resident, so the next kernel is scheduled only once this one exits.
    pdl_wait();
    const unsigned nR = *(volatile unsigned *)(j.ctl + C_RESCUE_N);
    if (nR == 0u) return;
    for (int i = threadIdx.x; i < kGTab; i += blockDim.x)
        gt[i] = __ldg(j.gtab + i);
    __syncthreads();
    const double Tq = (j.kind == K_PACKED) ? (double)j.Tp : (double)j.Tq;

    // ---- phase 1: fp64 log-sum-exps ----
    const unsigned items1 = nR * kMaxPairs * 2 * kRescueChunks;
    for (unsigned it = blockIdx.x; it < items1; it += gridDim.x) {
        int c = it % kRescueChunks;
        int r = (it / kRescueChunks) % 2;
        int i = (it / (kRescueChunks * 2)) % kMaxPairs;
        int e = it / (kRescueChunks * 2 * kMaxPairs);
        RescueEntry re = j.rescue[e];
        if (re.kind == 1 && re.bonus) continue;  // a bonus draw needs no log-sum-exp
        int lo = (re.kind == 0) ? 0 : re.h;
        int hi = (re.kind == 0) ? clamp_len(j, re.b) : re.h + 1;
        if (i < lo || i >= hi) continue;
        double M, S;
        lse_chunk64<In>(pair_row(j, re.b, i, r), chunk_lo(j.nvec, c, kRescueChunks),
                        chunk_lo(j.nvec, c + 1, kRescueChunks), r == 0 ? (double)j.Tp : Tq, sm,
                        M, S);
        if (threadIdx.x == 0) {
            double *q = lse64_rec(j, e, i, r, c);
            q[0] = M;
            q[1] = S;
        }
    }
    if (!grid_sync(j)) return;

    // ---- phase 2: exact decisions (one warp per sequence) ----
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kPostWarps + (threadIdx.x >> 5);
    const int nw = gridDim.x * kPostWarps;
    for (unsigned e = gw; e < nR; e += nw) {
        RescueEntry re = j.rescue[e];
        const int b = re.b;
        const int n = clamp_len(j, b);
        const bool cactus = j.kind == K_SAMPLE && j.amode == SV_LENIENT_CACTUS;
        if (re.kind == 1 && re.bonus) {
            if (lane == 0) {
                j.rescue[e].resid = 1;
                j.rescue[e].flags = 0;
            }
            continue;
        }
        if (re.kind == 1) {
            if (lane == 0) {
                double Lp = merge64(j, e, re.h, 0);
                if (cactus) {
                    // the residual [c p - q]_+ is [p - q]_+ with Lp lowered by log c
                    const int d = __ldg(j.ids + (int64_t)b * j.K + re.h);
                    const double lp =
                        (double)load_logit(j, slot_row(j, b, re.h), d) / (double)j.Tp - Lp;
                    Lp -= cactus_log_scale64(lp, (double)j.lam);
                }
                j.rescue[e].Lp = Lp;
                j.rescue[e].Lq = merge64(j, e, re.h, 1);
                j.rescue[e].resid = 1;
                j.rescue[e].flags = 0;
            }
            continue;
        }
        const int64_t p0 = pos0_of(j, b);
        const int Ks = (j.kind == K_PACKED) ? j.K - 1 : j.K;
        bool acc = false, fl = false;
        double Lp = 0, Lq = 0, lc = 0.0;
        if (lane < n) {
            Lp = merge64(j, e, lane, 0);
            Lq = merge64(j, e, lane, 1);
            int d = __ldg(j.ids + (int64_t)b * Ks + lane);
            double lp = -INFINITY, lq;
            if (d >= 0 && d < j.V)
                lp = (double)load_logit(j, slot_row(j, b, lane), d) / (double)j.Tp - Lp;
            if (j.kind == K_PACKED) {
                lq = log((double)__ldg(j.prev_q + (int64_t)b * Ks + lane));
            } else {
                lq = (d >= 0 && d < j.V)
                         ? (double)load_logit(j, slot_row(j, b, j.K + 1 + lane), d) / Tq - Lq
                         : 0.0;
            }
            double alpha = alpha_exact(j.kind == K_PACKED ? SV_LOSSLESS : j.amode, lp, lq,
                                       (double)j.lam);
            if (cactus)
                lc = cactus_log_scale64(lp, (double)j.lam);
            double u = uniform_at(rng_key(j.seed, kAccept, (uint64_t)b, p0 + lane, 0), 0, j.skip);
            acc = u < alpha;
            fl = fabs(u - alpha) < kFlagEps;
        }
        unsigned am = __ballot_sync(0xFFFFFFFFu, acc);
        int h = (~am == 0u) ? 32 : __ffs(~am) - 1;
        h = min(h, n);
        unsigned reached = (h >= 31) ? 0xFFFFFFFFu : ((2u << h) - 1u);
        int nfl = __popc(__ballot_sync(0xFFFFFFFFu, fl) & reached);
        double Lph = __shfl_sync(0xFFFFFFFFu, Lp, h & 31);
        double Lqh = __shfl_sync(0xFFFFFFFFu, Lq, h & 31);
        Lph -= __shfl_sync(0xFFFFFFFFu, lc, h & 31);  // Cactus: the residual's scale c
        if (h < n) {
            if (lane == 0) {
                j.rescue[e].h = h;
                j.rescue[e].resid = 1;
                j.rescue[e].bonus = 0;
                j.rescue[e].Lp = Lph;
                j.rescue[e].Lq = Lqh;
                j.rescue[e].flags = nfl;
                if (j.kind == K_SAMPLE) j.acc[b] = h;
            }
            continue;
        }
        // every draft accepted: the bonus token, the Gumbel-max of row n,
        // drawn in fp64 by the residual phase below
        if (lane == 0) {
            j.rescue[e].h = n;
            j.rescue[e].resid = 1;
            j.rescue[e].bonus = 1;
            j.rescue[e].flags = nfl;
            if (j.kind == K_SAMPLE) j.acc[b] = n;
        }
    }
    if (!grid_sync(j)) return;

    // ---- phase 3: residual draws with exact log-sum-exps ----
    const unsigned items3 = nR * kResidChunks;
    for (unsigned it = blockIdx.x; it < items3; it += gridDim.x) {
        int e = it / kResidChunks, c = it % kResidChunks;
        RescueEntry re = j.rescue[e];
        if (!re.resid) continue;
        RCtx ctx;
        if (re.bonus) {
            const char *row = slot_row(j, re.b, re.h);
            fill_ctx(j, ctx, row, row, 0.0, 0.0);
            ctx.bonus = true;
        } else {
            double D = re.Lq - re.Lp;
            double eD = 1e-10 * (1.0 + fabs(re.Lp) + fabs(re.Lq));
            fill_ctx(j, ctx, pair_row(j, re.b, re.h, 0), pair_row(j, re.b, re.h, 1), D, eD);
        }
        ctx.key = rng_key(j.seed, kSample, (uint64_t)re.b, pos0_of(j, re.b) + re.h, 0);
        Track64 tr;
        resid_scan<In>(ctx, chunk_lo(j.nvec, c, kResidChunks),
                       chunk_lo(j.nvec, c + 1, kResidChunks), gt, j.skip, sm, tr);
        RBest best;
        block_rbest(tr.r, sm, best);
        if (threadIdx.x == 0) {
            double *q = res64_rec(j, e, c);
            q[0] = best.lo;
            q[1] = best.hi;
            q[2] = best.hio;
            q[3] = (double)best.i;
        }
    }
    if (!grid_sync(j)) return;

    // ---- phase 4: outputs ----
    for (unsigned e = gw; e < nR; e += nw) {
        RescueEntry re = j.rescue[e];
        if (!re.resid) continue;
        int c = -1, fl = 0;
        if (lane == 0) {
            RBest all;
            all.init();
            for (int q = 0; q < kResidChunks; ++q) {
                double *r = res64_rec(j, e, q);
                RBest t;
                t.lo = __ldcg(r + 0);
                t.hi = __ldcg(r + 1);
                t.hio = __ldcg(r + 2);
                t.i = (int)__ldcg(r + 3);
                all.merge(t);
            }
            c = all.i;
            fl = (all.lo - all.hio < kFlagEps) ? 1 : 0;
            if (c < 0) latch(j.err, SV_ERR_TIMEOUT);
        }
        c = __shfl_sync(0xFFFFFFFFu, c, 0);
        fl = __shfl_sync(0xFFFFFFFFu, fl, 0);
        if (j.kind == K_SAMPLE) {
            if (lane == 0) {
                j.acc[re.b] = re.h;
                j.next[re.b] = c;
                if (j.flags) j.flags[re.b] = re.flags + fl;
            }
        } else {
            packed_commit(j, re.b, re.h, c, true, re.flags + fl);
        }
    }
    if (!grid_sync(j)) return;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        j.ctl[C_RESCUED] += nR;
        j.ctl[C_RESCUE_N] = 0u;
        __threadfence();
    }
}

// Host-side launchers.
// Resident CTAs per SM of the total-variation kernel (occ[0], which takes
// work items from a counter, so its grid fills the GPU) and of the residual
// kernel's 512-thread instance (occ[1]; two per SM let the residual pass
// draw up to two sequences per SM in one wave).
cudaError_t post_setup(int occ[2])
{
    int a = 0, b = 0, c = 0, d = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, tv_kernel<uint16_t>,
                                                                  kPostThreads, 0);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, tv_kernel<float>, kPostThreads, 0);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c, resid_kernel<uint16_t, 512>, 512, 0);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d, resid_kernel<float, 512>, 512, 0);
    occ[0] = a < b ? a : b;
    occ[1] = c < d ? c : d;
    return e;
}

cudaError_t post_launch(const Job &j, int tv_grid, int resid_grid, int coop_grid, bool tv,
                        cudaStream_t s)
{
    const bool bf = j.dtype == SV_BF16;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    cudaError_t e;
    if (tv) {
        pdl_config(cfg, at, dim3(tv_grid), dim3(kPostThreads), 0, s);
        e = bf ? cudaLaunchKernelEx(&cfg, tv_kernel<uint16_t>, j)
               : cudaLaunchKernelEx(&cfg, tv_kernel<float>, j);
        if (e != cudaSuccess) return e;
    }
    // more sequences than SMs: two CTAs of 512 threads per SM
    const bool half = j.B > coop_grid && resid_grid > coop_grid;
    pdl_config(cfg, at, dim3(resid_grid), dim3(half ? 512 : 1024), 0, s);
    if (half)
        e = bf ? cudaLaunchKernelEx(&cfg, resid_kernel<uint16_t, 512>, j)
               : cudaLaunchKernelEx(&cfg, resid_kernel<float, 512>, j);
    else
        e = bf ? cudaLaunchKernelEx(&cfg, resid_kernel<uint16_t, 1024>, j)
               : cudaLaunchKernelEx(&cfg, resid_kernel<float, 1024>, j);
    if (e != cudaSuccess) return e;
    // The fp64 path's grid barriers need every CTA resident: a cooperative
    // launch guarantees it (or fails).  It returns at once when no sequence
    // was listed.
    Job jj = j;
    void *args[] = {(void *)&jj};
    return cudaLaunchCooperativeKernel(bf ? (const void *)rescue_kernel<uint16_t>
                                          : (const void *)rescue_kernel<float>,
                                       dim3(coop_grid), dim3(kPostThreads), args, 0, s);
}

size_t rescue_scratch_doubles(int B)
{
    return (size_t)B * kResidChunks * 8 + (size_t)B * kMaxPairs * 2 * kRescueChunks * 2 +
           (size_t)B * kResidChunks * 4;
}

}  // namespace sv
