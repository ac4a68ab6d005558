// sv_topk.cu -- the Packed-SS step with top-k truncated target and drafter
// distributions ("One Call Ahead: Packed Self-Speculative Decoding with
// Diffusion Drafting", §3.2, last paragraph: with top-k truncation only the
// nonzero entries of the stored drafter distribution Q are kept; Alg. 2).
//
// Truncation keeps a row's k largest logits (ties to the lowest id) and
// renormalises softmax(x/T) over them: kp entries for the target's verify
// rows, kq for the drafter's proposal rows.  With the lists in hand the step
// needs no pass over the vocabulary: the acceptance test, the residual
// [p - Q]_+ and every Gumbel-max run over at most 64 entries, in fp64.
#include "sv_common.cuh"
#include "sv_topk.cuh"

namespace sv {

namespace {

constexpr int kTkThreads = 256;
constexpr int kTkLocal = 4;   // entries each thread keeps while it streams
constexpr int kTkBatch = 8;   // vectors a thread has in flight
constexpr int kTkCand = kTkThreads * kTkLocal;
constexpr int kTkUnsafe = kTopkMax / kTkLocal;  // see the selection below

// Order key: larger logit first, then lower id (0 = no entry).
__device__ __forceinline__ uint64_t tk_key(float x, uint32_t v)
{
    return ((uint64_t)f2ord(x) << 32) | (uint32_t)~v;
}

// Insert (x, v) into a thread's list, sorted by decreasing logit, given
// x > lx[3].  Elements reach a thread in increasing id order, so an element
// equal to a listed logit comes after it.
__device__ __forceinline__ void tk_insert(float (&lx)[kTkLocal], int (&lv)[kTkLocal], float x,
                                          int v)
{
    if (x > lx[2]) {
        lx[3] = lx[2];
        lv[3] = lv[2];
        if (x > lx[1]) {
            lx[2] = lx[1];
            lv[2] = lv[1];
            if (x > lx[0]) {
                lx[1] = lx[0];
                lv[1] = lv[0];
                lx[0] = x;
                lv[0] = v;
            } else {
                lx[1] = x;
                lv[1] = v;
            }
        } else {
            lx[2] = x;
            lv[2] = v;
        }
    } else {
        lx[3] = x;
        lv[3] = v;
    }
}

// Sort a[0..N-1] (N a power of two) into decreasing order; whole CTA.
__device__ void bitonic_desc(uint64_t *a, int N)
{
    for (int size = 2; size <= N; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < N; i += blockDim.x) {
                const int jx = i ^ stride;
                if (jx > i) {
                    const uint64_t x = a[i], y = a[jx];
                    const bool desc = (i & size) == 0;
                    if (desc ? (x < y) : (x > y)) {
                        a[i] = y;
                        a[jx] = x;
                    }
                }
            }
            __syncthreads();
        }
}

__device__ __forceinline__ int tk_len(const TopkJob &j, int b)
{
    return min(max(__ldg(j.prev_len + b), 0), j.K - 1);
}

}  // namespace

// ---------------------------------------------------------------------------
// Selection: one CTA per row of the step (verify rows beyond prev_len exit at
// once); thread t streams vectors t, t + 256, ... (16-byte loads, eight in
// flight).
//
// Fast path.  Each thread takes the largest logit of its first eight
// vectors, and tau = the k-th largest of those 256 maxima (a bitwise search
// with CTA-wide counts): k elements of the row are >= tau, so its top k are.
// The stream then compares each vector's largest logit with tau and appends
// the elements >= tau, as order keys (logit, then lower id), to a shared
// buffer -- a few hundred for k = 64 on the rows here -- which is sorted at
// the end.
//
// Exact fallback, for a row that overflows the buffer (many equal logits,
// say): the row is streamed again; each thread keeps its four largest
// elements, the CTA sorts the 1024 candidates and takes the k-th, m_k.  A
// thread whose fourth entry is still at least m_k may have dropped an
// element of the top k; there are at most k/4 such threads (each holds four
// of the k candidates at or above m_k), and each rescans its share with a
// list of k entries, which then replaces its four.  Every other dropped
// element lies below its thread's fourth, hence below m_k, hence below the
// row's k-th.
// ---------------------------------------------------------------------------
constexpr int kTkBuf = 2048;  // fast-path candidate buffer (order keys)

template <typename In>
__device__ void topk_fallback(const TopkJob &j, const uint4 *rv, int k, uint64_t *keys,
                              uint64_t (*ul)[kTopkMax], int *nuns)
{
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    const int t = threadIdx.x;
    float lx[kTkLocal];
    int lv[kTkLocal];
#pragma unroll
    for (int i = 0; i < kTkLocal; ++i) {
        lx[i] = -INFINITY;
        lv[i] = -1;
    }
    for (int base = t; base < j.nvec; base += kTkThreads * kTkBatch) {
        uint4 q[kTkBatch];
#pragma unroll
        for (int u = 0; u < kTkBatch; ++u) {
            const int idx = base + u * kTkThreads;
            q[u] = idx < j.nvec ? __ldg(rv + idx) : VT::neg_inf_vec();
        }
#pragma unroll
        for (int u = 0; u < kTkBatch; ++u) {
            if (VT::hi_of(VT::pmax(q[u])) > lx[kTkLocal - 1]) {
                const int v0 = (base + u * kTkThreads) * E;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float x = VT::elem(q[u], e);
                    if (x > lx[kTkLocal - 1])
                        tk_insert(lx, lv, x, v0 + e);
                }
            }
        }
    }
    __syncthreads();  // the fast path's keys are no longer read
#pragma unroll
    for (int i = 0; i < kTkLocal; ++i)
        keys[t * kTkLocal + i] = lv[i] >= 0 ? tk_key(lx[i], (uint32_t)lv[i]) : 0ull;
    if (t == 0)
        *nuns = 0;
    __syncthreads();
    bitonic_desc(keys, kTkCand);
    const uint64_t mk = keys[k - 1];
    const bool uns = lv[kTkLocal - 1] >= 0 &&
                     tk_key(lx[kTkLocal - 1], (uint32_t)lv[kTkLocal - 1]) >= mk;
    if (__syncthreads_or(uns)) {
        if (uns) {
            const int slot = atomicAdd(nuns, 1);
            if (slot < kTkUnsafe) {
                uint64_t *L = ul[slot];
                for (int m = 0; m < kTopkMax; ++m)
                    L[m] = 0ull;
                for (int idx = t; idx < j.nvec; idx += kTkThreads) {
                    const uint4 q = __ldg(rv + idx);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const uint64_t key = tk_key(VT::elem(q, e), (uint32_t)(idx * E + e));
                        if (key > L[k - 1]) {
                            int p = k - 1;
                            while (p > 0 && L[p - 1] < key) {
                                L[p] = L[p - 1];
                                --p;
                            }
                            L[p] = key;
                        }
                    }
                }
            } else {
                latch(j.err, SV_ERR_DEVICE_BOUNDS);  // cannot happen: at most k/4 threads
            }
        }
        __syncthreads();
        // the rescanned threads' lists replace their four entries
#pragma unroll
        for (int i = 0; i < kTkLocal; ++i)
            keys[t * kTkLocal + i] =
                (!uns && lv[i] >= 0) ? tk_key(lx[i], (uint32_t)lv[i]) : 0ull;
        const int nu = min(*nuns, kTkUnsafe);
        for (int i = t; i < kTkCand; i += kTkThreads) {
            const int s2 = i / kTopkMax, m = i - s2 * kTopkMax;
            keys[kTkCand + i] = (s2 < nu && m < k) ? ul[s2][m] : 0ull;
        }
        __syncthreads();
        bitonic_desc(keys, 2 * kTkCand);
    }
}

template <typename In>
__global__ void __launch_bounds__(kTkThreads) topk_select_kernel(const __grid_constant__ TopkJob j)
{
    __shared__ uint64_t keys[kTkBuf];
    __shared__ uint64_t ul[kTkUnsafe][kTopkMax];
    __shared__ int ncand, nuns;
    pdl_wait();
    pdl_trigger();
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    static_assert(kTkBuf >= 2 * kTkCand, "the fallback sorts 2 x 1024 keys in the buffer");
    const int R = j.K + j.W;
    const int row = blockIdx.x;
    const int b = row / R, r = row - b * R;
    if (r < j.K && r > tk_len(j, b))
        return;  // a verify row the step does not need (uniform in the CTA)
    const int k = r < j.K ? j.kp : j.kq;
    const uint4 *rv = reinterpret_cast<const uint4 *>(j.src + (int64_t)row * j.rs);
    const int t = threadIdx.x;
    if (t == 0)
        ncand = 0;
    // first batch: the thread's largest logit, and tau from the 256 maxima
    uint4 q[kTkBatch];
    float tmax = -INFINITY;
#pragma unroll
    for (int u = 0; u < kTkBatch; ++u) {
        const int idx = t + u * kTkThreads;
        q[u] = idx < j.nvec ? __ldg(rv + idx) : VT::neg_inf_vec();
        tmax = fmaxf(tmax, VT::hi_of(VT::pmax(q[u])));
    }
    // the search fixes the top 16 bits of the k-th largest order key and
    // leaves the rest zero: a value at most the k-th largest maximum
    float tau = -INFINITY;
    if (__syncthreads_count(tmax > -INFINITY) >= k) {
        const uint32_t key = f2ord(tmax);
        uint32_t T = 0u;
        for (int bit = 31; bit >= 16; --bit) {
            const uint32_t c = T | (1u << bit);
            if (__syncthreads_count(key >= c) >= k)
                T = c;
        }
        tau = ord2f(T);
    }
    // the stream: elements >= tau go to the buffer
    for (int base = t;; base += kTkThreads * kTkBatch) {
#pragma unroll
        for (int u = 0; u < kTkBatch; ++u) {
            if (VT::hi_of(VT::pmax(q[u])) >= tau) {
                const int v0 = (base + u * kTkThreads) * E;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float x = VT::elem(q[u], e);
                    if (x >= tau) {
                        const int p = atomicAdd(&ncand, 1);
                        if (p < kTkBuf)
                            keys[p] = tk_key(x, (uint32_t)(v0 + e));
                    }
                }
            }
        }
        const int nb = base + kTkThreads * kTkBatch;
        if (nb - t >= j.nvec)
            break;
#pragma unroll
        for (int u = 0; u < kTkBatch; ++u) {
            const int idx = nb + u * kTkThreads;
            q[u] = idx < j.nvec ? __ldg(rv + idx) : VT::neg_inf_vec();
        }
    }
    __syncthreads();
    const int nc = ncand;
    if (nc <= kTkBuf) {
        int N = 64;
        while (N < nc)
            N <<= 1;
        for (int i = nc + t; i < N; i += kTkThreads)
            keys[i] = 0ull;
        __syncthreads();
        bitonic_desc(keys, N);
    } else {
        topk_fallback<In>(j, rv, k, keys, ul, &nuns);
    }
    for (int m = t; m < k; m += kTkThreads) {
        const uint64_t key = keys[m];
        j.lval[(int64_t)row * kTopkMax + m] = ord2f((uint32_t)(key >> 32));
        j.lid[(int64_t)row * kTopkMax + m] = (int32_t)~(uint32_t)key;
    }
}

// ---------------------------------------------------------------------------
// Decision step: one CTA of 128 threads per sequence, fp64, on the lists
// (Alg. 2 with the truncated distributions).
//  1. Every thread takes list entries of the rows the step uses (verify rows
//     0..prev_len, the W proposal rows): e = exp(x/T - m) with m the list's
//     first (largest) logit / T; one thread per row then sums its entries in
//     list order, L = m + log(sum), the list's log-sum-exp at T.  The terms
//     of proposal rows, which only feed fp32 outputs (the stored
//     probabilities), are taken in fp32.
//  2. Warp 0, lane i: p(d_i) = exp(x_d/T - L) when d_i is in the target's
//     list, else 0; Q(d_i) from the stored list prev_off + i; accept when
//     u < min{1, p/Q}; h = the first rejection.
//  3. Every thread: the fp64 Gumbel scores of the entries of row h (the
//     correction or bonus key of position h), and fp32 intervals of x/T + G
//     for the entries of every proposal row (its draft key), with the
//     proposal lists and probabilities written out.
//  4. Warp 0 takes the correction (Gumbel-max of log [p - Q]_+ over row h's
//     list) or the bonus (Gumbel-max of x/T); thread j of the CTA takes
//     proposal j: the entry with the largest upper end wins when its lower
//     end clears every other upper end by 1e-9, else the row is scored in
//     fp64 like row h.
//  5. Warp 0 writes the committed block and the next draft.
// Decisions within 1e-9 of their threshold are counted in flags.
// ---------------------------------------------------------------------------
constexpr int kTdThreads = 128;
constexpr int kTdRows = 2 * kMaxK + 1;  // verify rows 0..K-1 and the proposals

__global__ void __launch_bounds__(kTdThreads) topk_decide_kernel(const __grid_constant__ TopkJob j)
{
    // verify rows: exp(x/T - m); entry kMaxK: row h's Gumbel scores
    __shared__ double ex[kMaxK + 1][kTopkMax];
    __shared__ float2 iv[kMaxK][kTopkMax];     // proposal rows: fp32 intervals of x/T + G
    __shared__ double Lrow[kTdRows];
    __shared__ int hs, as_, zs[kMaxK];
    __shared__ double qzs[kMaxK], gaps[kMaxK];
    __shared__ uint64_t rkey[kMaxK];  // the proposal rows' draft keys
    __shared__ int nfl;
    pdl_wait();
    pdl_trigger();
    const int t = threadIdx.x, lane = t & 31;
    const int b = blockIdx.x;
    const int R = j.K + j.W;
    const int len = __ldg(j.prev_len + b);
    const int n = tk_len(j, b);
    int off = __ldg(j.prev_off + b);
    if (t == 0) {
        nfl = 0;
        if (len < 0 || len > j.K - 1 || off < 0 || off + n > j.W)
            latch(j.err, SV_ERR_DEVICE_BOUNDS);
    }
    off = min(max(off, 0), j.W - n);
    const int64_t p0 = j.pos_base ? __ldg(j.pos_base + b) : 0;
    const double T = (double)j.T;
    const int64_t row0 = (int64_t)b * R;
    // local row q: verify rows 0..n are q = 0..n, proposal j is q = K + j
    auto gro = [&](int q) { return row0 + q; };

    // ---- 1. list terms and log-sum-exps (entries spread over all threads) ----
    if (t < j.W)
        rkey[t] = rng_key(j.seed, kDraft, (uint64_t)b, p0 + t, j.iter);
    const int items = (n + 1) * j.kp;
    for (int it = t; it < items; it += kTdThreads) {
        const int q = it / j.kp, e = it - q * j.kp;
        const float *xv = j.lval + gro(q) * kTopkMax;
        ex[q][e] = exp((double)xv[e] / T - (double)xv[0] / T);
    }
    __syncthreads();
    for (int qi = t; qi < n + 1 + j.W; qi += kTdThreads) {
        const int q = qi <= n ? qi : j.K + (qi - n - 1);
        const float *xv = j.lval + gro(q) * kTopkMax;
        double sum = 0.0;
        if (q < j.K) {
            for (int e = 0; e < j.kp; ++e)
                sum += ex[q][e];
        } else {
            const float m = (float)((double)xv[0] / T);
            for (int e = 0; e < j.kq; ++e)
                sum += (double)expf((float)((double)xv[e] / T) - m);
        }
        Lrow[q] = (double)xv[0] / T + log(sum);
    }
    __syncthreads();

    // ---- 2. verification of the previous draft (warp 0) ----
    if (t < 32) {
        bool acc = false;
        int nf = 0;
        if (lane < n) {
            const float *xv = j.lval + gro(lane) * kTopkMax;
            const int32_t *xi = j.lid + gro(lane) * kTopkMax;
            const int d = __ldg(j.prev_draft + (int64_t)b * (j.K - 1) + lane);
            double log_p = -INFINITY;
            for (int e = 0; e < j.kp; ++e)
                if (xi[e] == d)
                    log_p = (double)xv[e] / T - Lrow[lane];
            const int32_t *qi = j.prev_q_ids + ((int64_t)b * j.W + off + lane) * j.kq;
            const float *qp = j.prev_q_probs + ((int64_t)b * j.W + off + lane) * j.kq;
            double Qd = 0.0;
            for (int e = 0; e < j.kq; ++e)
                if (__ldg(qi + e) == d)
                    Qd = (double)__ldg(qp + e);
            if (!(Qd > 0.0)) {
                latch(j.err, SV_ERR_DEVICE_BOUNDS);  // the draft is not in its stored list
            } else {
                const double a = fmin(1.0, exp(log_p - log(Qd)));
                const double u = uniform_at(rng_key(j.seed, kAccept, (uint64_t)b, p0 + lane, 0),
                                            0, j.skip);
                acc = u < a;
                nf = fabs(u - a) < kFlagEps;
            }
        }
        const unsigned am = __ballot_sync(0xFFFFFFFFu, acc);
        const int h = min((~am == 0u) ? 32 : __ffs(~am) - 1, n);
        nf = __reduce_add_sync(0xFFFFFFFFu, nf);
        if (lane == 0) {
            hs = h;
            nfl += nf;
        }
    }
    __syncthreads();
    const int h = hs;

    // ---- 3. scores: row h's correction / bonus terms (every second thread,
    // so that the fp64 work spreads over the warps), then the proposal terms
    const uint64_t hkey = rng_key(j.seed, kSample, (uint64_t)b, p0 + h, 0);
    const int items3 = 2 * j.kp + j.W * j.kq;
    for (int it = t; it < items3; it += kTdThreads) {
        const bool corr = it < 2 * j.kp;
        if (corr && (it & 1))
            continue;
        const int qi = corr ? 0 : 1 + (it - 2 * j.kp) / j.kq;
        const int e = corr ? it >> 1 : (it - 2 * j.kp) - (qi - 1) * j.kq;
        const int q = qi == 0 ? h : j.K + qi - 1;
        const int64_t gr = gro(q);
        const int v = j.lid[gr * kTopkMax + e];
        const double x = (double)j.lval[gr * kTopkMax + e] / T;
        double w = x;
        uint64_t key;
        if (qi == 0) {
            key = hkey;
            if (h < n) {
                const int32_t *qv = j.prev_q_ids + ((int64_t)b * j.W + off + h) * j.kq;
                const float *qp = j.prev_q_probs + ((int64_t)b * j.W + off + h) * j.kq;
                double qq = 0.0;
                for (int f = 0; f < j.kq; ++f)
                    if (__ldg(qv + f) == v)
                        qq = (double)__ldg(qp + f);
                const double rr = exp(x - Lrow[q]) - qq;
                w = rr > 0.0 ? log(rr) : -INFINITY;
            }
            ex[kMaxK][e] =
                w == -INFINITY
                    ? -INFINITY
                    : w + gumbel64(fine52(key, (uint32_t)v), is_top(key, (uint32_t)v, j.skip));
        } else {
            key = rkey[qi - 1];
            const int64_t o = ((int64_t)b * j.W + (qi - 1)) * j.kq + e;
            j.q_ids[o] = v;
            j.q_probs[o] = expf((float)(x - Lrow[q]));
            iv[qi - 1][e] = logit_interval_m(j.lval[gr * kTopkMax + e], (float)(1.0 / T),
                                             fine52(key, (uint32_t)v),
                                             is_top(key, (uint32_t)v, j.skip));
        }
    }
    __syncthreads();

    // ---- 4. correction / bonus (warp 0) and proposals (thread j) ----
    if (t < 32) {
        double best = -INFINITY, second = -INFINITY;
        int bv = 0x7FFFFFFF;
        for (int e = lane; e < j.kp; e += 32) {
            const double sc = ex[kMaxK][e];
            if (sc == -INFINITY)
                continue;
            const int v = j.lid[gro(h) * kTopkMax + e];
            if (sc > best || (sc == best && v < bv)) {
                second = best;
                best = sc;
                bv = v;
            } else if (sc > second) {
                second = sc;
            }
        }
        double wb = best;
        for (int o = 16; o > 0; o >>= 1)
            wb = fmax(wb, __shfl_xor_sync(0xFFFFFFFFu, wb, o));
        const int c = __reduce_min_sync(0xFFFFFFFFu, (best == wb) ? bv : 0x7FFFFFFF);
        double run = (best == wb && bv == c) ? second : best;
        for (int o = 16; o > 0; o >>= 1)
            run = fmax(run, __shfl_xor_sync(0xFFFFFFFFu, run, o));
        // committed block and stopping index
        const int tok = lane < h ? __ldg(j.prev_draft + (int64_t)b * (j.K - 1) + lane)
                                 : (lane == h ? c : -1);
        int a = h + 1;
        if (j.remaining) {
            const int rem = __ldg(j.remaining + b);
            if (rem < a)
                a = max(rem, 0);
        }
        if (j.eos >= 0) {
            const unsigned em = __ballot_sync(0xFFFFFFFFu, lane <= h && tok == j.eos);
            if (em)
                a = min(a, __ffs(em));
        }
        if (lane < j.K)
            j.committed[(int64_t)b * j.K + lane] = lane < a ? tok : -1;
        if (lane == 0) {
            as_ = a;
            if (wb - run < kFlagEps)
                ++nfl;
        }
    }
    if (t >= 32 && t - 32 < j.W) {
        const int jj = t - 32, q = j.K + jj;
        const int32_t *yi = j.lid + gro(q) * kTopkMax;
        const float *yv = j.lval + gro(q) * kTopkMax;
        // the largest upper end (lowest id on ties), and every other upper end
        int eb = 0;
        for (int e = 1; e < j.kq; ++e)
            if (iv[jj][e].y > iv[jj][eb].y || (iv[jj][e].y == iv[jj][eb].y && yi[e] < yi[eb]))
                eb = e;
        float ho = -INFINITY;
        for (int e = 0; e < j.kq; ++e)
            if (e != eb)
                ho = fmaxf(ho, iv[jj][e].y);
        int z = yi[eb], ze = eb;
        double gap = INFINITY;  // certified: above 1e-9
        if (!((double)iv[jj][eb].x - 1e-9 > (double)ho)) {
            // not certified in fp32: the row's scores in fp64
            const uint64_t key = rkey[jj];
            double zb = -INFINITY, z2 = -INFINITY;
            z = -1;
            for (int e = 0; e < j.kq; ++e) {
                const int v = yi[e];
                const double sc = (double)yv[e] / T +
                                  gumbel64(fine52(key, (uint32_t)v), is_top(key, (uint32_t)v, j.skip));
                if (sc > zb || (sc == zb && v < z)) {
                    z2 = zb;
                    zb = sc;
                    z = v;
                    ze = e;
                } else if (sc > z2) {
                    z2 = sc;
                }
            }
            gap = zb - z2;
        }
        zs[jj] = z;
        qzs[jj] = (double)expf((float)((double)yv[ze] / T - Lrow[q]));
        gaps[jj] = gap;
    }
    __syncthreads();

    // ---- 5. next draft and per-sequence results (warp 0) ----
    if (t < 32) {
        const int a = as_;
        const int nl = max(j.W - a, 0);
        int nf = 0;
        if (lane < j.W) {
            const int src = lane + a;
            j.next_draft[(int64_t)b * j.W + lane] = lane < nl ? zs[src] : -1;
            if (j.next_q)
                j.next_q[(int64_t)b * j.W + lane] =
                    lane < nl ? (float)qzs[src] : __int_as_float(0x7FC00000);
            nf = lane >= a && gaps[lane] < kFlagEps;
        }
        nf = __reduce_add_sync(0xFFFFFFFFu, nf);
        if (lane == 0) {
            j.acc[b] = h;
            j.commit_len[b] = a;
            j.next_len[b] = nl;
            if (j.flags)
                j.flags[b] = nfl + nf;
        }
    }
}

cudaError_t topk_select_launch(const TopkJob &t, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    pdl_config(cfg, at, dim3(t.B * (t.K + t.W)), dim3(kTkThreads), 0, s);
    return t.dtype == SV_BF16 ? cudaLaunchKernelEx(&cfg, topk_select_kernel<uint16_t>, t)
                              : cudaLaunchKernelEx(&cfg, topk_select_kernel<float>, t);
}

cudaError_t topk_decide_launch(const TopkJob &t, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    pdl_config(cfg, at, dim3(t.B), dim3(kTdThreads), 0, s);
    return cudaLaunchKernelEx(&cfg, topk_decide_kernel, t);
}

}  // namespace sv
