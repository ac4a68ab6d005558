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
// once).  Each thread streams vectors t, t + 256, ... (16-byte loads, eight
// in flight) and keeps its four largest elements; a vector is looked at
// element by element only when its largest element beats the thread's
// fourth.  The CTA then sorts the 1024 candidates and takes the k-th, m_k.
// A thread whose fourth entry is still at least m_k may have dropped an
// element of the top k; there are at most k/4 such threads (each holds four
// of the k candidates at or above m_k), and each of them rescans its share
// with a list of k entries, which then replaces its four.  Every other
// dropped element lies below its thread's fourth, hence below m_k, hence
// below the row's k-th: the sorted candidates then start with the row's top
// k, exactly.
// ---------------------------------------------------------------------------
template <typename In>
__global__ void __launch_bounds__(kTkThreads) topk_select_kernel(const __grid_constant__ TopkJob j)
{
    __shared__ uint64_t keys[2 * kTkCand];
    __shared__ uint64_t ul[kTkUnsafe][kTopkMax];
    __shared__ int nuns;
    pdl_wait();
    pdl_trigger();
    using VT = VecTraits<In>;
    constexpr int E = VT::N;
    const int R = j.K + j.W;
    const int row = blockIdx.x;
    const int b = row / R, r = row - b * R;
    if (r < j.K && r > tk_len(j, b))
        return;  // a verify row the step does not need (uniform in the CTA)
    const int k = r < j.K ? j.kp : j.kq;
    const uint4 *rv = reinterpret_cast<const uint4 *>(j.src + (int64_t)row * j.rs);
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
#pragma unroll
    for (int i = 0; i < kTkLocal; ++i)
        keys[t * kTkLocal + i] = lv[i] >= 0 ? tk_key(lx[i], (uint32_t)lv[i]) : 0ull;
    if (t == 0)
        nuns = 0;
    __syncthreads();
    bitonic_desc(keys, kTkCand);
    const uint64_t mk = keys[k - 1];
    const bool uns = lv[kTkLocal - 1] >= 0 &&
                     tk_key(lx[kTkLocal - 1], (uint32_t)lv[kTkLocal - 1]) >= mk;
    if (__syncthreads_or(uns)) {
        if (uns) {
            const int slot = atomicAdd(&nuns, 1);
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
        const int nu = min(nuns, kTkUnsafe);
        for (int i = t; i < kTkCand; i += kTkThreads) {
            const int s = i / kTopkMax, m = i - s * kTopkMax;
            keys[kTkCand + i] = (s < nu && m < k) ? ul[s][m] : 0ull;
        }
        __syncthreads();
        bitonic_desc(keys, 2 * kTkCand);
    }
    for (int m = t; m < k; m += kTkThreads) {
        const uint64_t key = keys[m];
        j.lval[(int64_t)row * kTopkMax + m] = ord2f((uint32_t)(key >> 32));
        j.lid[(int64_t)row * kTopkMax + m] = (int32_t)~(uint32_t)key;
    }
}

// ---------------------------------------------------------------------------
// Decision step: one warp per sequence, fp64, on the lists (Alg. 2 with the
// truncated distributions).  Lane i tests draft position i: p(d_i) =
// exp(x_d/T - L) when d_i is in the target's list (L: the log-sum-exp of the
// list at T), else 0; Q(d_i) from the stored list prev_off + i; accept when
// u < min{1, p/Q}.  At the first rejection h the correction is the
// Gumbel-max of log [p(v) - Q(v)]_+ over the target list of row h (lanes
// over its entries); with every draft accepted, the bonus is the Gumbel-max
// of x/T over that list.  Lane j then draws proposal j over its list of kq
// entries and writes the list with its probabilities.  Decisions within
// 1e-9 of their threshold are counted in flags.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) topk_decide_kernel(const __grid_constant__ TopkJob j)
{
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (b >= j.B)
        return;
    const int R = j.K + j.W;
    const int len = __ldg(j.prev_len + b);
    const int n = tk_len(j, b);
    int off = __ldg(j.prev_off + b);
    if (lane == 0 && (len < 0 || len > j.K - 1 || off < 0 || off + n > j.W))
        latch(j.err, SV_ERR_DEVICE_BOUNDS);
    off = min(max(off, 0), j.W - n);
    const int64_t p0 = j.pos_base ? __ldg(j.pos_base + b) : 0;
    const double T = (double)j.T;
    const float *lval = j.lval + (int64_t)b * R * kTopkMax;
    const int32_t *lid = j.lid + (int64_t)b * R * kTopkMax;
    int nflag = 0;

    // ---- verification of the previous draft ----
    bool acc = false;
    if (lane < n) {
        const float *xv = lval + lane * kTopkMax;
        const int32_t *xi = lid + lane * kTopkMax;
        const double m = (double)xv[0] / T;
        double s = 0.0;
        for (int e = 0; e < j.kp; ++e)
            s += exp((double)xv[e] / T - m);
        const double L = m + log(s);
        const int d = __ldg(j.prev_draft + (int64_t)b * (j.K - 1) + lane);
        double log_p = -INFINITY;
        for (int e = 0; e < j.kp; ++e)
            if (xi[e] == d)
                log_p = (double)xv[e] / T - L;
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
            const double u = uniform_at(rng_key(j.seed, kAccept, (uint64_t)b, p0 + lane, 0), 0,
                                        j.skip);
            acc = u < a;
            nflag += fabs(u - a) < kFlagEps;
        }
    }
    const unsigned am = __ballot_sync(0xFFFFFFFFu, acc);
    int h = (~am == 0u) ? 32 : __ffs(~am) - 1;
    h = min(h, n);

    // ---- correction (h < n) or bonus (h == n) from the target list of row h ----
    const float *xv = lval + h * kTopkMax;
    const int32_t *xi = lid + h * kTopkMax;
    const double mh = (double)xv[0] / T;
    double sp = 0.0;
    for (int e = lane; e < j.kp; e += 32)
        sp += exp((double)xv[e] / T - mh);
    for (int o = 16; o > 0; o >>= 1)
        sp += __shfl_xor_sync(0xFFFFFFFFu, sp, o);
    const double Lh = mh + log(sp);
    const uint64_t key = rng_key(j.seed, kSample, (uint64_t)b, p0 + h, 0);
    double best = -INFINITY, second = -INFINITY;
    int bv = 0x7FFFFFFF;
    for (int e = lane; e < j.kp; e += 32) {
        const int v = xi[e];
        double w = (double)xv[e] / T;
        if (h < n) {
            const int32_t *qi = j.prev_q_ids + ((int64_t)b * j.W + off + h) * j.kq;
            const float *qp = j.prev_q_probs + ((int64_t)b * j.W + off + h) * j.kq;
            double q = 0.0;
            for (int f = 0; f < j.kq; ++f)
                if (__ldg(qi + f) == v)
                    q = (double)__ldg(qp + f);
            const double rr = exp(w - Lh) - q;
            w = rr > 0.0 ? log(rr) : -INFINITY;
        }
        if (w == -INFINITY)
            continue;
        const double sc = w + gumbel64(fine52(key, (uint32_t)v), is_top(key, (uint32_t)v, j.skip));
        if (sc > best || (sc == best && v < bv)) {
            second = best;
            best = sc;
            bv = v;
        } else if (sc > second) {
            second = sc;
        }
    }
    // warp best (score desc, id asc) and the runner-up score
    double wb = best;
    for (int o = 16; o > 0; o >>= 1)
        wb = fmax(wb, __shfl_xor_sync(0xFFFFFFFFu, wb, o));
    int cand = (best == wb) ? bv : 0x7FFFFFFF;
    const int c = __reduce_min_sync(0xFFFFFFFFu, cand);
    double run = (best == wb && bv == c) ? second : best;
    for (int o = 16; o > 0; o >>= 1)
        run = fmax(run, __shfl_xor_sync(0xFFFFFFFFu, run, o));
    if (wb - run < kFlagEps)
        nflag += lane == 0;

    // ---- committed block and stopping index ----
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

    // ---- proposals over the drafter lists: lane = proposal j ----
    int z = -1;
    double qz = 0.0;
    if (lane < j.W) {
        const int rr = j.K + lane;
        const float *yv = lval + rr * kTopkMax;
        const int32_t *yi = lid + rr * kTopkMax;
        const double m = (double)yv[0] / T;
        double s = 0.0;
        for (int e = 0; e < j.kq; ++e)
            s += exp((double)yv[e] / T - m);
        const double L = m + log(s);
        const uint64_t kd = rng_key(j.seed, kDraft, (uint64_t)b, p0 + lane, j.iter);
        double zb = -INFINITY, z2 = -INFINITY, zx = 0.0;
        for (int e = 0; e < j.kq; ++e) {
            const int v = yi[e];
            const double x = (double)yv[e] / T;
            const double sc = x + gumbel64(fine52(kd, (uint32_t)v), is_top(kd, (uint32_t)v, j.skip));
            if (sc > zb || (sc == zb && v < z)) {
                z2 = zb;
                zb = sc;
                z = v;
                zx = x;
            } else if (sc > z2) {
                z2 = sc;
            }
            j.q_ids[((int64_t)b * j.W + lane) * j.kq + e] = v;
            j.q_probs[((int64_t)b * j.W + lane) * j.kq + e] = (float)exp(x - L);
        }
        qz = exp(zx - L);
        if (lane >= a && zb - z2 < kFlagEps)
            ++nflag;
    }
    const int nl = max(j.W - a, 0);
    const int zs = __shfl_sync(0xFFFFFFFFu, z, min(lane + a, 31));
    const double qs = __shfl_sync(0xFFFFFFFFu, qz, min(lane + a, 31));
    if (lane < j.W) {
        j.next_draft[(int64_t)b * j.W + lane] = lane < nl ? zs : -1;
        if (j.next_q)
            j.next_q[(int64_t)b * j.W + lane] = lane < nl ? (float)qs : __int_as_float(0x7FC00000);
    }
    for (int o = 16; o > 0; o >>= 1)
        nflag += __shfl_xor_sync(0xFFFFFFFFu, nflag, o);
    if (lane == 0) {
        j.acc[b] = h;
        j.commit_len[b] = a;
        j.next_len[b] = nl;
        if (j.flags)
            j.flags[b] = nflag;
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
    pdl_config(cfg, at, dim3((t.B + 3) / 4), dim3(128), 0, s);
    return cudaLaunchKernelEx(&cfg, topk_decide_kernel, t);
}

}  // namespace sv
