/*
 * sv_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct fp64 CPU restatement of draft-block
 * verification.  The tests, the smoke check and the benchmark's CPU-baseline
 * leg use it to check the CUDA library; no product code path calls it, and it
 * shares no source (no header, helper, table or constant generator) with the
 * CUDA library.
 *
 * Sources, cited below by short name with the section / equation / algorithm:
 *   [PackedSS] "One Call Ahead: Packed Self-Speculative Decoding with Diffusion
 *              Drafting"
 *   [SPOT]     "On the SPOT: Enhancing Speculative Decoding for Diffusion
 *              Language Models via Commit-Order Prediction"
 *   [TwoTrade] "Speculative Diffusion is a Tale of Two Tradeoffs"
 *
 * Precision: every logit is upcast exactly to double; all arithmetic is fp64.
 * Where the pages leave a step open, the choice is marked READING.
 * Parity unpinned (no page fixes the result): the residual law of the ratio
 * lenience mode for lambda > 1, and the tie-break between equally deep tree
 * paths.  Everything else is pinned by the tests in tests/test_oracle_*.py.
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1 };
enum { OR_LOSSLESS = 0, OR_RATIO = 1, OR_LINEAR = 2, OR_CACTUS = 3 };
/* Random-number streams (READING: the pages only ask for independent uniforms
 * and Gumbels; [PackedSS] App. B.2 "Conditioning information" requires draft
 * sampling, acceptance tests and corrections to use independent numbers). */
enum { ST_ACCEPT = 1, ST_SAMPLE = 2, ST_DRAFT = 3, ST_TREE = 4 };
/* A decision within this distance of its threshold is flagged, not compared. */
#define OR_FLAG_EPS 1e-9

/* ------------------------------------------------------------------------ */
/* Counter-based random numbers.                                             */
/* ------------------------------------------------------------------------ */

/* SplitMix64 output function (Steele, Lea & Flood 2014; Vigna's reference
 * splitmix64.c): advance by the golden gamma, then two xor-shift-multiply
 * rounds and a final xor-shift. */
uint64_t or_mix64(uint64_t x)
{
    uint64_t z = x + 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Row key: a chain of the 64-bit mixer over the counter fields. */
uint64_t or_key(uint64_t seed, uint32_t stream, uint64_t seq, int64_t pos, uint64_t iter)
{
    uint64_t k = or_mix64(seed);
    k = or_mix64(k ^ (uint64_t)stream);
    k = or_mix64(k ^ seq);
    k = or_mix64(k ^ (uint64_t)pos);
    k = or_mix64(k ^ iter);
    return k;
}

/* Uniforms of a row (row key k, vocabulary id v).  All randomness of a row is
 * read from the SplitMix64 stream seeded with k: output number n + 1 is
 * S(k, n) = or_mix64(k + n * 0x9E3779B97F4A7C15).
 *
 * The ids are split into blocks of 256 (block b = v div 256).  Which ids of a
 * block fall into the top 1/256 of the unit interval ("top" ids) is drawn as
 * i.i.d. Bernoulli(1/256) trials by geometric skipping (the number of failures
 * before each success is geometric; the classical skip method for Bernoulli
 * sequences): draw i of block b is M = S(k, b * 2^16 + i), its gap is the
 * number of g in 1..256 with M < C_g, C_g = ceil(2^64 (255/256)^g), so that
 * P(gap >= g) = C_g / 2^64 = (255/256)^g to within 2^-64; the first top
 * offset is gap_0 and each next one is the previous plus 1 + gap_i, until an
 * offset passes 255.
 * Fine bits: m = S(k, 2^40 + v) >> 12 (52 bits), w = (2m + 1) / 2^53.
 * Uniform: u = w * 255/256 for an ordinary id, and 1 - u = (1 - w) / 256
 * (exact) for a top id, so that u is uniform on (0, 1) and G = -log(-log u)
 * is standard Gumbel. */
static uint64_t or_stream(uint64_t k, uint64_t n)
{
    return or_mix64(k + n * 0x9E3779B97F4A7C15ULL);
}

/* C_g for g = 1..256 (index 0 unused), exact: 255^g as a multi-word integer,
 * times 2^(64 - 8g), rounded up. */
static uint64_t or_skip_c[257];
static int or_skip_ready = 0;

static void or_skip_init(void)
{
    if (or_skip_ready)
        return;
    uint32_t big[80];              /* 255^g, base 2^32, least significant first */
    memset(big, 0, sizeof big);
    big[0] = 1;
    int len = 1;
    for (int g = 1; g <= 256; ++g) {
        uint64_t carry = 0;
        for (int i = 0; i < len; ++i) {
            uint64_t t = (uint64_t)big[i] * 255u + carry;
            big[i] = (uint32_t)t;
            carry = t >> 32;
        }
        if (carry)
            big[len++] = (uint32_t)carry;
        int shift = 8 * g - 64;        /* value = 255^g / 2^shift */
        if (shift <= 0) {
            uint64_t v = (uint64_t)big[0] | ((len > 1 ? (uint64_t)big[1] : 0) << 32);
            or_skip_c[g] = v << (-shift);
        } else {
            /* floor(255^g / 2^shift), plus one if any dropped bit is set */
            int w = shift / 32, r = shift % 32, dropped = 0;
            for (int i = 0; i < w && i < len; ++i)
                dropped |= big[i] != 0;
            if (r && w < len && (big[w] & ((1u << r) - 1u)))
                dropped = 1;
            uint64_t v = 0;
            for (int i = 0; i < 3; ++i) {
                int idx = w + i;
                uint64_t limb = idx < len ? big[idx] : 0;
                if (r == 0) {
                    if (i < 2) v |= limb << (32 * i);
                } else {
                    if (i == 0) v |= limb >> r;
                    else if (i == 1) v |= limb << (32 - r);
                    else v |= limb << (64 - r);
                }
            }
            or_skip_c[g] = v + (uint64_t)dropped;
        }
    }
    or_skip_ready = 1;
}

uint64_t or_skip_threshold(int g)
{
    or_skip_init();
    return (g >= 1 && g <= 256) ? or_skip_c[g] : 0;
}

static int or_gap(uint64_t M)
{
    int g = 0;
    while (g < 256 && M < or_skip_c[g + 1])
        ++g;
    return g;
}

/* 1 if v is a top id of its block under key k. */
int or_is_top(uint64_t key, uint32_t v)
{
    or_skip_init();
    const uint64_t b = v >> 8;
    const int o = (int)(v & 255u);
    int pos = -1;
    for (uint64_t i = 0;; ++i) {
        pos += or_gap(or_stream(key, (b << 16) | i)) + 1;
        if (pos >= o)
            return pos == o;
    }
}

uint64_t or_fine52(uint64_t key, uint32_t v)
{
    return or_stream(key, (1ULL << 40) + v) >> 12;
}

/* Uniform in (0,1) (see above). */
double or_uniform(uint64_t key, uint32_t v)
{
    const double w = (double)(2 * or_fine52(key, v) + 1) * 0x1p-53;
    if (or_is_top(key, v))
        return 1.0 - (1.0 - w) / 256.0;
    return w * (255.0 / 256.0);
}

/* Uniforms and top flags of ids 0..V-1 (for tests). */
void or_row_uniforms(uint64_t key, int V, double *u, uint8_t *top)
{
    for (int v = 0; v < V; ++v) {
        u[v] = or_uniform(key, (uint32_t)v);
        top[v] = (uint8_t)or_is_top(key, (uint32_t)v);
    }
}

/* Standard Gumbel by inversion, G = -log(-log u); for a top id from the exact
 * 1 - u as -log(-log1p(-(1 - u))). */
double or_gumbel(uint64_t key, uint32_t v)
{
    const double w = (double)(2 * or_fine52(key, v) + 1) * 0x1p-53;
    if (or_is_top(key, v))
        return -log(-log1p(-((1.0 - w) / 256.0)));
    return -log(-log(w * (255.0 / 256.0)));
}

/* ------------------------------------------------------------------------ */
/* Rows.                                                                     */
/* ------------------------------------------------------------------------ */

static double bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Copy row r (row_stride elements apart) of a logit tensor into fp64. */
static void load_row(const void *base, int dtype, int64_t r, int64_t row_stride, int V, double *out)
{
    if (dtype == OR_BF16) {
        const uint16_t *p = (const uint16_t *)base + r * row_stride;
        for (int v = 0; v < V; ++v)
            out[v] = bf16_to_double(p[v]);
    } else {
        const float *p = (const float *)base + r * row_stride;
        for (int v = 0; v < V; ++v)
            out[v] = (double)p[v];
    }
}

/* log-sum-exp of x/T in index order: m + log(sum exp(z - m)), z = x/T.
 * The temperature law pi_T ∝ p^(1/T) = softmax(x/T) is [SPOT] eq. (2). */
double or_lse(const double *x, int V, double T)
{
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double z = x[v] / T;
        if (z > m)
            m = z;
    }
    double s = 0.0;
    for (int v = 0; v < V; ++v)
        s += exp(x[v] / T - m);
    return m + log(s);
}

/* argmax with the lowest index winning ties.  The pages ask only for a fixed
 * deterministic rule ([SPOT] App. A.1 "Position selection"; [PackedSS]
 * App. B.2 "Greedy decoding"); lowest index is the READING. */
int or_argmax(const double *x, int V)
{
    int best = 0;
    for (int v = 1; v < V; ++v)
        if (x[v] > x[best])
            best = v;
    return best;
}

/* Gumbel-max sample: argmax over v of score[v] + G(key, v), skipping entries
 * whose score is -inf (zero weight).  Pr[argmax = u] = softmax(score)_u is the
 * Gumbel-argmax identity, [SPOT] App. A.3 eqs. (5)-(7).  *gap receives the
 * difference between the best and second-best perturbed scores (+inf when
 * only one entry is eligible).  Lowest index wins exact ties (READING). */
int or_gumbel_argmax(const double *score, int V, uint64_t key, double *gap)
{
    int best = -1;
    double b1 = -INFINITY, b2 = -INFINITY;
    for (int v = 0; v < V; ++v) {
        if (score[v] == -INFINITY)
            continue;
        double s = score[v] + or_gumbel(key, (uint32_t)v);
        if (best < 0 || s > b1) {
            b2 = b1;
            b1 = s;
            best = v;
        } else if (s > b2) {
            b2 = s;
        }
    }
    if (gap)
        *gap = (b2 == -INFINITY) ? INFINITY : b1 - b2;
    return best;
}

/* Modified Cactus ([TwoTrade] App. E).  Given the target probability p of
 * the drafted token y and the KL budget delta, the modified target puts
 * gamma* on y, the largest gamma with
 *   Phi(gamma) = gamma log(gamma/p) + (1-gamma) log((1-gamma)/(1-p)) <= delta
 * (eq. 17), and rescales every other token by (1-gamma*)/(1-p).  Phi is 0 at
 * gamma = p, grows on [p, 1] and reaches log(1/p) at 1, so gamma* is 1 when
 * delta >= log(1/p) and otherwise the root of Phi(gamma) = delta above p.
 * The page solves it with Newton's method; so does this function, started
 * from the page's second-order (Taylor) solution p + sqrt(2 delta p (1-p))
 * (eq. 18) and kept inside a shrinking bracket [lo, hi] around the root (a
 * step that would leave it is replaced by the bracket's midpoint).
 * READING: p = 0 (a token the target cannot produce) keeps gamma* = 0. */
double or_cactus_gamma(double p, double delta)
{
    if (!(p > 0.0))
        return 0.0;
    if (p >= 1.0)
        return 1.0;
    if (!(delta > 0.0))
        return p;
    if (delta >= -log(p))
        return 1.0;
    double lo = p, hi = 1.0;
    double g = p + sqrt(2.0 * delta * p * (1.0 - p));
    if (!(g > lo && g < hi))
        g = 0.5 * (lo + hi);
    /* log(gamma/p) and log((1-gamma)/(1-p)) as log1p of (gamma-p)/p and of
     * (p-gamma)/(1-p): both quotients are near 1 when gamma is near p (small
     * delta), where their plain logs would lose most of the digits */
    for (int it = 0; it < 200; ++it) {
        double l0 = log1p((g - p) / p);
        double l1 = log1p((p - g) / (1.0 - p));
        double phi = g * l0 + (1.0 - g) * l1;
        double f = phi - delta;
        if (f == 0.0)
            break;
        if (f > 0.0)
            hi = g;
        else
            lo = g;
        double d1 = l0 - l1; /* Phi'(gamma) */
        double gn = g - f / d1;
        if (!(gn > lo && gn < hi))
            gn = 0.5 * (lo + hi);
        if (gn == g || hi - lo <= 2e-16 * hi)
            break;
        g = gn;
    }
    return g;
}

/* Acceptance probability of a draft token from log p(d) and log q(d).
 *   LOSSLESS: min{1, p/q}                      [PackedSS] §2.2; [TwoTrade] §2
 *   RATIO:    min{1, lam p/q}, lam >= 1         READING of the "predefined
 *             ratio" lenience named in [TwoTrade] §1
 *   LINEAR:   min{1, ptilde/q}, ptilde = (1-mu)p + mu q, mu = lam in [0,1]
 *                                              [TwoTrade] eq. (5), Alg. 1
 *   CACTUS:   min{1, gamma* / q}, delta = lam >= 0 [TwoTrade] App. E
 *             (gamma* = p when delta = 0, which is then the lossless rule
 *             to the last bit) */
double or_accept_prob(double log_p, double log_q, int mode, double lam)
{
    double a;
    if (mode == OR_CACTUS) {
        double p = exp(log_p);
        double g = or_cactus_gamma(p, lam);
        double lg = (g == p) ? log_p : log(g);
        a = exp(lg - log_q);
        return a < 1.0 ? a : 1.0;
    }
    double r = exp(log_p - log_q);
    if (mode == OR_RATIO)
        a = lam * r;
    else if (mode == OR_LINEAR)
        a = (1.0 - lam) * r + lam;
    else
        a = r;
    return a < 1.0 ? a : 1.0;
}

/* The factor c = (1 - gamma*)/(1 - p(d)) by which the modified Cactus
 * target rescales every token other than the drafted one d ([TwoTrade]
 * App. E); 1 for the other modes.  READING: p(d) = 1 (gamma* = 1, so d is
 * always accepted and no residual is drawn) gives 0. */
double or_residual_scale(double log_pd, int mode, double lam)
{
    if (mode != OR_CACTUS)
        return 1.0;
    double p = exp(log_pd);
    if (p >= 1.0)
        return 0.0;
    double g = or_cactus_gamma(p, lam);
    return (g == p) ? 1.0 : (1.0 - g) / (1.0 - p);
}

/* Residual weights (unnormalised) used after the first rejection.
 *   LOSSLESS: [p - q]_+                         [PackedSS] §2.2, Alg. 2
 *   LINEAR:   [ptilde - q]_+                    [TwoTrade] Alg. 1
 *   RATIO:    [p - q]_+  (READING: the lenience changes only the test;
 *             parity unpinned for lam > 1)
 *   CACTUS:   [ptilde - q]_+ with ptilde = c p off the drafted token d and
 *             gamma* on it ([TwoTrade] App. E); c = or_residual_scale().
 *             A rejection implies gamma* < q(d), and c p(d) <= p(d) <= gamma*,
 *             so both ptilde(d) - q(d) and c p(d) - q(d) are negative: the
 *             weight of every id, d included, is [c p - q]_+.
 * p and q are the normalised rows exp(x/Tp - Lp) and exp(y/Tq - Lq); c is
 * the residual scale (1 for the other modes). */
void or_residual_weights(const double *x, const double *y, int V, double Tp, double Tq,
                         double Lp, double Lq, int mode, double lam, double c, double *w)
{
    for (int v = 0; v < V; ++v) {
        double p = exp(x[v] / Tp - Lp);
        double q = exp(y[v] / Tq - Lq);
        double pt = (mode == OR_LINEAR) ? (1.0 - lam) * p + lam * q
                  : (mode == OR_CACTUS) ? c * p
                                        : p;
        double d = pt - q;
        w[v] = d > 0.0 ? d : 0.0;
    }
}

/* Total variation 1 - sum_v min{p_v, q_v}  ([TwoTrade] eq. (1); [SPOT]
 * App. B.2 Step 4). */
double or_tv(const double *x, const double *y, int V, double Tp, double Tq, double Lp, double Lq)
{
    double s = 0.0;
    for (int v = 0; v < V; ++v) {
        double p = exp(x[v] / Tp - Lp);
        double q = exp(y[v] / Tq - Lq);
        s += p < q ? p : q;
    }
    return 1.0 - s;
}

/* ------------------------------------------------------------------------ */
/* State-equality verification of a SPOT draft tree with the target's own    */
/* position selection, [SPOT] App. A.1 ("Position selection", "Greedy        */
/* transition", "Shared Gumbel representation", "State-equality verifier"),  */
/* §4.3 eq. (4).                                                             */
/*   A block state holds L positions, each a token or masked.  The root      */
/*   state's masked positions are the bits of root_mask[b]; tree node n     */
/*   commits token node_tok[n] at the masked position node_pos[n] of its     */
/*   parent's state (parent[b,n] in [-1, n-1], -1 = the root), so its own    */
/*   state has that position filled.  State 0 is the root, state 1 + n the   */
/*   state of node n.                                                        */
/*   state_logits [B, 1+N, L, V]: row (b, state, s) is the target's          */
/*   conditional at that state for position s (read for masked s only).      */
/*   The target's transition Phi(state), for a state with a masked position: */
/*     s* = argmax over masked s of max_v p_s(v), p_s = softmax(row) at      */
/*          temperature 1 (the model's own conditional); lowest s on exact   */
/*          ties (READING of "a fixed deterministic tie-breaking rule");     */
/*     v* = argmax_v row_{s*}(v) at T = 0; at T > 0 the Gumbel-max of        */
/*          row_{s*}/T with the row G(seed, TREE, b, pos_base + s*, 0, .),   */
/*          shared by every state at that absolute position.                 */
/*   A child is accepted when its commitment equals Phi of its parent's      */
/*   state; the verifier walks from the root through accepted children (the */
/*   lowest index among equal children, READING) and commits Phi of the      */
/*   last state reached, unless that state has no masked position left.      */
/* Outputs: path_len, path_nodes [B, max_depth] (-1 padded), commit_count   */
/* (path_len + 1, or path_len at a full block), commit_pos / commit_tok      */
/* (Phi of the last state, -1 at a full block), match [B, N] (the node's     */
/* commitment equals Phi of its parent's state), state_pos / state_tok       */
/* [B, 1+N] (Phi of every state, -1 for a full one; may be NULL), flags [B]: */
/* decisions within 1e-9 over all states (0 < best - runner-up confidence    */
/* < 1e-9 for s*, a Gumbel-max top-two gap below 1e-9 for v*).               */
/* ------------------------------------------------------------------------ */
int or_verify_spot(const void *state_logits, int dtype, int64_t row_stride, int B, int N, int L,
                   int V, const int32_t *parent, const int32_t *node_pos,
                   const int32_t *node_tok, const uint64_t *root_mask, double T, uint64_t seed,
                   const int64_t *pos_base, int32_t *path_len, int32_t *path_nodes, int max_depth,
                   int32_t *commit_count, int32_t *commit_pos, int32_t *commit_tok,
                   uint8_t *match, int32_t *state_pos, int32_t *state_tok, int32_t *flags)
{
    if (L < 1 || L > 64 || N < 0)
        return -1;
    int err = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        const int S = N + 1;
        const uint64_t all = (L == 64) ? ~0ULL : ((1ULL << L) - 1);
        uint64_t *mask = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)S);
        int *ps = (int *)malloc(sizeof(int) * (size_t)S);  /* s* of each state */
        int *pv = (int *)malloc(sizeof(int) * (size_t)S);  /* v* of each state */
        double *x = (double *)malloc(sizeof(double) * (size_t)V);
        const int64_t pos0 = pos_base ? pos_base[b] : 0;
        int nflag = 0;
        /* masked positions of every state */
        mask[0] = root_mask[b] & all;
        for (int n = 0; n < N; ++n) {
            const int par = parent[(int64_t)b * N + n], s = node_pos[(int64_t)b * N + n];
            if (par < -1 || par >= n || s < 0 || s >= L || !((mask[par + 1] >> s) & 1ULL)) {
                err |= 1;
                mask[n + 1] = 0;
                continue;
            }
            mask[n + 1] = mask[par + 1] & ~(1ULL << s);
        }
        /* Phi of every state */
        for (int st = 0; st < S; ++st) {
            ps[st] = pv[st] = -1;
            if (mask[st] == 0)
                continue;
            double c1 = -INFINITY, c2 = -INFINITY;
            for (int s = 0; s < L; ++s) {
                if (!((mask[st] >> s) & 1ULL))
                    continue;
                load_row(state_logits, dtype, ((int64_t)b * S + st) * L + s, row_stride, V, x);
                const double conf = exp(x[or_argmax(x, V)] - or_lse(x, V, 1.0));
                if (conf > c1) {
                    c2 = c1;
                    c1 = conf;
                    ps[st] = s;
                } else if (conf > c2) {
                    c2 = conf;
                }
            }
            if (c1 - c2 > 0.0 && c1 - c2 < OR_FLAG_EPS)
                ++nflag;
            load_row(state_logits, dtype, ((int64_t)b * S + st) * L + ps[st], row_stride, V, x);
            if (T == 0.0) {
                pv[st] = or_argmax(x, V);
            } else {
                double gap;
                for (int v = 0; v < V; ++v)
                    x[v] = x[v] / T;
                pv[st] = or_gumbel_argmax(
                    x, V, or_key(seed, ST_TREE, (uint64_t)b, pos0 + ps[st], 0), &gap);
                if (gap < OR_FLAG_EPS)
                    ++nflag;
            }
        }
        /* match bits; the walk from the root */
        for (int n = 0; n < N; ++n) {
            const int par = parent[(int64_t)b * N + n];
            const int m = par >= -1 && par < n && ps[par + 1] >= 0 &&
                          node_pos[(int64_t)b * N + n] == ps[par + 1] &&
                          node_tok[(int64_t)b * N + n] == pv[par + 1];
            if (match)
                match[(int64_t)b * N + n] = (uint8_t)m;
        }
        for (int k = 0; k < max_depth; ++k)
            path_nodes[(int64_t)b * max_depth + k] = -1;
        int y = -1, len = 0; /* y: the node whose state was reached (-1: root) */
        for (;;) {
            int next = -1;
            for (int n = y + 1; n < N && next < 0; ++n)
                if (parent[(int64_t)b * N + n] == y && ps[y + 1] >= 0 &&
                    node_pos[(int64_t)b * N + n] == ps[y + 1] &&
                    node_tok[(int64_t)b * N + n] == pv[y + 1])
                    next = n;
            if (next < 0)
                break;
            if (len < max_depth)
                path_nodes[(int64_t)b * max_depth + len] = next;
            ++len;
            y = next;
        }
        path_len[b] = len;
        commit_pos[b] = ps[y + 1];
        commit_tok[b] = pv[y + 1];
        commit_count[b] = len + (ps[y + 1] >= 0 ? 1 : 0);
        for (int st = 0; st < S; ++st) {
            if (state_pos) state_pos[(int64_t)b * S + st] = ps[st];
            if (state_tok) state_tok[(int64_t)b * S + st] = pv[st];
        }
        if (flags)
            flags[b] = nflag;
        free(x);
        free(pv);
        free(ps);
        free(mask);
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* One iteration of Packed-SS with any-order greedy decoding, [PackedSS]     */
/* App. C "Procedure", Alg. 3 lines 6-15, eq. (8); confidence scores of       */
/* App. E.6 "Confidence scores".                                             */
/*   The active window U_t holds u <= W unresolved output positions,         */
/*   win_pos[b, 0..u-1] (ascending).  order[b, r] is the index into the      */
/*   window of the position checked at rank r (pi_t, a permutation of        */
/*   0..u-1).  draft[b, i] is the draft token at win_pos[i], or -1 if the    */
/*   position has none.                                                      */
/*   kappa = the number of leading ranks whose position has a draft token.   */
/*   logits [B, Kv + W, V]: verify row r (r < min(kappa+1, u) <= Kv) is the  */
/*   verifier's prediction at rank r, given the drafts of ranks < r;         */
/*   proposal row Kv + i (i < u) is the drafter's row at win_pos[i].         */
/*     v_r = argmax verify row r (eq. 8); h = the leading ranks r < kappa    */
/*     with draft = v_r; A = min(h + 1, u); C = (win_pos[order[r]], v_r),    */
/*     r < A; an accepted EOS at position j lowers the end E to min(E, j),   */
/*     and pairs beyond E are dropped (lines 11-12).                         */
/*     z_i = argmax proposal row i; score_i = its softmax probability at     */
/*     temperature 1 (the probability of the draft token when proposed).     */
/*     Retained positions J: window positions <= E that were not accepted;   */
/*     next_draft[i] = z_i on J, else -1 (line 15).                          */
/*     next_order: the window indices of J by decreasing score, ties by      */
/*     position (App. E.6), -1 padded.                                       */
/* Outputs: accept_len (h), commit_len (pairs kept), commit_pos / commit_tok */
/* [B, W] (rank order, -1 padded), end_out (E), next_draft [B, W], score     */
/* [B, W] (every proposal row i < u; NaN beyond), next_order [B, W].         */
/* ------------------------------------------------------------------------ */
int or_packed_anyorder_step(const void *logits, int dtype, int64_t row_stride, int B, int Kv,
                            int W, int V, const int32_t *u_in, const int32_t *win_pos,
                            const int32_t *order, const int32_t *draft, const int32_t *end_in,
                            int32_t eos_id, int32_t *accept_len, int32_t *commit_len,
                            int32_t *commit_pos, int32_t *commit_tok, int32_t *end_out,
                            int32_t *next_draft, double *score, int32_t *next_order)
{
    if (W < 1 || W > 64 || Kv < 0)
        return -1;
    int err = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        const int R = Kv + W;
        const int u = u_in[b];
        const int32_t *wp = win_pos + (int64_t)b * W, *od = order + (int64_t)b * W;
        const int32_t *dr = draft + (int64_t)b * W;
        double *x = (double *)malloc(sizeof(double) * (size_t)V);
        int seen[64] = {0};
        int bad = u < 0 || u > W;
        for (int r = 0; r < u && !bad; ++r) {
            bad |= od[r] < 0 || od[r] >= u || seen[od[r]];
            if (!bad)
                seen[od[r]] = 1;
        }
        int kappa = 0;
        while (!bad && kappa < u && dr[od[kappa]] >= 0)
            ++kappa;
        const int nreq = (kappa + 1 < u) ? kappa + 1 : u;
        if (bad || nreq > Kv) {
            err |= 1;
            free(x);
            continue;
        }
        /* verifier predictions, rank order (line 7) */
        int v[64];
        for (int r = 0; r < nreq; ++r) {
            load_row(logits, dtype, (int64_t)b * R + r, row_stride, V, x);
            v[r] = or_argmax(x, V);
        }
        /* matches, accepted count (lines 9-10) */
        int h = 0;
        while (h < kappa && dr[od[h]] == v[h])
            ++h;
        const int A = (h + 1 < u) ? h + 1 : u;
        /* the end position E after accepted EOS tokens (line 11) */
        int E = end_in[b];
        for (int r = 0; r < A; ++r)
            if (eos_id >= 0 && v[r] == eos_id && wp[od[r]] < E)
                E = wp[od[r]];
        /* accepted pairs within E, in rank order (lines 12-13) */
        int kept = 0, acc[64] = {0};
        for (int r = 0; r < W; ++r) {
            commit_pos[(int64_t)b * W + r] = -1;
            commit_tok[(int64_t)b * W + r] = -1;
        }
        for (int r = 0; r < A; ++r) {
            if (wp[od[r]] > E)
                continue;
            acc[od[r]] = 1;
            commit_pos[(int64_t)b * W + kept] = wp[od[r]];
            commit_tok[(int64_t)b * W + kept] = v[r];
            ++kept;
        }
        /* proposals and their scores (line 8; App. E.6) */
        double sc[64];
        int z[64];
        for (int i = 0; i < W; ++i) {
            sc[i] = NAN;
            z[i] = -1;
            if (i >= u)
                continue;
            load_row(logits, dtype, (int64_t)b * R + Kv + i, row_stride, V, x);
            z[i] = or_argmax(x, V);
            sc[i] = exp(x[z[i]] - or_lse(x, V, 1.0));
        }
        /* retained draft positions and the next draft (lines 14-15) */
        int nj = 0, jl[64];
        for (int i = 0; i < W; ++i) {
            const int keep = i < u && !acc[i] && wp[i] <= E;
            next_draft[(int64_t)b * W + i] = keep ? z[i] : -1;
            score[(int64_t)b * W + i] = sc[i];
            if (keep)
                jl[nj++] = i;
        }
        /* confidence order of the retained positions: decreasing score, ties
         * by position (insertion sort, stable on the ascending positions) */
        for (int a = 1; a < nj; ++a) {
            const int t = jl[a];
            int c = a - 1;
            while (c >= 0 && sc[jl[c]] < sc[t]) {
                jl[c + 1] = jl[c];
                --c;
            }
            jl[c + 1] = t;
        }
        for (int i = 0; i < W; ++i)
            next_order[(int64_t)b * W + i] = i < nj ? jl[i] : -1;
        accept_len[b] = h;
        commit_len[b] = kept;
        end_out[b] = E;
        free(x);
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Greedy verification, [PackedSS] §3.1 eqs. (1)-(2), Alg. 1 lines 3, 5-6.   */
/* target: [B, K+1, V] rows; draft_ids: [B, K]; draft_len: [B] or NULL (=K). */
/* ------------------------------------------------------------------------ */
int or_verify_greedy(const void *target, int dtype, int64_t row_stride, int B, int K, int V,
                     const int32_t *draft_ids, const int32_t *draft_len,
                     int32_t *accept_len, int32_t *next_token)
{
    int err = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        int n = draft_len ? draft_len[b] : K;
        if (n < 0 || n > K) {
            err |= 1;
            continue;
        }
        double *x = (double *)malloc(sizeof(double) * (size_t)V);
        int h = 0, v_next = -1;
        for (int i = 0; i <= n; ++i) {
            load_row(target, dtype, (int64_t)b * (K + 1) + i, row_stride, V, x);
            int v_i = or_argmax(x, V);
            if (i < n && draft_ids[(int64_t)b * K + i] == v_i) {
                ++h;
                continue;
            }
            v_next = v_i; /* correction at the first mismatch, or bonus */
            break;
        }
        accept_len[b] = h;
        next_token[b] = v_next;
        free(x);
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Speculative sampling with lossless or lenient acceptance.                 */
/* [PackedSS] §2.2 and Alg. 2 lines 5-8; [TwoTrade] §2 and Alg. 1 lines 7-12; */
/* [SPOT] App. B.1 eqs. (13)-(14).                                           */
/*   target [B, K+1, V], draft [B, K, V]; row i of a sequence predicts the   */
/*   token at absolute position pos_base[b] + i.                             */
/*   u_i   = U(seed, ACCEPT, b, pos_base + i, 0, v=0)                        */
/*   next  = Gumbel-max of the residual (SAMPLE stream at the position of    */
/*           the first rejection) or of the bonus row (SAMPLE at pos + n).   */
/* Optional outputs (NULL to skip): p_at/q_at [B,K], lse_p [B,K+1],          */
/* lse_q [B,K], tv [B,K], flags [B].  Rows beyond draft_len get NaN.         */
/* ------------------------------------------------------------------------ */
int or_verify_sample(const void *target, const void *draft, int dtype, int64_t row_stride,
                     int B, int K, int V, const int32_t *draft_ids, const int32_t *draft_len,
                     double Tp, double Tq, int mode, double lam, uint64_t seed,
                     const int64_t *pos_base, int32_t *accept_len, int32_t *next_token,
                     double *p_at, double *q_at, double *lse_p, double *lse_q, double *tv,
                     int32_t *flags)
{
    int err = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        int n = draft_len ? draft_len[b] : K;
        if (n < 0 || n > K) {
            err |= 1;
            continue;
        }
        int64_t pos0 = pos_base ? pos_base[b] : 0;
        double *x = (double *)malloc(sizeof(double) * (size_t)V);
        double *y = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
        int h = 0, rejected = 0, nflag = 0;
        /* per-row quantities for every verify row 0..n (outputs) */
        for (int i = 0; i <= n; ++i) {
            load_row(target, dtype, (int64_t)b * (K + 1) + i, row_stride, V, x);
            double Lp = or_lse(x, V, Tp);
            if (lse_p)
                lse_p[(int64_t)b * (K + 1) + i] = Lp;
            if (i == n)
                break;
            load_row(draft, dtype, (int64_t)b * K + i, row_stride, V, y);
            double Lq = or_lse(y, V, Tq);
            int d = draft_ids[(int64_t)b * K + i];
            if (d < 0 || d >= V) {
                err |= 2;
                break;
            }
            double log_p = x[d] / Tp - Lp, log_q = y[d] / Tq - Lq;
            if (lse_q)
                lse_q[(int64_t)b * K + i] = Lq;
            if (p_at)
                p_at[(int64_t)b * K + i] = exp(log_p);
            if (q_at)
                q_at[(int64_t)b * K + i] = exp(log_q);
            if (tv)
                tv[(int64_t)b * K + i] = or_tv(x, y, V, Tp, Tq, Lp, Lq);
            if (!rejected) {
                /* left-to-right test; only positions up to the first
                 * rejection are reached ([PackedSS] Alg. 2 line 6) */
                double alpha = or_accept_prob(log_p, log_q, mode, lam);
                double u = or_uniform(or_key(seed, ST_ACCEPT, (uint64_t)b, pos0 + i, 0), 0);
                if (fabs(u - alpha) < OR_FLAG_EPS)
                    ++nflag;
                if (u < alpha)
                    ++h;
                else
                    rejected = 1;
            }
        }
        /* rows beyond the sequence's draft are not part of it */
        for (int i = n; i < K; ++i) {
            if (p_at) p_at[(int64_t)b * K + i] = NAN;
            if (q_at) q_at[(int64_t)b * K + i] = NAN;
            if (lse_q) lse_q[(int64_t)b * K + i] = NAN;
            if (tv) tv[(int64_t)b * K + i] = NAN;
            if (lse_p && i + 1 <= K) lse_p[(int64_t)b * (K + 1) + i + 1] = NAN;
        }
        /* correction or bonus ([PackedSS] Alg. 2 line 7) */
        double gap = INFINITY;
        int c;
        load_row(target, dtype, (int64_t)b * (K + 1) + h, row_stride, V, x);
        double Lp = or_lse(x, V, Tp);
        uint64_t key = or_key(seed, ST_SAMPLE, (uint64_t)b, pos0 + h, 0);
        if (h < n) {
            load_row(draft, dtype, (int64_t)b * K + h, row_stride, V, y);
            double Lq = or_lse(y, V, Tq);
            int dh = draft_ids[(int64_t)b * K + h];
            double scale = or_residual_scale(x[dh] / Tp - Lp, mode, lam);
            or_residual_weights(x, y, V, Tp, Tq, Lp, Lq, mode, lam, scale, w);
            for (int v = 0; v < V; ++v)
                w[v] = w[v] > 0.0 ? log(w[v]) : -INFINITY;
            c = or_gumbel_argmax(w, V, key, &gap);
        } else {
            for (int v = 0; v < V; ++v)
                w[v] = x[v] / Tp;
            c = or_gumbel_argmax(w, V, key, &gap);
        }
        if (gap < OR_FLAG_EPS)
            ++nflag;
        accept_len[b] = h;
        next_token[b] = c;
        if (flags)
            flags[b] = nflag;
        free(x);
        free(y);
        free(w);
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Tree verification by state equality, [SPOT] §4.3 and App. A.1 "Draft      */
/* trees", "State-equality verifier"; coupled noise [SPOT] eq. (4).          */
/*   node_logits [B, N, V]: row n is the target conditional, at the state of */
/*   node n's parent, for block position node_pos[n]; the node commits       */
/*   token node_tok[n] there.  parent[b,n] in [-1, n-1] (-1: child of root). */
/*   A node matches when the target's own commitment equals its token:       */
/*     T == 0: argmax_v x_v;                                                 */
/*     T > 0:  argmax_v x_v/T + G(seed, TREE, b, pos_base + node_pos, 0, v)  */
/*   (the Gumbel row is shared by every node at the same absolute position). */
/*   The accepted set is the deepest node whose whole root path matches      */
/*   (READING for ties in depth: smallest node index; parity unpinned).      */
/*   commit_count = path_len + 1: the verifier always commits the target's   */
/*   own transition after the last accepted state.                           */
/* ------------------------------------------------------------------------ */
int or_verify_tree(const void *node_logits, int dtype, int64_t row_stride, int B, int N, int V,
                   const int32_t *parent, const int32_t *node_pos, const int32_t *node_tok,
                   double T, uint64_t seed, const int64_t *pos_base, int32_t *path_len,
                   int32_t *path_nodes, int max_depth, int32_t *commit_count, uint8_t *match,
                   int32_t *flags)
{
    int err = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        int64_t pos0 = pos_base ? pos_base[b] : 0;
        double *x = (double *)malloc(sizeof(double) * (size_t)V);
        int *ok = (int *)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
        int *depth = (int *)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
        int nflag = 0, best = -1;
        for (int n = 0; n < N; ++n) {
            int par = parent[(int64_t)b * N + n];
            int pos = node_pos[(int64_t)b * N + n];
            if (par < -1 || par >= n || pos < 0) {
                err |= 1;
                ok[n] = 0;
                depth[n] = 0;
                continue;
            }
            load_row(node_logits, dtype, (int64_t)b * N + n, row_stride, V, x);
            int win;
            if (T == 0.0) {
                win = or_argmax(x, V);
            } else {
                double gap;
                for (int v = 0; v < V; ++v)
                    x[v] = x[v] / T;
                win = or_gumbel_argmax(x, V, or_key(seed, ST_TREE, (uint64_t)b, pos0 + pos, 0), &gap);
                if (gap < OR_FLAG_EPS)
                    ++nflag;
            }
            int m = (win == node_tok[(int64_t)b * N + n]);
            if (match)
                match[(int64_t)b * N + n] = (uint8_t)m;
            ok[n] = m && (par < 0 || ok[par]);
            depth[n] = (par < 0) ? 1 : depth[par] + 1;
            if (ok[n] && (best < 0 || depth[n] > depth[best]))
                best = n;
        }
        int len = best < 0 ? 0 : depth[best];
        path_len[b] = len;
        commit_count[b] = len + 1;
        for (int k = 0; k < max_depth; ++k)
            path_nodes[(int64_t)b * max_depth + k] = -1;
        for (int n = best, d = len; n >= 0; n = parent[(int64_t)b * N + n], --d)
            if (d - 1 < max_depth)
                path_nodes[(int64_t)b * max_depth + d - 1] = n;
        if (flags)
            flags[b] = nflag;
        free(x);
        free(ok);
        free(depth);
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* One Packed-SS iteration, [PackedSS] §3.1 Alg. 1 (T == 0) and §3.2 Alg. 2  */
/* (T > 0).                                                                  */
/*   logits [B, K+W, V]: rows 0..K-1 verify rows (row i predicts absolute    */
/*   position pos_base + i), rows K..K+W-1 drafter rows for positions        */
/*   pos_base + j (draft, verifier and proposal share columns, Fig. 2).      */
/*   prev_draft [B, K-1], prev_len [B] <= K-1: the draft D_{t-1}.            */
/*   T > 0: prev_q_at_draft [B, K-1] holds Q_{t-1}(d) for each draft token;  */
/*   prev_draft_logits [B, W, V] are the previous call's drafter rows and    */
/*   prev_q_offset [B] = a_{t-1}, so Q_{t-1}^(i) is row a_{t-1} + i - 1      */
/*   (Alg. 2 line 12: Q_t^(j) = q_t^(a+j)).                                  */
/*   Stopping index a = min({A, remaining} ∪ {i : C_i = EOS}) (Alg. 1 l. 7). */
/*   Next draft (z_{a+1}, ..., z_W) (eq. (4)); drafts at T > 0 are Gumbel-max */
/*   samples keyed by the call index iter (DRAFT stream).                    */
/*   confidence_j = max_v softmax(y_j)_v at temperature 1 (READING).          */
/* ------------------------------------------------------------------------ */
int or_packed_step(const void *logits, int dtype, int64_t row_stride, int B, int K, int W, int V,
                   const int32_t *prev_draft, const int32_t *prev_len, const float *prev_q_at_draft,
                   const void *prev_draft_logits, const int32_t *prev_q_offset, double T,
                   uint64_t seed, uint64_t iter, const int64_t *pos_base, int32_t eos_id,
                   const int32_t *remaining, int32_t *accept_len, int32_t *commit_len,
                   int32_t *committed, int32_t *next_draft, int32_t *next_len,
                   double *next_q_at_draft, double *confidence, int32_t *flags)
{
    int err = 0;
    int R = K + W;
#pragma omp parallel for schedule(dynamic) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        int64_t pos0 = pos_base ? pos_base[b] : 0;
        int n = prev_len[b];
        int off = prev_q_offset ? prev_q_offset[b] : 0;
        if (n < 0 || n > K - 1 || (T > 0.0 && (off < 0 || off + n > W))) {
            err |= 1;
            continue;
        }
        double *x = (double *)malloc(sizeof(double) * (size_t)V);
        double *y = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
        int32_t *C = (int32_t *)malloc(sizeof(int32_t) * (size_t)K);
        int32_t *z = (int32_t *)malloc(sizeof(int32_t) * (size_t)W);
        double *qz = (double *)malloc(sizeof(double) * (size_t)W);
        int h = 0, c = -1, nflag = 0;
        double gap = INFINITY;

        /* ---- verification of D_{t-1} ---- */
        if (T == 0.0) {
            for (int i = 0; i <= n; ++i) {
                load_row(logits, dtype, (int64_t)b * R + i, row_stride, V, x);
                int v_i = or_argmax(x, V);
                if (i < n && prev_draft[(int64_t)b * (K - 1) + i] == v_i) {
                    ++h;
                    continue;
                }
                c = v_i;
                break;
            }
        } else {
            int rejected = 0;
            for (int i = 0; i < n && !rejected; ++i) {
                int d = prev_draft[(int64_t)b * (K - 1) + i];
                if (d < 0 || d >= V) {
                    err |= 2;
                    break;
                }
                load_row(logits, dtype, (int64_t)b * R + i, row_stride, V, x);
                double Lp = or_lse(x, V, T);
                double log_p = x[d] / T - Lp;
                double log_q = log((double)prev_q_at_draft[(int64_t)b * (K - 1) + i]);
                double alpha = or_accept_prob(log_p, log_q, OR_LOSSLESS, 0.0);
                double u = or_uniform(or_key(seed, ST_ACCEPT, (uint64_t)b, pos0 + i, 0), 0);
                if (fabs(u - alpha) < OR_FLAG_EPS)
                    ++nflag;
                if (u < alpha)
                    ++h;
                else
                    rejected = 1;
            }
            uint64_t key = or_key(seed, ST_SAMPLE, (uint64_t)b, pos0 + h, 0);
            load_row(logits, dtype, (int64_t)b * R + h, row_stride, V, x);
            double Lp = or_lse(x, V, T);
            if (h < n) {
                /* correction from [p - Q]_+ with the stored proposal row */
                load_row(prev_draft_logits, dtype, (int64_t)b * W + off + h, row_stride, V, y);
                double Lq = or_lse(y, V, T);
                or_residual_weights(x, y, V, T, T, Lp, Lq, OR_LOSSLESS, 0.0, 1.0, w);
                for (int v = 0; v < V; ++v)
                    w[v] = w[v] > 0.0 ? log(w[v]) : -INFINITY;
            } else {
                for (int v = 0; v < V; ++v)
                    w[v] = x[v] / T;
            }
            c = or_gumbel_argmax(w, V, key, &gap);
            if (gap < OR_FLAG_EPS)
                ++nflag;
        }
        for (int i = 0; i < h; ++i)
            C[i] = prev_draft[(int64_t)b * (K - 1) + i];
        C[h] = c;
        int A = h + 1;
        int a = A;
        if (remaining && remaining[b] < a)
            a = remaining[b] < 0 ? 0 : remaining[b];
        if (eos_id >= 0)
            for (int i = 0; i < A; ++i)
                if (C[i] == eos_id) {
                    if (i + 1 < a)
                        a = i + 1;
                    break;
                }

        /* ---- drafting Z_t from the same call ---- */
        for (int j = 0; j < W; ++j) {
            load_row(logits, dtype, (int64_t)b * R + K + j, row_stride, V, y);
            double L1 = or_lse(y, V, 1.0);
            int zm = or_argmax(y, V);
            if (confidence)
                confidence[(int64_t)b * W + j] = exp(y[zm] - L1);
            if (T == 0.0) {
                z[j] = zm;
                qz[j] = 1.0;
            } else {
                double LT = or_lse(y, V, T);
                for (int v = 0; v < V; ++v)
                    w[v] = y[v] / T;
                double g;
                z[j] = or_gumbel_argmax(w, V, or_key(seed, ST_DRAFT, (uint64_t)b, pos0 + j, iter), &g);
                qz[j] = exp(y[z[j]] / T - LT);
                if (j >= a && g < OR_FLAG_EPS)
                    ++nflag;
            }
        }

        accept_len[b] = h;
        commit_len[b] = a;
        for (int i = 0; i < K; ++i)
            committed[(int64_t)b * K + i] = i < a ? C[i] : -1;
        int nl = W - a > 0 ? W - a : 0;
        next_len[b] = nl;
        for (int j = 0; j < W; ++j) {
            next_draft[(int64_t)b * W + j] = j < nl ? z[a + j] : -1;
            if (next_q_at_draft)
                next_q_at_draft[(int64_t)b * W + j] = j < nl ? qz[a + j] : NAN;
        }
        if (flags)
            flags[b] = nflag;
        free(x);
        free(y);
        free(w);
        free(C);
        free(z);
        free(qz);
    }
    return err ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Packed-SS with top-k truncated distributions ([PackedSS] §3.2, last       */
/* paragraph: with top-k truncation only the nonzero entries of the stored   */
/* drafter distribution Q need to be kept; Alg. 2 otherwise unchanged).      */
/*   READING: top-k of a row keeps its k largest logits (ties to the lowest  */
/*   id) and renormalises softmax(x/T) over them.  Both sides are truncated, */
/*   as in a sampler that applies top-k to the verifier (the AR mode whose   */
/*   law the step preserves, Thm. 3.3) and to the drafter: the target p of   */
/*   verify rows keeps kp entries, the drafter Q of proposal rows kq.        */
/*   The previous call's Q rows arrive as (id, probability) lists:           */
/*   prev_q_ids / prev_q_probs [B, W, kq] (ids -1 padded); Q_{t-1}^(i) is    */
/*   list prev_q_offset[b] + i (Alg. 2 line 12).                             */
/*   Verify position i < prev_len: accept d_i w.p. min{1, p(d_i)/Q(d_i)},    */
/*   p(d) = 0 off its support; d_i must be in its list.  First rejection h:  */
/*   the correction is the Gumbel-max over v with [p(v) - Q(v)]_+ > 0 of     */
/*   log [p(v) - Q(v)]_+ + G(SAMPLE, b, pos + h); all accepted: the bonus is  */
/*   the Gumbel-max of x/T + G over the support of p.  Proposal j: z_j the   */
/*   Gumbel-max of y_j/T + G(DRAFT, b, pos + j, iter) over the top-kq ids,   */
/*   and the list (ids by logit desc, id asc; probabilities) is written to   */
/*   q_ids / q_probs [B, W, kq] for the next call.                           */
/*   Stopping, committed tokens and the shift of the next draft are those of */
/*   or_packed_step.  T > 0.                                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    double x;
    int32_t v;
} or_entry;

/* Larger logit first; equal logits: lower id first. */
static int or_entry_cmp(const void *a, const void *b)
{
    const or_entry *p = (const or_entry *)a, *q = (const or_entry *)b;
    if (p->x != q->x)
        return p->x > q->x ? -1 : 1;
    return p->v < q->v ? -1 : (p->v > q->v ? 1 : 0);
}

/* The k largest entries of x[0..V-1] (ties to the lowest id), in that order
 * (a full sort of the row, then its first k). */
void or_topk(const double *x, int V, int k, int32_t *ids)
{
    or_entry *e = (or_entry *)malloc(sizeof(or_entry) * (size_t)V);
    for (int v = 0; v < V; ++v) {
        e[v].x = x[v];
        e[v].v = v;
    }
    qsort(e, (size_t)V, sizeof(or_entry), or_entry_cmp);
    for (int m = 0; m < k; ++m)
        ids[m] = e[m].v;
    free(e);
}

/* log of the sum over the k listed ids of exp(x/T): m + log(sum exp(z - m)). */
static double or_lse_list(const double *x, const int32_t *ids, int k, double T)
{
    double m = -INFINITY, s = 0.0;
    for (int i = 0; i < k; ++i)
        if (x[ids[i]] / T > m)
            m = x[ids[i]] / T;
    for (int i = 0; i < k; ++i)
        s += exp(x[ids[i]] / T - m);
    return m + log(s);
}

/* Probability of v in a stored list (0 when absent). */
static double or_list_prob(const int32_t *ids, const float *probs, int k, int v)
{
    for (int i = 0; i < k; ++i)
        if (ids[i] == v)
            return (double)probs[i];
    return 0.0;
}

int or_packed_topk_step(const void *logits, int dtype, int64_t row_stride, int B, int K, int W,
                        int V, int kp, int kq, const int32_t *prev_draft,
                        const int32_t *prev_len, const int32_t *prev_q_ids,
                        const float *prev_q_probs, const int32_t *prev_q_offset, double T,
                        uint64_t seed, uint64_t iter, const int64_t *pos_base, int32_t eos_id,
                        const int32_t *remaining, int32_t *accept_len, int32_t *commit_len,
                        int32_t *committed, int32_t *next_draft, int32_t *next_len,
                        double *next_q_at_draft, int32_t *q_ids, double *q_probs,
                        int32_t *flags)
{
    if (!(T > 0.0) || kp < 1 || kp > V || kq < 1 || kq > V)
        return -1;
    int err = 0;
    int R = K + W;
#pragma omp parallel for schedule(dynamic) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        int64_t pos0 = pos_base ? pos_base[b] : 0;
        int n = prev_len[b];
        int off = prev_q_offset ? prev_q_offset[b] : 0;
        if (n < 0 || n > K - 1 || off < 0 || off + n > W) {
            err |= 1;
            continue;
        }
        double *x = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
        int32_t *S = (int32_t *)malloc(sizeof(int32_t) * (size_t)(kp > kq ? kp : kq));
        int32_t *C = (int32_t *)malloc(sizeof(int32_t) * (size_t)K);
        int32_t *z = (int32_t *)malloc(sizeof(int32_t) * (size_t)W);
        double *qz = (double *)malloc(sizeof(double) * (size_t)W);
        int h = 0, nflag = 0, bad = 0;
        double gap = INFINITY;

        /* ---- verification of D_{t-1} against the truncated target ---- */
        int rejected = 0;
        for (int i = 0; i < n && !rejected; ++i) {
            int d = prev_draft[(int64_t)b * (K - 1) + i];
            const int32_t *qi = prev_q_ids + ((int64_t)b * W + off + i) * kq;
            const float *qp = prev_q_probs + ((int64_t)b * W + off + i) * kq;
            double Qd = (d >= 0 && d < V) ? or_list_prob(qi, qp, kq, d) : 0.0;
            if (!(Qd > 0.0)) {
                bad = 1;  /* the draft is not in the list it was drawn from */
                break;
            }
            load_row(logits, dtype, (int64_t)b * R + i, row_stride, V, x);
            or_topk(x, V, kp, S);
            double L = or_lse_list(x, S, kp, T);
            double log_p = -INFINITY;
            for (int m = 0; m < kp; ++m)
                if (S[m] == d)
                    log_p = x[d] / T - L;
            double alpha = or_accept_prob(log_p, log(Qd), OR_LOSSLESS, 0.0);
            double u = or_uniform(or_key(seed, ST_ACCEPT, (uint64_t)b, pos0 + i, 0), 0);
            if (fabs(u - alpha) < OR_FLAG_EPS)
                ++nflag;
            if (u < alpha)
                ++h;
            else
                rejected = 1;
        }
        if (bad) {
            err |= 2;
            free(x), free(w), free(S), free(C), free(z), free(qz);
            continue;
        }
        load_row(logits, dtype, (int64_t)b * R + h, row_stride, V, x);
        or_topk(x, V, kp, S);
        double L = or_lse_list(x, S, kp, T);
        for (int v = 0; v < V; ++v)
            w[v] = -INFINITY;
        if (h < n) {
            /* correction from [p - Q]_+ over the support of p */
            const int32_t *qi = prev_q_ids + ((int64_t)b * W + off + h) * kq;
            const float *qp = prev_q_probs + ((int64_t)b * W + off + h) * kq;
            for (int m = 0; m < kp; ++m) {
                int v = S[m];
                double r = exp(x[v] / T - L) - or_list_prob(qi, qp, kq, v);
                if (r > 0.0)
                    w[v] = log(r);
            }
        } else {
            for (int m = 0; m < kp; ++m)
                w[S[m]] = x[S[m]] / T;
        }
        int c = or_gumbel_argmax(w, V, or_key(seed, ST_SAMPLE, (uint64_t)b, pos0 + h, 0), &gap);
        if (gap < OR_FLAG_EPS)
            ++nflag;
        for (int i = 0; i < h; ++i)
            C[i] = prev_draft[(int64_t)b * (K - 1) + i];
        C[h] = c;
        int A = h + 1;
        int a = A;
        if (remaining && remaining[b] < a)
            a = remaining[b] < 0 ? 0 : remaining[b];
        if (eos_id >= 0)
            for (int i = 0; i < A; ++i)
                if (C[i] == eos_id) {
                    if (i + 1 < a)
                        a = i + 1;
                    break;
                }

        /* ---- drafting Z_t from the truncated drafter rows ---- */
        for (int j = 0; j < W; ++j) {
            load_row(logits, dtype, (int64_t)b * R + K + j, row_stride, V, x);
            or_topk(x, V, kq, S);
            double Lq = or_lse_list(x, S, kq, T);
            for (int v = 0; v < V; ++v)
                w[v] = -INFINITY;
            for (int m = 0; m < kq; ++m) {
                w[S[m]] = x[S[m]] / T;
                q_ids[((int64_t)b * W + j) * kq + m] = S[m];
                q_probs[((int64_t)b * W + j) * kq + m] = exp(x[S[m]] / T - Lq);
            }
            double g;
            z[j] = or_gumbel_argmax(w, V, or_key(seed, ST_DRAFT, (uint64_t)b, pos0 + j, iter), &g);
            qz[j] = exp(x[z[j]] / T - Lq);
            if (j >= a && g < OR_FLAG_EPS)
                ++nflag;
        }

        accept_len[b] = h;
        commit_len[b] = a;
        for (int i = 0; i < K; ++i)
            committed[(int64_t)b * K + i] = i < a ? C[i] : -1;
        int nl = W - a > 0 ? W - a : 0;
        next_len[b] = nl;
        for (int j = 0; j < W; ++j) {
            next_draft[(int64_t)b * W + j] = j < nl ? z[a + j] : -1;
            if (next_q_at_draft)
                next_q_at_draft[(int64_t)b * W + j] = j < nl ? qz[a + j] : NAN;
        }
        if (flags)
            flags[b] = nflag;
        free(x), free(w), free(S), free(C), free(z), free(qz);
    }
    return err ? -1 : 0;
}

/* Number of threads the parallel loops above use (for reporting). */
int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
