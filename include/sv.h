/*
 * sv.h -- draft-block verification on NVIDIA GB300 (sm_103a): C ABI of libsv.so.
 *
 * Sources the operations follow (cited by short name):
 *   [PackedSS] "One Call Ahead: Packed Self-Speculative Decoding with Diffusion
 *              Drafting"
 *   [SPOT]     "On the SPOT: Enhancing Speculative Decoding for Diffusion
 *              Language Models via Commit-Order Prediction"
 *   [TwoTrade] "Speculative Diffusion is a Tale of Two Tradeoffs"
 *
 * Conventions shared by every call
 * ---------------------------------
 * - Tensor pointers are DEVICE pointers owned by the caller; they must stay
 *   valid until the stream has executed the call.  Logit tensors are row-major
 *   with the vocabulary fastest; consecutive rows are row_stride elements
 *   apart.  Logit base pointers must be 16-byte aligned and row_stride * the
 *   element size a multiple of 16 bytes; V must be a multiple of 8 (bf16) or
 *   4 (fp32).  Logits must be finite.
 * - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *   default stream) and never synchronises the host.  The return value
 *   reports only host-detectable problems (bad arguments, launch failures).
 *   Problems found on the device (an out-of-range token id, node position or
 *   parent; a bounded wait that expired) are latched in the handle and
 *   returned by sv_sync_status().
 * - Integer outputs are int32; accept lengths count draft tokens.  Float
 *   outputs are fp32; entries that do not exist for a sequence (beyond its
 *   draft length) are written as NaN (floats) or -1 (token ids).
 * - Random numbers come from a counter-based generator: a row key
 *   k = key(seed, stream, sequence b, absolute position, call index) seeds a
 *   SplitMix64 stream; every uniform u(k, v) of the row (vocabulary id v) is
 *   read from that stream, and G(k, v) = -log(-log u).  Which ids land in
 *   the top 1/256 of (0, 1) is an i.i.d. Bernoulli(1/256) process drawn by
 *   geometric skipping in blocks of 256 ids; 52 fine bits m per id place u
 *   at w * 255/256 (other ids) or 1 - (1 - w)/256 (top ids), w =
 *   (2m + 1) / 2^53.  Streams: ACCEPT = 1 (acceptance uniforms, v = 0),
 *   SAMPLE = 2 (corrections and bonus tokens), DRAFT = 3 (Packed-SS
 *   proposals, keyed by the call index), TREE = 4 (coupled noise shared by
 *   every tree node at the same absolute position).  The layout is fixed:
 *   equal arguments give equal results on any GB300.
 * - Decisions are exact with respect to fp64 arithmetic on the upcast logits:
 *   the kernels decide in fp32 with a proved error bound and recompute in
 *   fp64 whenever a decision falls inside that bound.  A decision whose fp64
 *   value lies within 1e-9 of its threshold (|u - alpha| < 1e-9, or a
 *   Gumbel-max winner less than 1e-9 ahead of the runner-up) is counted in
 *   the optional `flags` output.
 * - K (draft tokens), W (packed width) <= 32; N (tree nodes) <= 64.
 * - Fault injection for tests of a caller's failure handling: the
 *   environment variable SV_FAULT_INJECT="call:code[,call:code...]" makes
 *   each listed entry point (sv_create, sv_verify_greedy,
 *   sv_verify_greedy_static, sv_verify_sample, sv_verify_tree,
 *   sv_verify_spot, sv_packed_step, sv_packed_topk_step,
 *   sv_packed_anyorder_step) return the
 *   status `code` (1..6) at its launch point,
 *   after its argument checks and before anything is enqueued.  It is read
 *   at every call; unset, nothing is injected.
 */
#ifndef SV_H
#define SV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,   /* rejected on the host; nothing was enqueued */
    SV_ERR_CUDA = 2,          /* a CUDA runtime call failed */
    SV_ERR_OOM = 3,           /* workspace allocation failed */
    SV_ERR_TIMEOUT = 4,       /* a bounded device wait expired (latched) */
    SV_ERR_UNSUPPORTED = 5,   /* no sm_103 device, or shape beyond limits */
    SV_ERR_DEVICE_BOUNDS = 6  /* id / position / parent out of range (latched) */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Acceptance rules of sv_verify_sample. */
typedef enum {
    SV_LOSSLESS = 0,       /* accept w.p. min{1, p(d)/q(d)}; residual [p-q]_+
                              ([PackedSS] §2.2, Alg. 2; [SPOT] App. B eqs. 13-14) */
    SV_LENIENT_RATIO = 1,  /* accept w.p. min{1, lam p(d)/q(d)}, lam >= 1;
                              residual [p-q]_+ (the "predefined ratio" lenience
                              named in [TwoTrade] §1) */
    SV_LENIENT_LINEAR = 2, /* target ptilde = (1-lam) p + lam q, lam in [0,1]:
                              accept w.p. min{1, ptilde(d)/q(d)}, residual
                              [ptilde-q]_+ ([TwoTrade] eq. 5, Alg. 1) */
    SV_LENIENT_CACTUS = 3  /* modified Cactus, KL budget delta = lam >= 0:
                              gamma* = the largest gamma with
                              gamma log(gamma/p(d)) + (1-gamma)
                              log((1-gamma)/(1-p(d))) <= delta (solved by
                              Newton's method); accept w.p.
                              min{1, gamma* / q(d)}; residual [c p - q]_+ with
                              c = (1-gamma*)/(1-p(d)) ([TwoTrade] App. E,
                              eq. 17); delta = 0 is the lossless rule */
} sv_accept_mode;

typedef struct sv_handle sv_handle;

/* Create a handle on the current CUDA device.  It owns a device workspace and
 * a device error word; the workspace grows (stream-ordered) when a call needs
 * more.  Errors: SV_ERR_INVALID_ARG (h == NULL), SV_ERR_UNSUPPORTED (no
 * device), SV_ERR_OOM, SV_ERR_CUDA. */
sv_status sv_create(sv_handle **h);

/* Synchronise the device and free the handle's memory.  NULL is a no-op. */
sv_status sv_destroy(sv_handle *h);

/* Synchronise `stream`, return the first device-side error latched since the
 * last call of this function (or SV_OK), and clear it. */
sv_status sv_sync_status(sv_handle *h, void *stream);

/* Static description of a status code. */
const char *sv_status_string(sv_status s);

/* Number of sequences whose decisions were recomputed on the fp64 path by the
 * calls since the last sv_sync_status (synchronises `stream`). */
sv_status sv_rescue_count(sv_handle *h, void *stream, int64_t *count);

/* ---------------------------------------------------------------------------
 * Greedy verification -- [PackedSS] §3.1 eqs. (1)-(2); [SPOT] Prop. 1.
 *   target     [B, K+1, V] logits: row i of sequence b is the target's
 *              conditional after the prefix and draft tokens d_0..d_{i-1}.
 *   draft_ids  [B, K] int32 draft tokens.
 *   draft_len  [B] int32 in [0, K], or NULL (every sequence has K drafts).
 *   accept_len [B] out: h = number of leading drafts equal to argmax_v x_{i,v}
 *              (lowest id wins ties).
 *   next_token [B] out: argmax of row h (correction, or bonus when h = n).
 * Only rows 0..h of each sequence are needed; rows beyond draft_len are not
 * read.
 * ------------------------------------------------------------------------- */
sv_status sv_verify_greedy(sv_handle *h, const void *target, sv_dtype dtype, int64_t row_stride,
                           int B, int K, int V, const int32_t *draft_ids,
                           const int32_t *draft_len, int32_t *accept_len, int32_t *next_token,
                           void *stream);

/* ---------------------------------------------------------------------------
 * Greedy verification without any device allocation.  The papers have no
 * counterpart: this is a deployment variant of sv_verify_greedy, same inputs,
 * outputs and results, for callers that cannot let a library allocate device
 * memory -- a serving engine that reserves all free memory for its own pools
 * (a KV cache, say) up front, or a memory-capped process in which an
 * allocation in the middle of a step could fail or stall on the allocator.
 * No handle: the scratch is one fixed device array of about 2.1 MB per device
 * that ships with the library.
 *   status [1] int32, device, out: written 0 at the start of the call (in
 *          stream order), then the first device-side error (SV_ERR_TIMEOUT,
 *          SV_ERR_DEVICE_BOUNDS) if one occurs.  Nothing else needs to start
 *          at zero: the call clears its own counters.
 * B = 0 only writes 0 to status (the logit and id pointers may be NULL).
 * Limits: B <= 4096 and B * (K + 1) <= 32768; larger shapes return
 * SV_ERR_UNSUPPORTED with nothing enqueued.  Other argument errors return
 * SV_ERR_INVALID_ARG as in sv_verify_greedy.
 * Calls on one device share the scratch and must not overlap: issue them on
 * one stream, or order the streams with events.  The first call on a device
 * looks up the scratch and sets kernel attributes; make it before any stream
 * capture.  If that set-up fails with a CUDA error the call returns
 * SV_ERR_CUDA and the next call on the device tries the set-up again.
 * ------------------------------------------------------------------------- */
sv_status sv_verify_greedy_static(const void *target, sv_dtype dtype, int64_t row_stride, int B,
                                  int K, int V, const int32_t *draft_ids,
                                  const int32_t *draft_len, int32_t *accept_len,
                                  int32_t *next_token, int32_t *status, void *stream);

/* ---------------------------------------------------------------------------
 * Speculative sampling: lossless, ratio-lenient or linear-lenient acceptance
 * ([PackedSS] §2.2 and Alg. 2; [TwoTrade] §2 and Alg. 1; [SPOT] App. B).
 *   target [B, K+1, V], draft [B, K, V]: logits of the target p and the
 *   drafter q; p_i = softmax(x_i / T_p), q_i = softmax(y_i / T_q), T_p, T_q > 0
 *   (temperature law of [SPOT] eq. 2).  Row i predicts the token at absolute
 *   position pos_base[b] + i (pos_base NULL = 0).
 *   Test i (left to right, stopping at the first rejection):
 *     u_i = u(key(seed, ACCEPT, b, pos_base + i, 0), 0);  accept iff u_i < alpha_i.
 *   Correction at the first rejection h < n: Gumbel-max over the residual
 *   weights with key (seed, SAMPLE, b, pos_base + h, 0); bonus when all n are
 *   accepted: Gumbel-max of x_n / T_p with key (seed, SAMPLE, b, pos_base + n, 0).
 *   lam: lambda >= 1 for SV_LENIENT_RATIO, mu in [0,1] for SV_LENIENT_LINEAR,
 *   the KL budget delta >= 0 for SV_LENIENT_CACTUS, ignored for SV_LOSSLESS.
 * Outputs (NULL to skip the optional ones):
 *   accept_len [B], next_token [B];
 *   p_at_draft, q_at_draft [B, K]: p_i(d_i), q_i(d_i);
 *   lse_p [B, K+1], lse_q [B, K]: log-sum-exp of x / T_p and y / T_q;
 *   tv [B, K]: total variation 1 - sum_v min(p_i, q_i) ([TwoTrade] eq. 1);
 *     asking for it adds a second streaming pass over every (p, q) row pair;
 *   flags [B]: near-threshold decisions (see the conventions).
 * ------------------------------------------------------------------------- */
sv_status sv_verify_sample(sv_handle *h, const void *target, const void *draft, sv_dtype dtype,
                           int64_t row_stride, int B, int K, int V, const int32_t *draft_ids,
                           const int32_t *draft_len, float T_p, float T_q, sv_accept_mode mode,
                           float lam, uint64_t seed, const int64_t *pos_base,
                           int32_t *accept_len, int32_t *next_token, float *p_at_draft,
                           float *q_at_draft, float *lse_p, float *lse_q, float *tv,
                           int32_t *flags, void *stream);

/* ---------------------------------------------------------------------------
 * Coupled-noise state-equality verification of draft trees
 * ([SPOT] §4.3 eq. 4; App. A.1 "Draft trees", "State-equality verifier").
 *   node_logits [B, N, V]: row n is the target's conditional, at the state of
 *     node n's parent, for the block position node_pos[b, n].
 *   parent [B, N] in [-1, n-1] (-1 = child of the root); node_pos [B, N] >= 0
 *     (block position; its absolute position is pos_base[b] + node_pos);
 *   node_tok [B, N] the token node n commits.
 *   Node n matches iff node_tok = argmax_v x_v (T = 0), or
 *     argmax_v x_v / T + G(key(seed, TREE, b, pos_base + node_pos, 0), v) (T > 0).
 *   path_len [B] out: depth of the deepest node whose whole root path matches
 *     (0 if none; ties between equally deep nodes go to the smaller index).
 *   path_nodes [B, max_depth] out: that path from the root side, -1 padded.
 *   commit_count [B] out: path_len + 1 (the verifier's own transition after
 *     the last accepted state is always committed).
 *   match [B, N] out (optional, uint8): per-node match bit.
 *   flags [B] out (optional): nodes whose Gumbel-max winner is < 1e-9 ahead.
 * ------------------------------------------------------------------------- */
sv_status sv_verify_tree(sv_handle *h, const void *node_logits, sv_dtype dtype, int64_t row_stride,
                         int B, int N, int V, const int32_t *parent, const int32_t *node_pos,
                         const int32_t *node_tok, float T, uint64_t seed,
                         const int64_t *pos_base, int32_t *path_len, int32_t *path_nodes,
                         int max_depth, int32_t *commit_count, uint8_t *match, int32_t *flags,
                         void *stream);

/* ---------------------------------------------------------------------------
 * SPOT verification with the target's own position selection ([SPOT] App.
 * A.1 "Position selection", "Greedy transition", "Shared Gumbel
 * representation", "State-equality verifier"; §4.3 eq. 4).
 *   A block state has L <= 32 positions, each holding a token or masked.
 *   root_mask [B] (uint64, device): bit s set = position s is masked in the
 *     root state (bits at or above L are ignored).
 *   parent [B, N] in [-1, n-1] (-1 = the root), node_pos [B, N], node_tok
 *     [B, N] (N <= 64; may be NULL when N = 0): node n commits token
 *     node_tok at position node_pos, which must be masked in its parent's
 *     state; the node's own state has it filled.  State 0 is the root,
 *     state 1 + n the state of node n.
 *   state_logits [B, 1+N, L, V]: row (b, state, s) is the target's
 *     conditional at that state for position s.  Only rows of masked
 *     positions are read.
 *   The target's transition Phi(state): s* = the masked position with the
 *     largest max_v softmax(row)_v (the model's own probabilities, at
 *     temperature 1; lowest position on exact ties), then the token
 *     argmax_v row_{s*} (T = 0) or argmax_v row_{s*}/T + G(key(seed, TREE,
 *     b, pos_base + s*, 0), v) (T > 0: the noise row of an absolute position
 *     is shared by every state).
 *   A child is accepted when its commitment equals Phi of its parent's
 *   state; the walk from the root follows accepted children (the lowest
 *   index among equal children) and then commits Phi of the state reached.
 * Outputs: path_len [B] (accepted nodes), path_nodes [B, max_depth] (-1
 *   padded), commit_count [B] (path_len + 1, or path_len when the state
 *   reached has nothing masked), commit_pos / commit_tok [B] (Phi of the
 *   state reached; -1 when nothing is masked), match [B, N] (optional,
 *   uint8: the node equals Phi of its parent's state), state_pos /
 *   state_tok [B, 1+N] (optional: Phi of every state, -1 where nothing is
 *   masked), flags [B] (optional: decisions within 1e-9 -- a confidence
 *   runner-up less than 1e-9 behind s*, or a Gumbel-max top-two gap below
 *   1e-9 -- over all states).
 * Errors: SV_ERR_INVALID_ARG (shapes, L > 32, N > 64, T < 0); latched
 *   SV_ERR_DEVICE_BOUNDS for a parent out of range or a position that is
 *   not masked in the parent's state.
 * ------------------------------------------------------------------------- */
sv_status sv_verify_spot(sv_handle *h, const void *state_logits, sv_dtype dtype,
                         int64_t row_stride, int B, int N, int L, int V, const int32_t *parent,
                         const int32_t *node_pos, const int32_t *node_tok,
                         const uint64_t *root_mask, float T, uint64_t seed,
                         const int64_t *pos_base, int32_t *path_len, int32_t *path_nodes,
                         int max_depth, int32_t *commit_count, int32_t *commit_pos,
                         int32_t *commit_tok, uint8_t *match, int32_t *state_pos,
                         int32_t *state_tok, int32_t *flags, void *stream);

/* ---------------------------------------------------------------------------
 * One Packed-SS iteration: verify the previous draft and propose the next
 * block from the same model call ([PackedSS] §3.1 Alg. 1, §3.2 Alg. 2).
 *   logits [B, K+W, V]: rows 0..K-1 are verify rows (row i predicts absolute
 *     position pos_base[b] + i), rows K..K+W-1 are drafter rows for positions
 *     pos_base[b] + j (draft, verifier and proposal share columns, Fig. 2).
 *   prev_draft [B, K-1] (may be NULL when K == 1), prev_len [B] in [0, K-1].
 *   T == 0: greedy (Alg. 1).  T > 0: rejection sampling with the stored
 *     proposal (Alg. 2):
 *     prev_q_at_draft [B, K-1]  Q_{t-1}(d_i) of every draft token (NULL
 *       allowed when K == 1);
 *     prev_draft_logits [B, W, V] the previous call's drafter rows;
 *     prev_q_offset [B]  a_{t-1}: Q_{t-1}^(i) is row a_{t-1} + i of them
 *       (Alg. 2 line 12), so a_{t-1} + prev_len <= W.
 *   Stopping index a = min({h+1, remaining[b]} ∪ {i : C_i = eos_id})
 *     (Alg. 1 line 7; remaining NULL = no cap, eos_id < 0 = no EOS).
 *   Proposals: z_j = argmax (T = 0) or Gumbel-max of y_j / T with key
 *     (seed, DRAFT, b, pos_base + j, iter) (T > 0); q(z_j) = softmax(y_j/T)(z_j)
 *     (1 at T = 0); confidence_j = max_v softmax(y_j)_v at temperature 1.
 * Outputs: accept_len [B] (h), commit_len [B] (a), committed [B, K] (C_t, -1
 *   padded), next_draft [B, W] (z_{a+1..W}, -1 padded), next_len [B]
 *   (max(0, W - a)), next_q_at_draft [B, W] (optional, NaN padded),
 *   confidence [B, W] (optional, every proposal row), flags [B] (optional).
 * ------------------------------------------------------------------------- */
sv_status sv_packed_step(sv_handle *h, const void *logits, sv_dtype dtype, int64_t row_stride,
                         int B, int K, int W, int V, const int32_t *prev_draft,
                         const int32_t *prev_len, const float *prev_q_at_draft,
                         const void *prev_draft_logits, const int32_t *prev_q_offset, float T,
                         uint64_t seed, uint64_t iter, const int64_t *pos_base, int32_t eos_id,
                         const int32_t *remaining, int32_t *accept_len, int32_t *commit_len,
                         int32_t *committed, int32_t *next_draft, int32_t *next_len,
                         float *next_q_at_draft, float *confidence, int32_t *flags,
                         void *stream);

/* ---------------------------------------------------------------------------
 * One Packed-SS iteration at T > 0 with top-k truncated distributions
 * ([PackedSS] §3.2, last paragraph: with top-k truncation only the nonzero
 * entries of the stored drafter distribution Q need to be kept; Alg. 2).
 *   Truncation keeps a row's k largest logits (ties to the lowest id) and
 *   renormalises softmax(x/T) over them: kp entries for the target p of
 *   verify rows, kq for the drafter Q of proposal rows (1 <= kp, kq <=
 *   min(64, V)).
 *   logits [B, K+W, V], prev_draft, prev_len, pos_base, eos_id, remaining,
 *   seed, iter and the outputs shared with sv_packed_step mean what they
 *   mean there (K, W <= 32).
 *   prev_q_ids [B, W, kq] (int32), prev_q_probs [B, W, kq] (float32): the
 *     previous call's drafter lists (its q_ids / q_probs); Q_{t-1}^(i) is
 *     list prev_q_offset[b] + i (Alg. 2 line 12).  Each draft token must be
 *     in its list.
 *   Verify position i: accept d_i w.p. min{1, p(d_i)/Q(d_i)}, p(d) = 0 off
 *   the target list.  First rejection h: the correction is the Gumbel-max
 *   over v with [p(v) - Q(v)]_+ > 0 of log [p(v) - Q(v)]_+ + G(key (seed,
 *   SAMPLE, b, pos_base + h, 0)); no rejection: the bonus is the Gumbel-max
 *   of x/T + G over the target list.  Proposal j: z_j is the Gumbel-max of
 *   y_j/T + G(key (seed, DRAFT, b, pos_base + j, iter)) over its list.
 * Outputs: accept_len, commit_len, committed, next_draft, next_len,
 *   next_q_at_draft (optional) as in sv_packed_step; q_ids [B, W, kq] and
 *   q_probs [B, W, kq]: every proposal row's list (ids by logit desc, id
 *   asc) and truncated probabilities, to be passed back as prev_q_ids /
 *   prev_q_probs; flags [B] (optional: acceptance tests within 1e-9 and
 *   Gumbel-max top-two gaps below 1e-9).
 *   Every row the step needs is read once (a streaming top-k selection);
 *   the decisions run in fp64 on the lists.  The caller's buffers are not
 *   kept; the handle's workspace holds B (K+W) 64 (logit, id) pairs.
 * Errors: SV_ERR_INVALID_ARG (shapes, T <= 0, kp or kq out of range);
 *   latched SV_ERR_DEVICE_BOUNDS for prev_len or prev_q_offset out of range,
 *   or a draft token missing from its stored list.
 * ------------------------------------------------------------------------- */
sv_status sv_packed_topk_step(sv_handle *h, const void *logits, sv_dtype dtype,
                              int64_t row_stride, int B, int K, int W, int V, int kp, int kq,
                              const int32_t *prev_draft, const int32_t *prev_len,
                              const int32_t *prev_q_ids, const float *prev_q_probs,
                              const int32_t *prev_q_offset, float T, uint64_t seed, uint64_t iter,
                              const int64_t *pos_base, int32_t eos_id, const int32_t *remaining,
                              int32_t *accept_len, int32_t *commit_len, int32_t *committed,
                              int32_t *next_draft, int32_t *next_len, float *next_q_at_draft,
                              int32_t *q_ids, float *q_probs, int32_t *flags, void *stream);

/* ---------------------------------------------------------------------------
 * One iteration of Packed-SS with any-order greedy verification ([PackedSS]
 * App. C "Procedure", Alg. 3 lines 6-15, eq. 8; confidence scores of App.
 * E.6 "Confidence scores").
 *   u [B] in [0, W]: unresolved positions of the active window;
 *   win_pos [B, W]: those output positions, ascending (first u entries);
 *   order [B, W]: pi_t, the window index checked at each rank (its first u
 *     entries a permutation of 0..u-1);
 *   draft [B, W]: the draft token at each window position, -1 if none;
 *   end_pos [B]: E, the last output position to generate.
 *   kappa = the number of leading ranks whose position has a draft token.
 *   logits [B, Kv + W, V]: verify row r (r < min(kappa + 1, u), which must
 *     be <= Kv) is the verifier's prediction at rank r given the draft tokens
 *     of the earlier ranks; proposal row Kv + i (i < u) is the drafter's row
 *     at win_pos[i].  Other rows are not read.
 *   v_r = argmax of verify row r (lowest id on ties); h = the leading ranks
 *   r < kappa whose draft equals v_r; A = min(h + 1, u); the pairs
 *   (win_pos[order[r]], v_r), r < A, are accepted; an accepted eos_id at
 *   position p lowers E to min(E, p) and pairs beyond E are dropped.
 * Outputs: accept_len [B] (h), commit_len [B] (pairs kept), commit_pos /
 *   commit_tok [B, W] (rank order, -1 padded), end_out [B] (E),
 *   next_draft [B, W] (argmax of proposal row i at window positions that
 *   stay unresolved and <= E, else -1), score [B, W] (optional: the
 *   probability at temperature 1 of each proposal row's argmax, NaN beyond
 *   u; the confidence scores by which a caller's order policy ranks the
 *   next window, App. E.6).
 * Errors: SV_ERR_INVALID_ARG; latched SV_ERR_DEVICE_BOUNDS for u outside
 *   [0, W], an order that is not a permutation, or min(kappa + 1, u) > Kv.
 * ------------------------------------------------------------------------- */
sv_status sv_packed_anyorder_step(sv_handle *h, const void *logits, sv_dtype dtype,
                                  int64_t row_stride, int B, int Kv, int W, int V,
                                  const int32_t *u, const int32_t *win_pos, const int32_t *order,
                                  const int32_t *draft, const int32_t *end_pos, int32_t eos_id,
                                  int32_t *accept_len, int32_t *commit_len, int32_t *commit_pos,
                                  int32_t *commit_tok, int32_t *end_out, int32_t *next_draft,
                                  float *score, void *stream);

/* ---------------------------------------------------------------------------
 * Options (testing and measurement).
 *   SV_OPT_FORCE_RESCUE (value 0/1): decide every sampled sequence on the
 *     fp64 path, as if every fast decision fell inside its error bound.
 *   SV_OPT_TIMING_EVENTS: value is a pointer to two cudaEvent_t (start, stop)
 *     recorded around the streaming pass of the next calls, together with
 *     the kernels that prepare it (SPOT state masks, any-order preparation,
 *     the seed records of Gumbel-max rows), or around the top-k selection
 *     of sv_packed_topk_step; 0 = off.  The events stay owned by the
 *     caller.
 * ------------------------------------------------------------------------- */
typedef enum { SV_OPT_FORCE_RESCUE = 1, SV_OPT_TIMING_EVENTS = 2 } sv_option;
sv_status sv_set_option(sv_handle *h, sv_option opt, int64_t value);

/* ---------------------------------------------------------------------------
 * Self-test of the fp32 arithmetic behind the certified decisions, measured
 * on the device against fp64 over n samples (synchronises `stream`):
 *   ratios[0] = max |G32 - G| / 2^-17   (fp32 Gumbel, including u -> 0, 1)
 *   ratios[1] = max relative error of ex2.approx / 2^-21
 *   ratios[2] = max error of lg2.approx / (2^-22 max(1, |log2 x|))
 *   ratios[3] = number of skip draws whose gap (the fast evaluation the
 *               kernels use) differs from the exact threshold search: 0
 *   ratios[4] = number of ids whose G lies outside the Gumbel bound tables
 *               for the top byte of their fine bits: 0
 * Every ratio must stay below 1 for the error bounds the kernels use.
 * `ratios` is a caller-owned array of 5 doubles.
 * ------------------------------------------------------------------------- */
sv_status sv_selftest(sv_handle *h, uint64_t seed, int64_t n, double *ratios, void *stream);

/* ---------------------------------------------------------------------------
 * Self-test of the bounded waits (enqueued on `stream`, asynchronous).  One
 * small kernel waits, with at most `limit` tries each (0 <= limit <= 2^24,
 * the kernels' own limit), on an mbarrier that nothing arrives at and on a
 * device word that nothing changes -- the two wait forms every kernel of the
 * library uses.  Both waits expire, the kernel latches SV_ERR_TIMEOUT in the
 * handle and returns, so the next sv_sync_status returns SV_ERR_TIMEOUT and
 * the handle stays usable.  Errors: SV_ERR_INVALID_ARG, SV_ERR_CUDA.
 * ------------------------------------------------------------------------- */
sv_status sv_wait_selftest(sv_handle *h, int64_t limit, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SV_H */
