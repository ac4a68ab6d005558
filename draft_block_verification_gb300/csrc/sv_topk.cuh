// sv_topk.cuh -- the Packed-SS step with top-k truncated distributions
// ("One Call Ahead: Packed Self-Speculative Decoding with Diffusion
// Drafting", §3.2, last paragraph; Alg. 2).
//
// Two kernels.  topk_select_kernel streams every row the step needs (verify
// rows 0..prev_len and the W proposal rows) once from HBM and writes its k
// largest logits (ties to the lowest id) as a sorted list; topk_decide_kernel
// runs the step on those lists, one warp per sequence, in fp64.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kTopkMax = 64;  // largest k of either side

struct TopkJob {
    const char *src;       // logits [B, K+W, V] rows, rs bytes apart
    int64_t rs;
    int dtype;             // SV_F32 / SV_BF16
    int V, nvec;           // vocabulary; 16-byte vectors per row
    int B, K, W, kp, kq;
    float T;
    uint64_t seed, iter;
    const int64_t *pos_base;
    int eos;
    const int32_t *remaining;
    const int32_t *prev_draft;    // [B, K-1]
    const int32_t *prev_len;      // [B]
    const int32_t *prev_q_ids;    // [B, W, kq]
    const float *prev_q_probs;    // [B, W, kq]
    const int32_t *prev_off;      // [B]
    const uint64_t *skip;         // skip thresholds of the top-id draws
    float *lval;                  // [B * (K+W), kTopkMax] list logits (workspace)
    int32_t *lid;                 // [B * (K+W), kTopkMax] list ids (workspace)
    double *lg;                   // [B * (K+W), kTopkMax] Gumbel value of each entry
    double *lL;                   // [B * (K+W)] log-sum-exp of the list at T
    int32_t *acc, *commit_len, *committed, *next_draft, *next_len;
    float *next_q;                // [B, W] (optional)
    int32_t *q_ids;               // [B, W, kq]
    float *q_probs;               // [B, W, kq]
    int32_t *flags;               // [B] (optional)
    int *err;
};

cudaError_t topk_select_launch(const TopkJob &t, cudaStream_t s);
cudaError_t topk_decide_launch(const TopkJob &t, cudaStream_t s);

}  // namespace sv
