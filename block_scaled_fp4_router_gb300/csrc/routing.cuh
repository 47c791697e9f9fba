// Softmax top-k routing of one token per warp (A2), shared by the router
// kernels and the fused decode.  AMD technical article "MiniMax-M3.1 on AMD
// Instinct GPUs", section "MiniMax-M3.1 at a glance": 4 of 128 routed experts
// are active per token.
#pragma once

#include "common.cuh"

namespace moefp4 {

// Lane l loads logits l, l+32, ... (E <= 256) of one row; coherent = read
// through L2 (for rows written earlier in the same launch).
__device__ __forceinline__ void load_logit_row(const float* row, int E, float (&v)[8], bool coherent) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? (coherent ? __ldcg(row + e) : row[e]) : 0.0f;
  }
}

// Order-preserving integer image of a float (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Score functions of the router (moe_layer_desc_t.score_func).
enum ScoreFunc { SCORE_SOFTMAX = 0, SCORE_SIGMOID = 1 };

// Top-k of one row of E <= 256 keys held by one warp (lane l holds experts
// l, l+32, ...; see load_logit_row); ties go to the lower expert index.  Every
// lane returns the ids in descending key order and, for each, the payload
// value pay of that expert.
__device__ __forceinline__ void warp_topk(const float (&v)[8], const float (&pay)[8], int E, int k,
                                          int (&ids)[MAX_TOPK], float (&vals)[MAX_TOPK]) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (lane + 32 * i >= E) taken |= 1u << i;
  for (int j = 0; j < k; ++j) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (!(taken >> i & 1)) {
        const uint32_t e = lane + 32 * i;
        const uint64_t key = ((uint64_t)float_key(v[i]) << 32) | (0xffffffffu - e);
        best = key > best ? key : best;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(FULL, best, o);
      best = other > best ? other : best;
    }
    const int e = (int)(0xffffffffu - (uint32_t)best);
    if ((e & 31) == lane) taken |= 1u << (e >> 5);
    ids[j] = e;
    // the selected payload, from its owner lane
    float mine = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i == (e >> 5)) mine = pay[i];
    vals[j] = __shfl_sync(FULL, mine, e & 31);
  }
}

// Renormalised weights of the selected logits: softmax over them, which is
// p_j / sum p_sel for the softmax p over all experts.  (Sigmoid scoring:
// route_row below.)
__device__ __forceinline__ void topk_weights(const float (&vals)[MAX_TOPK], int k, float (&w)[MAX_TOPK]) {
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < MAX_TOPK; ++j) {
    w[j] = j < k ? expf(vals[j] - vals[0]) : 0.0f;
    sum += w[j];
  }
  const float inv = 1.0f / sum;
#pragma unroll
  for (int j = 0; j < MAX_TOPK; ++j) w[j] *= inv;
}

// The routing of one token row held by one warp (lane l holds the logits of
// experts l, l+32, ...):
//  SCORE_SOFTMAX  v are the logits with the router bias already added: the
//                 top-k logits, weights softmax over the selected ones;
//  SCORE_SIGMOID  v are the raw logits: scores s = sigmoid(v), the top-k of
//                 s + bias (bias may be null: 0), weights s_sel / sum s_sel
//                 (the bias only corrects the choice).
// Every lane returns the ids (descending key, ties to the lower index) and
// the renormalised weights.
__device__ __forceinline__ void route_row(const float (&v)[8], int E, int k, int score, const float* bias,
                                          int (&ids)[MAX_TOPK], float (&w)[MAX_TOPK]) {
  float vals[MAX_TOPK];
  if (score == SCORE_SIGMOID) {
    const int lane = threadIdx.x & 31;
    float sc[8], key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      sc[i] = e < E ? 1.0f / (1.0f + expf(-v[i])) : 0.0f;
      key[i] = sc[i] + ((bias && e < E) ? __ldg(bias + e) : 0.0f);
    }
    warp_topk(key, sc, E, k, ids, vals);
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j < k) sum += vals[j];
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j) w[j] = j < k ? vals[j] / sum : 0.0f;
  } else {
    warp_topk(v, v, E, k, ids, vals);
    topk_weights(vals, k, w);
  }
}

}  // namespace moefp4
