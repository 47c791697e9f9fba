// A1 router logits, A2 softmax top-k with renormalisation, A3 token-to-expert
// permutation, A4 dynamic MXFP4 activation quantisation.
//
// AMD technical article "MiniMax-M3.1 on AMD Instinct GPUs: Day-0 support and
// optimization": section "MiniMax-M3.1 at a glance" (128 routed experts, 4
// active per token; the router is high precision) and section "What we
// Optimized" (a stacked router GEMM ahead of the fused MXFP4 MoE).  Model card
// "amd/MiniMax-M3.1-Flash-Quark-MXFP4", section "Model Overview": routed-expert
// activations are quantised to OCP MXFP4 at run time.
#include "common.cuh"
#include "kernels.h"
#include "routing.cuh"

namespace moefp4 {

// ------------------------------------------------------------------ A4

// One thread per 8 elements (see quant8_group).  Requires K % 32 == 0.
__global__ void __launch_bounds__(256) k_quant_mxfp4(const uint16_t* __restrict__ x, size_t ngroups,
                                                     uint8_t* __restrict__ codes,
                                                     uint8_t* __restrict__ scales) {
  const size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  quant8_group(x, g, g < ngroups, codes, scales);
}

cudaError_t launch_quant_mxfp4(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                               cudaStream_t s) {
  const size_t ngroups = (size_t)rows * K / 8;
  if (ngroups == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((ngroups + 255) / 256);
  k_quant_mxfp4<<<blocks, 256, 0, s>>>(x, ngroups, codes, scales);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ A1

// Router up to a few hundred tokens: one block per (expert row, tile of 16 tokens); the 256
// threads stride over H eight elements at a time (two float4 of Wr, one uint4
// of x per token), then reduce over lanes and warps in a fixed order.
__global__ void __launch_bounds__(256) k_router_gemv(const uint16_t* __restrict__ x,
                                                     const float* __restrict__ wr,
                                                     const float* __restrict__ bias,
                                                     float* __restrict__ logits, int T, int H, int E) {
  const int e = blockIdx.x;
  const int t0 = blockIdx.y * 16;
  const int nt = min(16, T - t0);
  float acc[16];
#pragma unroll
  for (int t = 0; t < 16; ++t) acc[t] = 0.0f;
  const float* wrow = wr + (size_t)e * H;
  for (int k = threadIdx.x * 8; k < H; k += blockDim.x * 8) {
    const float4 wa = __ldg(reinterpret_cast<const float4*>(wrow + k));
    const float4 wb = __ldg(reinterpret_cast<const float4*>(wrow + k + 4));
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      if (t < nt) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * H + k));
        float a = acc[t];
        a = fmaf(bf16_lo(q.x), wa.x, a);
        a = fmaf(bf16_hi(q.x), wa.y, a);
        a = fmaf(bf16_lo(q.y), wa.z, a);
        a = fmaf(bf16_hi(q.y), wa.w, a);
        a = fmaf(bf16_lo(q.z), wb.x, a);
        a = fmaf(bf16_hi(q.z), wb.y, a);
        a = fmaf(bf16_lo(q.w), wb.z, a);
        a = fmaf(bf16_hi(q.w), wb.w, a);
        acc[t] = a;
      }
    }
  }
  __shared__ float part[8][16];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    const float v = warp_sum(acc[t]);
    if (lane == 0) part[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += part[w][threadIdx.x];
    if (bias) s += bias[e];
    logits[(size_t)(t0 + threadIdx.x) * E + e] = s;
  }
}

// Batched router: a 64-token x 64-expert tile per block, K staged 32 at a
// time through shared memory, 4x4 outputs per thread, FP32 FMA in k order.
constexpr int RBM = 64, RBN = 64, RBK = 32;
__global__ void __launch_bounds__(256) k_router_gemm(const uint16_t* __restrict__ x,
                                                     const float* __restrict__ wr,
                                                     const float* __restrict__ bias,
                                                     float* __restrict__ logits, int T, int H, int E) {
  __shared__ float xs_[RBK][RBM + 4];
  __shared__ float ws_[RBK][RBN + 4];
  const int m0 = blockIdx.x * RBM, n0 = blockIdx.y * RBN;
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;  // 16 x 16 threads, 4x4 outputs each
  float acc[4][4] = {};
  // loaders: x tile 64 rows x 32 bf16 -> thread loads 8 bf16 (row tid/4, cols (tid%4)*8)
  const int lr = tid >> 2, lc = (tid & 3) * 8;
  for (int k0 = 0; k0 < H; k0 += RBK) {
    {
      const int m = m0 + lr;
      uint4 q = make_uint4(0, 0, 0, 0);
      if (m < T) q = __ldg(reinterpret_cast<const uint4*>(x + (size_t)m * H + k0 + lc));
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xs_[lc + 2 * i][lr] = bf16_lo(w[i]);
        xs_[lc + 2 * i + 1][lr] = bf16_hi(w[i]);
      }
      const int n = n0 + lr;
      float4 a = make_float4(0, 0, 0, 0), b = a;
      if (n < E) {
        a = __ldg(reinterpret_cast<const float4*>(wr + (size_t)n * H + k0 + lc));
        b = __ldg(reinterpret_cast<const float4*>(wr + (size_t)n * H + k0 + lc + 4));
      }
      ws_[lc + 0][lr] = a.x; ws_[lc + 1][lr] = a.y; ws_[lc + 2][lr] = a.z; ws_[lc + 3][lr] = a.w;
      ws_[lc + 4][lr] = b.x; ws_[lc + 5][lr] = b.y; ws_[lc + 6][lr] = b.z; ws_[lc + 7][lr] = b.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < RBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&xs_[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&ws_[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < E) logits[(size_t)m * E + n] = acc[i][j] + (bias ? bias[n] : 0.0f);
    }
  }
}

cudaError_t launch_router_logits(const uint16_t* x, const float* wr, const float* bias, float* logits,
                                 int T, int H, int E, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  // Up to a few hundred tokens one block per (expert row, 16 tokens) keeps
  // every SM busy (the x re-reads hit L2); beyond that the tiled GEMM.
  if (T <= 512) {
    dim3 grid(E, (T + 15) / 16);
    k_router_gemv<<<grid, 256, 0, s>>>(x, wr, bias, logits, T, H, E);
  } else {
    dim3 grid((T + RBM - 1) / RBM, (E + RBN - 1) / RBN);
    k_router_gemm<<<grid, 256, 0, s>>>(x, wr, bias, logits, T, H, E);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ A2

__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int T, int E, int k,
                                              int* __restrict__ ids, float* __restrict__ wts) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  int sel[MAX_TOPK];
  float vals[MAX_TOPK], w[MAX_TOPK];
  float v[8];
  load_logit_row(logits + (size_t)t * E, E, v, false);
  warp_topk(v, E, k, sel, vals);
  topk_weights(vals, k, w);
  const int lane = threadIdx.x & 31;
  if (lane < k) {
    int id = 0;
    float wv = 0.0f;
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j == lane) { id = sel[j]; wv = w[j]; }
    ids[(size_t)t * k + lane] = id;
    wts[(size_t)t * k + lane] = wv;
  }
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int* ids, float* w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  k_topk<<<(T + 7) / 8, 256, 0, s>>>(logits, T, E, k, ids, w);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ A3

// Pass 1: per chunk of PERM_CHUNK assignments, the stable rank of each
// assignment among the chunk's assignments to the same expert, and the
// chunk's per-expert counts.  Within a warp peers are found with match_any;
// across warps a per-expert exclusive scan over the 32 warp counts.
__global__ void __launch_bounds__(PERM_CHUNK) k_perm_rank(const int* __restrict__ ids, int n, int E,
                                                          int* __restrict__ rank,
                                                          int* __restrict__ chunk_cnt) {
  __shared__ int wc[32][MAX_E];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32 * MAX_E; i += blockDim.x) (&wc[0][0])[i] = 0;
  __syncthreads();
  const int a = blockIdx.x * PERM_CHUNK + threadIdx.x;
  const int e0 = a < n ? ids[a] : -1;
  const int e = (e0 >= 0 && e0 < E) ? e0 : -1;  // out-of-range ids are left out
  const uint32_t peers = __match_any_sync(FULL, e);
  const int r = __popc(peers & ((1u << lane) - 1));
  if (e >= 0 && r == 0) wc[warp][e] = __popc(peers);
  __syncthreads();
  for (int ex = threadIdx.x; ex < E; ex += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = wc[w][ex];
      wc[w][ex] = run;
      run += c;
    }
    chunk_cnt[(size_t)blockIdx.x * E + ex] = run;
  }
  __syncthreads();
  if (e >= 0) rank[a] = wc[warp][e] + r;
}

// Pass 2 (one block): per-expert totals, chunk bases, exclusive offsets.
__global__ void __launch_bounds__(MAX_E) k_perm_scan(const int* __restrict__ chunk_cnt, int nchunks, int E,
                                                     int* __restrict__ chunk_base, int* __restrict__ counts,
                                                     int* __restrict__ offsets) {
  __shared__ int tot[MAX_E];
  const int ex = threadIdx.x;
  int run = 0;
  if (ex < E) {
    for (int c = 0; c < nchunks; ++c) {
      chunk_base[(size_t)c * E + ex] = run;
      run += chunk_cnt[(size_t)c * E + ex];
    }
    counts[ex] = run;
  }
  tot[ex] = ex < E ? run : 0;
  __syncthreads();
  if (ex == 0) {
    int o = 0;
    for (int i = 0; i < E; ++i) {
      offsets[i] = o;
      o += tot[i];
    }
    offsets[E] = o;
  }
}

// Pass 3: scatter.
__global__ void __launch_bounds__(256) k_perm_scatter(const int* __restrict__ ids, int n, int E,
                                                      const int* __restrict__ rank,
                                                      const int* __restrict__ chunk_base,
                                                      const int* __restrict__ offsets,
                                                      int* __restrict__ perm, int* __restrict__ inv_perm) {
  const int a = blockIdx.x * blockDim.x + threadIdx.x;
  if (a >= n) return;
  const int e = ids[a];
  if (e < 0 || e >= E) {
    inv_perm[a] = -1;
    return;
  }
  const int c = a / PERM_CHUNK;
  const int p = offsets[e] + chunk_base[(size_t)c * E + e] + rank[a];
  perm[p] = a;
  inv_perm[a] = p;
}

cudaError_t launch_permute(const int* ids, int T, int k, int E, int* counts, int* offsets, int* perm,
                           int* inv_perm, int* rank, int* chunk_cnt, int* chunk_base, cudaStream_t s) {
  const int n = T * k;
  const int nchunks = (n + PERM_CHUNK - 1) / PERM_CHUNK;
  if (nchunks > 0) {
    k_perm_rank<<<nchunks, PERM_CHUNK, 0, s>>>(ids, n, E, rank, chunk_cnt);
  }
  k_perm_scan<<<1, MAX_E, 0, s>>>(chunk_cnt, nchunks, E, chunk_base, counts, offsets);
  if (n > 0) k_perm_scatter<<<(n + 255) / 256, 256, 0, s>>>(ids, n, E, rank, chunk_base, offsets, perm, inv_perm);
  return cudaGetLastError();
}

}  // namespace moefp4
