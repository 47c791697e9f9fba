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

// Each thread quantises QG groups of 8 elements (see quant8_values), one per
// grid-wide stride, with all QG loads issued before the arithmetic so each
// thread keeps QG loads in flight.  Requires K % 32 == 0.
constexpr int QG = 4;
__global__ void __launch_bounds__(256) k_quant_mxfp4(const uint16_t* __restrict__ x, size_t ngroups,
                                                     uint8_t* __restrict__ codes,
                                                     uint8_t* __restrict__ scales) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t g0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint4 q[QG];
#pragma unroll
  for (int i = 0; i < QG; ++i) {
    const size_t g = g0 + i * stride;
    q[i] = g < ngroups ? __ldg(reinterpret_cast<const uint4*>(x + g * 8)) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < QG; ++i) quant8_values(q[i], g0 + i * stride, g0 + i * stride < ngroups, codes, scales);
}

cudaError_t launch_quant_mxfp4(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                               cudaStream_t s) {
  const size_t ngroups = (size_t)rows * K / 8;
  if (ngroups == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((ngroups + 256 * QG - 1) / (256 * QG));
  count_launch(), k_quant_mxfp4<<<blocks, 256, 0, s>>>(x, ngroups, codes, scales);
  return cudaGetLastError();
}

// MXFP8 (E4M3 elements, E8M0 per 32) activation quantisation: the same
// structure, QG groups of 8 per thread.
__global__ void __launch_bounds__(256) k_quant_mxfp8(const uint16_t* __restrict__ x, size_t ngroups,
                                                     uint8_t* __restrict__ codes,
                                                     uint8_t* __restrict__ scales) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t g0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint4 q[QG];
#pragma unroll
  for (int i = 0; i < QG; ++i) {
    const size_t g = g0 + i * stride;
    q[i] = g < ngroups ? __ldg(reinterpret_cast<const uint4*>(x + g * 8)) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < QG; ++i) quant8_values_mx8(q[i], g0 + i * stride, g0 + i * stride < ngroups, codes, scales);
}

cudaError_t launch_quant_mxfp8(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                               cudaStream_t s) {
  const size_t ngroups = (size_t)rows * K / 8;
  if (ngroups == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((ngroups + 256 * QG - 1) / (256 * QG));
  count_launch(), k_quant_mxfp8<<<blocks, 256, 0, s>>>(x, ngroups, codes, scales);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ A1

// Router up to 16 tokens: one block per (expert row, tile of 16 tokens); the 256
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

// Batched router: a 128-token x 128-expert tile per block, 256 threads with
// 8 x 8 outputs each (rows 4ty..4ty+3 and 64+4ty.., columns 4tx.. and
// 64+4tx.., so the shared-memory reads are conflict-free), K staged 16 at a
// time through double-buffered shared memory (the next slice is loaded into
// registers while the current one is used), FP32 FMA in k order.  Split-K
// part p covers k-steps [p*nk/S, (p+1)*nk/S) and writes out[p] ([S][T][E]);
// with S == 1 out is the logits and the bias is added here.
constexpr int RBM = 128, RBN = 128, RBK = 16;
__global__ void __launch_bounds__(256) k_router_sgemm(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                                                      const float* __restrict__ bias, float* __restrict__ out, int T,
                                                      int H, int E, int S) {
  __shared__ __align__(16) float As[2][RBK][RBM + 4];
  __shared__ __align__(16) float Bs[2][RBK][RBN + 4];
  const int m0 = blockIdx.x * RBM, n0 = blockIdx.y * RBN, p = blockIdx.z;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int nk = H / RBK;
  const int ks0 = p * nk / S, ks1 = (p + 1) * nk / S;
  // loader: row tid/2 of each tile, 8 consecutive k
  const int lr = tid >> 1, lc = (tid & 1) * 8;
  const bool xa = m0 + lr < T, wa = n0 + lr < E;
  const uint16_t* xrow = x + (size_t)(xa ? m0 + lr : 0) * H + lc;
  const float* wrow = wr + (size_t)(wa ? n0 + lr : 0) * H + lc;
  auto load = [&](int ks, uint4& xv, float4& w0, float4& w1) {
    xv = xa ? __ldg(reinterpret_cast<const uint4*>(xrow + ks * RBK)) : make_uint4(0, 0, 0, 0);
    w0 = wa ? __ldg(reinterpret_cast<const float4*>(wrow + ks * RBK)) : make_float4(0, 0, 0, 0);
    w1 = wa ? __ldg(reinterpret_cast<const float4*>(wrow + ks * RBK + 4)) : make_float4(0, 0, 0, 0);
  };
  auto store = [&](int buf, const uint4& xv, const float4& w0, const float4& w1) {
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      As[buf][lc + 2 * i][lr] = bf16_lo(xw[i]);
      As[buf][lc + 2 * i + 1][lr] = bf16_hi(xw[i]);
    }
    Bs[buf][lc + 0][lr] = w0.x;
    Bs[buf][lc + 1][lr] = w0.y;
    Bs[buf][lc + 2][lr] = w0.z;
    Bs[buf][lc + 3][lr] = w0.w;
    Bs[buf][lc + 4][lr] = w1.x;
    Bs[buf][lc + 5][lr] = w1.y;
    Bs[buf][lc + 6][lr] = w1.z;
    Bs[buf][lc + 7][lr] = w1.w;
  };
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
  uint4 xv;
  float4 w0, w1;
  if (ks0 < ks1) {
    load(ks0, xv, w0, w1);
    store(0, xv, w0, w1);
  }
  __syncthreads();
  for (int ks = ks0; ks < ks1; ++ks) {
    const int buf = (ks - ks0) & 1;
    if (ks + 1 < ks1) load(ks + 1, xv, w0, w1);
#pragma unroll
    for (int kk = 0; kk < RBK; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    if (ks + 1 < ks1) store(buf ^ 1, xv, w0, w1);
    __syncthreads();
  }
  float* o = out + (size_t)p * T * E;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
    if (m >= T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
      if (n < E) o[(size_t)m * E + n] = acc[i][j] + ((S == 1 && bias) ? bias[n] : 0.0f);
    }
  }
}

// Router for 16 < T <= 512: a 64-token x 64-expert tile and one K part of
// H / S elements per block (256 threads, 4 x 4 outputs each at rows 4ty..
// and columns 4tx..), K staged 32 at a time through shared memory, FP32 FMA
// in k order.  Part p writes out[p] ([S][T][E]); k_router_sum adds the parts
// in ascending order.  Enough blocks to cover the GPU where a per-row pass
// would re-read x once per expert.
constexpr int RSM = 64, RSK = 32;
__global__ void __launch_bounds__(256) k_router_splitk(const uint16_t* __restrict__ x, const float* __restrict__ wr,
                                                       float* __restrict__ out, int T, int H, int E, int S) {
  __shared__ __align__(16) float As[RSK][RSM + 4];
  __shared__ __align__(16) float Bs[RSK][RSM + 4];
  const int m0 = blockIdx.x * RSM, n0 = blockIdx.y * RSM, p = blockIdx.z;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int kc = H / S, kb = p * kc;
  // loader: row tid / 4 of each tile, 8 consecutive k at 8 (tid % 4)
  const int lr = tid >> 2, lc = (tid & 3) * 8;
  const bool xa = m0 + lr < T, wa = n0 + lr < E;
  const uint16_t* xrow = x + (size_t)(xa ? m0 + lr : 0) * H + kb + lc;
  const float* wrow = wr + (size_t)(wa ? n0 + lr : 0) * H + kb + lc;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int k0 = 0; k0 < kc; k0 += RSK) {
    const uint4 xv = xa ? __ldg(reinterpret_cast<const uint4*>(xrow + k0)) : make_uint4(0, 0, 0, 0);
    const float4 w0 = wa ? __ldg(reinterpret_cast<const float4*>(wrow + k0)) : make_float4(0, 0, 0, 0);
    const float4 w1 = wa ? __ldg(reinterpret_cast<const float4*>(wrow + k0 + 4)) : make_float4(0, 0, 0, 0);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      As[lc + 2 * i][lr] = bf16_lo(xw[i]);
      As[lc + 2 * i + 1][lr] = bf16_hi(xw[i]);
    }
    Bs[lc + 0][lr] = w0.x;
    Bs[lc + 1][lr] = w0.y;
    Bs[lc + 2][lr] = w0.z;
    Bs[lc + 3][lr] = w0.w;
    Bs[lc + 4][lr] = w1.x;
    Bs[lc + 5][lr] = w1.y;
    Bs[lc + 6][lr] = w1.z;
    Bs[lc + 7][lr] = w1.w;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < RSK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* o = out + (size_t)p * T * E;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < E) o[(size_t)m * E + n] = acc[i][j];
    }
  }
}

// logits = sum over the S split-K parts in ascending order, + bias; four
// consecutive logits per thread when E % 4 == 0 (all parts' loads issued
// before the sums), else one.
__global__ void __launch_bounds__(256) k_router_sum(const float* __restrict__ part, const float* __restrict__ bias,
                                                    float* __restrict__ logits, int T, int E, int S) {
  const size_t n = (size_t)T * E;
  if (E % 4 == 0) {
    const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= n) return;
    float4 v = *reinterpret_cast<const float4*>(part + i);
    constexpr int B = 8;  // parts loaded together
    for (int p0 = 1; p0 < S; p0 += B) {
      float4 q[B];
#pragma unroll
      for (int j = 0; j < B; ++j)
        q[j] = p0 + j < S ? *reinterpret_cast<const float4*>(part + (size_t)(p0 + j) * n + i) : make_float4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < B; ++j)
        if (p0 + j < S) {
          v.x += q[j].x;
          v.y += q[j].y;
          v.z += q[j].z;
          v.w += q[j].w;
        }
    }
    if (bias) {
      const int e = (int)(i % E);
      v.x += bias[e];
      v.y += bias[e + 1];
      v.z += bias[e + 2];
      v.w += bias[e + 3];
    }
    *reinterpret_cast<float4*>(logits + i) = v;
    return;
  }
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float v = part[i];
  for (int p = 1; p < S; ++p) v += part[(size_t)p * n + i];
  if (bias) v += bias[i % E];
  logits[i] = v;
}

cudaError_t launch_router_logits(const uint16_t* x, const float* wr, const float* bias, float* logits,
                                 int T, int H, int E, float* part, cudaStream_t s, uint16_t* wsplit, int* status,
                                 uint64_t limit_ns) {
  if (T == 0) return cudaSuccess;
  // Up to 16 tokens one block per expert row; up to 512 split-K 64 x 64
  // tiles; beyond that the tensor cores (E = 64 or 128) or the 128 x 128
  // tiled FP32 GEMM, split along K to balance the SMs.
  int S = router_splits(T, E, H);
  cudaError_t err;
  if (wsplit && status && router_tc_supported(T, H, E)) {
    S = router_tc_splits(T, H, E);
    if ((err = launch_router_tc(x, wr, bias, S == 1 ? logits : part, T, H, E, S, wsplit, status, limit_ns, s)) !=
        cudaSuccess || S == 1)
      return err;
    const size_t n = (size_t)T * E;
    count_launch(), k_router_sum<<<(unsigned)((n / 4 + 255) / 256), 256, 0, s>>>(part, bias, logits, T, E, S);
    return cudaGetLastError();
  }
  if (T <= 16) {
    dim3 grid(E, (T + 15) / 16);
    count_launch(), k_router_gemv<<<grid, 256, 0, s>>>(x, wr, bias, logits, T, H, E);
    return cudaGetLastError();
  }
  if (T <= 512) {
    dim3 grid((T + RSM - 1) / RSM, (E + RSM - 1) / RSM, S);
    count_launch(), k_router_splitk<<<grid, 256, 0, s>>>(x, wr, part, T, H, E, S);
  } else {
    dim3 grid((T + RBM - 1) / RBM, (E + RBN - 1) / RBN, S);
    count_launch(), k_router_sgemm<<<grid, 256, 0, s>>>(x, wr, bias, S == 1 ? logits : part, T, H, E, S);
  }
  err = cudaGetLastError();
  if (err != cudaSuccess || (S == 1 && T > 512)) return err;
  const size_t n = (size_t)T * E;
  const size_t threads = E % 4 == 0 ? n / 4 : n;
  count_launch(), k_router_sum<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(part, bias, logits, T, E, S);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ A2

// ids / wts: [T][k].  With ids_ext set, also [T][k + 1] copies whose last
// column is the shared expert folded into the table (expert E, weight 1).
__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int T, int E, int k, int score,
                                              const float* __restrict__ sel_bias, int* __restrict__ ids,
                                              float* __restrict__ wts, int* __restrict__ ids_ext,
                                              float* __restrict__ wts_ext) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  int sel[MAX_TOPK];
  float w[MAX_TOPK];
  float v[8];
  load_logit_row(logits + (size_t)t * E, E, v, false);
  route_row(v, E, k, score, sel_bias, sel, w);
  const int lane = threadIdx.x & 31;
  if (lane < k) {
    int id = 0;
    float wv = 0.0f;
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j == lane) { id = sel[j]; wv = w[j]; }
    ids[(size_t)t * k + lane] = id;
    wts[(size_t)t * k + lane] = wv;
    if (ids_ext) {
      ids_ext[(size_t)t * (k + 1) + lane] = id;
      wts_ext[(size_t)t * (k + 1) + lane] = wv;
    }
  }
  if (ids_ext && lane == k) {
    ids_ext[(size_t)t * (k + 1) + k] = E;
    wts_ext[(size_t)t * (k + 1) + k] = 1.0f;
  }
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int score, const float* sel_bias, int* ids,
                        float* w, cudaStream_t s, int* ids_ext, float* w_ext) {
  if (T == 0) return cudaSuccess;
  count_launch(), k_topk<<<(T + 7) / 8, 256, 0, s>>>(logits, T, E, k, score, sel_bias, ids, w, ids_ext, w_ext);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ A3

// Pass 1: per chunk of PERM_CHUNK assignments, the stable rank of each
// assignment among the chunk's assignments to the same expert, and the
// chunk's per-expert counts.  Within a warp peers are found with match_any;
// across warps a per-expert exclusive scan over the 32 warp counts.
__global__ void __launch_bounds__(PERM_CHUNK) k_perm_rank(const int* __restrict__ ids, int n, int E,
                                                          int* __restrict__ rank,
                                                          int* __restrict__ chunk_cnt, int* __restrict__ status) {
  __shared__ int wc[32][MAX_E];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32 * MAX_E; i += blockDim.x) (&wc[0][0])[i] = 0;
  __syncthreads();
  const int a = blockIdx.x * PERM_CHUNK + threadIdx.x;
  const int e0 = a < n ? ids[a] : -1;
  const int e = (e0 >= 0 && e0 < E) ? e0 : -1;  // out-of-range ids are left out
  if (a < n && e < 0) report_bad_index(status);
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
                           int* inv_perm, int* rank, int* chunk_cnt, int* chunk_base, cudaStream_t s, int* status) {
  const int n = T * k;
  const int nchunks = (n + PERM_CHUNK - 1) / PERM_CHUNK;
  if (nchunks > 0) {
    count_launch(), k_perm_rank<<<nchunks, PERM_CHUNK, 0, s>>>(ids, n, E, rank, chunk_cnt, status);
  }
  count_launch(), k_perm_scan<<<1, MAX_E, 0, s>>>(chunk_cnt, nchunks, E, chunk_base, counts, offsets);
  if (n > 0) count_launch(), k_perm_scatter<<<(n + 255) / 256, 256, 0, s>>>(ids, n, E, rank, chunk_base, offsets, perm, inv_perm);
  return cudaGetLastError();
}

}  // namespace moefp4
