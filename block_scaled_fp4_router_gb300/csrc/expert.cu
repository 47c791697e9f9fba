// A5 - A9 as separate launches for any number of tokens: routed gate/up with
// the SwiGLU + MXFP4 requantise epilogue, routed down projection, the BF16
// shared expert, and the weighted combine.
//
// AMD technical article "MiniMax-M3.1 on AMD Instinct GPUs", section "What we
// Optimized": the MXFP4 fused MoE with the shared expert; section "MiniMax-M3.1
// at a glance": every token passes through the shared expert.  vLLM PR #64273,
// commit list: the "MoE finalize" step is the combine.
//
// Work layout: one block per (expert, output block); tokens of the expert are
// processed in tiles of NT whose activations are staged in shared memory, so
// a weight row is streamed from HBM once per tile (once per call for decode).
#include "expert_units.cuh"
#include "kernels.h"

namespace moefp4 {

constexpr int NT = 16;       // token tile of the routed kernels
constexpr int NT_SH = 8;     // token tile of the shared-expert kernels
constexpr int THREADS = 512; // 16 warps

// ------------------------------------------------------------------ A5 + A6

// Block (e, b): gate rows 32b..32b+31 and up rows I+32b.. of expert e for all
// assignments routed to e, then h = SiLU(G) U quantised to MXFP4 per 32.
template <bool NV>
__global__ void __launch_bounds__(THREADS) k_routed_gate_up(Shape sh, ExpertsDev ex,
                                                            const uint8_t* __restrict__ xq,
                                                            const uint8_t* __restrict__ xs,
                                                            const int* __restrict__ offsets,
                                                            const int* __restrict__ perm,
                                                            uint8_t* __restrict__ hq,
                                                            uint8_t* __restrict__ hs, int* __restrict__ status) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int e = blockIdx.x, b = blockIdx.y;
  const int H = sh.H, I = sh.I, na = sh.T * sh.k;
  const int p0 = max(0, min(offsets[e], na)), n = max(0, min(offsets[e + 1], na) - p0);
  if (n == 0) return;
  uint8_t* xq_s = smem;                                              // [NT][H/2]
  float* xsc_s = reinterpret_cast<float*>(smem + NT * (H / 2));      // [NT][H/32]
  float* gu_s = xsc_s + NT * (H / 32);                               // [64][NT]
  int* rows_s = reinterpret_cast<int*>(gu_s + 64 * NT);              // [NT]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t rb13 = (size_t)H / 2, sb13 = NV ? H / 16 : H / 32;
  const uint8_t* w13 = ex.w13 + (size_t)e * 2 * I * rb13;
  const uint8_t* s13 = ex.w13s + (size_t)e * 2 * I * sb13;
  const float tg = NV ? ex.tscale[e * 3 + 0] : 1.0f, tu = NV ? ex.tscale[e * 3 + 1] : 1.0f;
  for (int t0 = 0; t0 < n; t0 += NT) {
    const int nt = min(NT, n - t0);
    if (threadIdx.x < nt) {
      const int a = perm[p0 + t0 + threadIdx.x];
      const bool ok = a >= 0 && a < na;
      if (!ok) report_bad_index(status);
      rows_s[threadIdx.x] = ok ? a / sh.k : 0;
    }
    __syncthreads();
    stage_mx_rows(xq, xs, H, rows_s, nt, xq_s, xsc_s, false);
    __syncthreads();
    for (int r = warp; r < 64; r += THREADS / 32) {
      const int row = r < 32 ? 32 * b + r : I + 32 * b + (r - 32);
      float acc[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
      fp4_row_dot<NT, NV>(w13 + row * rb13, s13 + row * sb13, H, xq_s, H / 2, xsc_s, H / 32, nullptr, nt,
                          acc);
      const float ts = r < 32 ? tg : tu;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0 && t < nt) gu_s[r * NT + t] = v * ts;
      }
    }
    __syncthreads();
    for (int t = warp; t < nt; t += THREADS / 32) {
      const size_t p = (size_t)p0 + t0 + t;
      swiglu_quant_block(gu_s[lane * NT + t], gu_s[(32 + lane) * NT + t], hq + p * (I / 2) + b * 16,
                         hs + p * (I / 32) + b);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ A7

// Block (e, g): rows 32g..32g+31 of W2[e] against the requantised h of every
// assignment routed to e; y_assign[p][row] = deq(hq[p]) . deq(W2[e][row]).
template <bool NV>
__global__ void __launch_bounds__(THREADS) k_routed_down(Shape sh, ExpertsDev ex,
                                                         const uint8_t* __restrict__ hq,
                                                         const uint8_t* __restrict__ hs,
                                                         const int* __restrict__ offsets,
                                                         float* __restrict__ y_assign) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int e = blockIdx.x, g = blockIdx.y;
  const int H = sh.H, I = sh.I, na = sh.T * sh.k;
  const int p0 = max(0, min(offsets[e], na)), n = max(0, min(offsets[e + 1], na) - p0);
  if (n == 0) return;
  uint8_t* hq_s = smem;                                          // [NT][I/2]
  float* hsc_s = reinterpret_cast<float*>(smem + NT * (I / 2));  // [NT][I/32]
  int* rows_s = reinterpret_cast<int*>(hsc_s + NT * (I / 32));   // [NT]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t rb2 = (size_t)I / 2, sb2 = NV ? I / 16 : I / 32;
  const uint8_t* w2 = ex.w2 + (size_t)e * H * rb2;
  const uint8_t* s2 = ex.w2s + (size_t)e * H * sb2;
  const float td = NV ? ex.tscale[e * 3 + 2] : 1.0f;
  for (int t0 = 0; t0 < n; t0 += NT) {
    const int nt = min(NT, n - t0);
    if (threadIdx.x < nt) rows_s[threadIdx.x] = p0 + t0 + threadIdx.x;
    __syncthreads();
    stage_mx_rows(hq, hs, I, rows_s, nt, hq_s, hsc_s, false);
    __syncthreads();
    for (int r = warp; r < 32; r += THREADS / 32) {
      const int row = 32 * g + r;
      float acc[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
      fp4_row_dot<NT, NV>(w2 + row * rb2, s2 + row * sb2, I, hq_s, I / 2, hsc_s, I / 32, nullptr, nt, acc);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0 && t < nt) y_assign[(size_t)(p0 + t0 + t) * H + row] = v * td;
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ A8

// Block u: shared-expert gate rows 8u..8u+7 and up rows I+8u..I+8u+7 (one row
// per warp) for all tokens, h = BF16(SiLU(G) U).
__global__ void __launch_bounds__(THREADS) k_shared_gate_up(Shape sh, SharedDev shd,
                                                            const uint16_t* __restrict__ x,
                                                            uint16_t* __restrict__ h_shared) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int u = blockIdx.x;
  const int H = sh.H, I = sh.I, T = sh.T;
  uint16_t* x_s = reinterpret_cast<uint16_t*>(smem);                     // [NT_SH][H]
  float* gu_s = reinterpret_cast<float*>(smem + (size_t)NT_SH * H * 2);  // [16][NT_SH]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t0 = 0; t0 < T; t0 += NT_SH) {
    const int nt = min(NT_SH, T - t0);
    const int cpr = H / 8;
    for (int i = threadIdx.x; i < nt * cpr; i += THREADS)
      reinterpret_cast<uint4*>(x_s)[i] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t0 * H) + i);
    __syncthreads();
    {
      const int r = warp;  // 16 warps, 16 rows
      const int row = r < 8 ? 8 * u + r : I + 8 * u + (r - 8);
      float acc[NT_SH];
#pragma unroll
      for (int t = 0; t < NT_SH; ++t) acc[t] = 0.0f;
      bf16_row_dot<NT_SH>(shd.w13 + (size_t)row * H, H, x_s, H, nt, acc);
#pragma unroll
      for (int t = 0; t < NT_SH; ++t) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) gu_s[r * NT_SH + t] = v;
      }
    }
    __syncthreads();
    if (threadIdx.x < nt * 8) {
      const int t = threadIdx.x >> 3, j = threadIdx.x & 7;
      const float h = silu(gu_s[j * NT_SH + t]) * gu_s[(8 + j) * NT_SH + t];
      h_shared[(size_t)(t0 + t) * I + 8 * u + j] = f32_to_bf16_rn(h);
    }
    __syncthreads();
  }
}

// Block g: shared-expert down rows 16g..16g+15 (one per warp) for all tokens.
__global__ void __launch_bounds__(THREADS) k_shared_down(Shape sh, SharedDev shd,
                                                         const uint16_t* __restrict__ h_shared,
                                                         float* __restrict__ y_shared) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int g = blockIdx.x;
  const int H = sh.H, I = sh.I, T = sh.T;
  uint16_t* h_s = reinterpret_cast<uint16_t*>(smem);  // [NT][I]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = 16 * g + warp;
  for (int t0 = 0; t0 < T; t0 += NT) {
    const int nt = min(NT, T - t0);
    const int cpr = I / 8;
    for (int i = threadIdx.x; i < nt * cpr; i += THREADS)
      reinterpret_cast<uint4*>(h_s)[i] = reinterpret_cast<const uint4*>(h_shared + (size_t)t0 * I)[i];
    __syncthreads();
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
    bf16_row_dot<NT>(shd.w2 + (size_t)row * I, I, h_s, I, nt, acc);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float v = warp_sum(acc[t]);
      if (lane == 0 && t < nt) y_shared[(size_t)(t0 + t) * H + row] = v;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ A9

// out[t][h] = BF16(ys[t][h] + sum_j w[t][j] * y_assign[inv_perm[t*k+j]][h]),
// summed in that order in FP32.  One thread per 4 consecutive h.
__global__ void __launch_bounds__(256) k_combine(Shape sh, const float* __restrict__ y_assign,
                                                 const int* __restrict__ inv_perm,
                                                 const float* __restrict__ w,
                                                 const float* __restrict__ y_shared,
                                                 uint16_t* __restrict__ out, int* __restrict__ status) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t q = (size_t)sh.H / 4;
  if (i >= (size_t)sh.T * q) return;
  const int t = (int)(i / q);
  const int h = (int)(i - (size_t)t * q) * 4;
  float4 acc = y_shared ? *reinterpret_cast<const float4*>(y_shared + (size_t)t * sh.H + h)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < sh.k; ++j) {
    const float wj = w[(size_t)t * sh.k + j];
    int p = inv_perm[(size_t)t * sh.k + j];
    if (p < 0 || p >= sh.T * sh.k) {
      report_bad_index(status);
      p = 0;
    }
    const float4 y = *reinterpret_cast<const float4*>(y_assign + (size_t)p * sh.H + h);
    acc.x = fmaf(wj, y.x, acc.x);
    acc.y = fmaf(wj, y.y, acc.y);
    acc.z = fmaf(wj, y.z, acc.z);
    acc.w = fmaf(wj, y.w, acc.w);
  }
  uint2 o;
  o.x = (uint32_t)f32_to_bf16_rn(acc.x) | ((uint32_t)f32_to_bf16_rn(acc.y) << 16);
  o.y = (uint32_t)f32_to_bf16_rn(acc.z) | ((uint32_t)f32_to_bf16_rn(acc.w) << 16);
  *reinterpret_cast<uint2*>(out + (size_t)t * sh.H + h) = o;
}

cudaError_t launch_combine(const Shape& sh, const float* y_assign, const int* inv_perm, const float* w,
                           const float* y_shared, uint16_t* out, cudaStream_t s, int* status) {
  const size_t n = (size_t)sh.T * sh.H / 4;
  if (n == 0) return cudaSuccess;
  count_launch(), k_combine<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(sh, y_assign, inv_perm, w, y_shared, out,
                                                                        status);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ launcher

static cudaError_t set_smem(const void* fn, size_t bytes) {
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t launch_routed_simt(const Shape& sh, const ExpertsDev& ex, const uint8_t* xq, const uint8_t* xs,
                               const int* offsets, const int* perm, uint8_t* hq, uint8_t* hs, float* y_assign,
                               cudaStream_t s, int* status) {
  if (sh.T == 0) return cudaSuccess;
  cudaError_t err;
  const int H = sh.H, I = sh.I;
  {
    const size_t smem = (size_t)NT * (H / 2) + sizeof(float) * NT * (H / 32) + sizeof(float) * 64 * NT +
                        sizeof(int) * NT;
    const void* fn = ex.nv ? (const void*)k_routed_gate_up<true> : (const void*)k_routed_gate_up<false>;
    if ((err = set_smem(fn, smem)) != cudaSuccess) return err;
    dim3 grid(sh.E, I / 32);
    if (ex.nv)
      count_launch(), k_routed_gate_up<true><<<grid, THREADS, smem, s>>>(sh, ex, xq, xs, offsets, perm, hq, hs, status);
    else
      count_launch(), k_routed_gate_up<false><<<grid, THREADS, smem, s>>>(sh, ex, xq, xs, offsets, perm, hq, hs,
                                                                          status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  {
    const size_t smem = (size_t)NT * (I / 2) + sizeof(float) * NT * (I / 32) + sizeof(int) * NT;
    const void* fn = ex.nv ? (const void*)k_routed_down<true> : (const void*)k_routed_down<false>;
    if ((err = set_smem(fn, smem)) != cudaSuccess) return err;
    dim3 grid(sh.E, H / 32);
    if (ex.nv)
      count_launch(), k_routed_down<true><<<grid, THREADS, smem, s>>>(sh, ex, hq, hs, offsets, y_assign);
    else
      count_launch(), k_routed_down<false><<<grid, THREADS, smem, s>>>(sh, ex, hq, hs, offsets, y_assign);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

cudaError_t launch_shared_simt(const Shape& sh, const SharedDev& shd, const uint16_t* x, uint16_t* h_shared,
                               float* y_shared, cudaStream_t s) {
  if (sh.T == 0 || !shd.w13) return cudaSuccess;
  cudaError_t err;
  const int H = sh.H, I = sh.I;
  {
    const size_t smem = (size_t)NT_SH * H * 2 + sizeof(float) * 16 * NT_SH;
    if ((err = set_smem((const void*)k_shared_gate_up, smem)) != cudaSuccess) return err;
    count_launch(), k_shared_gate_up<<<I / 8, THREADS, smem, s>>>(sh, shd, x, h_shared);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  {
    const size_t smem = (size_t)NT * I * 2;
    if ((err = set_smem((const void*)k_shared_down, smem)) != cudaSuccess) return err;
    count_launch(), k_shared_down<<<H / 16, THREADS, smem, s>>>(sh, shd, h_shared, y_shared);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace moefp4
