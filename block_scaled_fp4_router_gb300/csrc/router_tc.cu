// A1 for large batches on tensor cores, as accurate as an FP32 dot product:
// logits = x . Wr^T (+ bias) with FP32 router weights (the router is "high
// precision": AMD technical article "MiniMax-M3.1 on AMD Instinct GPUs",
// section "MiniMax-M3.1 at a glance"; "a stacked router GEMM": section "What
// we Optimized").
//
// x is BF16, so it is exact in BF16.  Wr is split into three BF16 terms,
// W1 = BF16(Wr), W2 = BF16(Wr - W1), W3 = BF16(Wr - W1 - W2) (each
// subtraction exact in FP32), which leaves |Wr - W1 - W2 - W3| below 2^-24
// |Wr|.  Every product x * W_i then has at most 16 significant bits and is
// exact in FP32.  The tensor cores (kind::f16, FP32 accumulation) sum the
// products of one 64-element K chunk, three terms x four MMAs of K = 16, into
// a fresh TMEM accumulator; the epilogue adds the chunks in K order in FP32
// registers.  The tensor cores' own accumulation thus never spans more than
// 64 x 3 products, which keeps its rounding near that of a plain FP32 sum
// (over all K at once it measured 5.4e-7 of sum |x w|).
//
// One block per (128-token tile, K part), persistent over nothing: warp 0
// issues TMA (the x tile and the three W terms per chunk) into a 3-stage
// ring, warp 1 issues the MMAs into two accumulator buffers of E columns,
// warps 2-9 add the chunks (two warps per TMEM lane quadrant, half of the E
// columns each) and store the tile's logits (one K part) or its partial sums.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moefp4 {
namespace {

constexpr int RT_M = 128;          // tokens per tile
constexpr int RT_K = 64;           // K elements per chunk (one 128-byte BF16 row segment)
constexpr int RT_STAGES = 3;
constexpr int RT_EPI_WARPS = 8;
constexpr int RT_THREADS = 64 + 32 * RT_EPI_WARPS;
constexpr uint32_t RT_A_BYTES = RT_M * 128;

__host__ __device__ constexpr uint32_t rt_stage_bytes(int E) { return RT_A_BYTES + 3u * (uint32_t)E * 128u; }

// W [E][H] FP32 -> three BF16 terms [3][E][H], one element per thread.
__global__ void __launch_bounds__(256) k_router_wsplit(const float* __restrict__ wr, size_t n,
                                                       uint16_t* __restrict__ w3) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float w = __ldg(wr + i);
  const uint16_t a = f32_to_bf16_rn(w);
  const float r1 = w - __uint_as_float((uint32_t)a << 16);
  const uint16_t b = f32_to_bf16_rn(r1);
  const float r2 = r1 - __uint_as_float((uint32_t)b << 16);
  w3[i] = a;
  w3[n + i] = b;
  w3[2 * n + i] = f32_to_bf16_rn(r2);
}

struct RouterArgs {
  int T, H, E, S;        // S: K parts (one per block of a tile)
  const float* bias;     // added when S == 1 (else by the part sum), may be null
  float* out;            // S == 1: logits [T][E]; else parts [S][T][E]
  int* status;
  uint64_t limit_ns;
};

__global__ void __launch_bounds__(RT_THREADS, 1)
    k_router_tc(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW, RouterArgs a) {
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[RT_STAGES], empty[RT_STAGES], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E;
  const uint32_t SB = rt_stage_bytes(E);
  const uint32_t ncols = E <= 64 ? 128u : 256u;  // two buffers of E columns (E = 64 or 128)
  const int tile = blockIdx.x / a.S, kp = blockIdx.x % a.S;
  const int nk = a.H / RT_K;
  const int c0 = kp * nk / a.S, c1 = (kp + 1) * nk / a.S;  // this block's chunks

  if (threadIdx.x == 0) {
    for (int s = 0; s < RT_STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], 32 * RT_EPI_WARPS);
    }
    tc::mbar_init(&drain, 1);
    tc::mbar_fence_init();
    abort_flag = 0;
    tc::prefetch_tensormap(&mapX);
    tc::prefetch_tensormap(&mapW);
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, ncols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const int never = 0;
  auto fail = [&]() {
    atomicCAS(a.status, 0, (int)MOE_DEV_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };

  if (warp == 0 && lane == 0) {
    // ---------------- producer: the x tile and the three W terms of each chunk
    uint32_t stage = 0, phase = 0, issued = 0, last_parity = 0;
    for (int c = c0; c < c1 && !abort_flag; ++c) {
      if (!tc::mbar_wait(&empty[stage], phase ^ 1, a.limit_ns, &abort_flag)) { fail(); break; }
      uint8_t* st = dsm + stage * SB;
      issued |= 1u << stage;
      last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
      tc::mbar_expect_tx(&full[stage], SB);
      tc::tma_load_2d(st, &mapX, c * 128, tile * RT_M, &full[stage]);
      for (int term = 0; term < 3; ++term)
        tc::tma_load_2d(st + RT_A_BYTES + term * E * 128, &mapW, c * 128, term * E, &full[stage]);
      if (++stage == RT_STAGES) { stage = 0; phase ^= 1; }
    }
    for (int s2 = 0; s2 < RT_STAGES; ++s2)
      if ((issued >> s2 & 1) && !tc::mbar_wait(&full[s2], last_parity >> s2 & 1, a.limit_ns, &never)) fail();
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer: one chunk per accumulator buffer, alternating
    uint32_t stage = 0, phase = 0;
    const uint32_t idesc = tc::idesc_bf16(RT_M, E);
    for (int c = c0; c < c1 && !abort_flag; ++c) {
      const int i = c - c0, buf = i & 1;
      if (!tc::mbar_wait(&acc_empty[buf], ((i >> 1) & 1) ^ 1, a.limit_ns, &abort_flag)) { fail(); break; }
      if (!tc::mbar_wait(&full[stage], phase, a.limit_ns, &abort_flag)) { fail(); break; }
      tc::fence_after_sync();
      const uint32_t sa = tc::smem_u32(dsm + stage * SB);
      const uint32_t d = tmem + buf * (uint32_t)E;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int term = 0; term < 3; ++term)
          tc::mma_bf16(d, tc::desc_sw128(sa + kk * 32), tc::desc_sw128(sa + RT_A_BYTES + term * E * 128 + kk * 32),
                       idesc, (kk | term) != 0);
      tc::mma_commit(&empty[stage]);
      tc::mma_commit(&acc_full[buf]);
      if (++stage == RT_STAGES) { stage = 0; phase ^= 1; }
    }
    tc::mma_commit(&drain);
    if (!tc::mbar_wait(&drain, 0, a.limit_ns, &never)) fail();
  } else if (warp >= 2) {
    // ---------------- epilogue: token row 32q + lane, columns [h E/2, (h+1) E/2)
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int m = q * 32 + lane;
    const int ncol = E / 2;  // a multiple of 16
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * ncol);
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.0f;
    bool ok = true;
    for (int c = c0; c < c1 && !abort_flag; ++c) {
      const int i = c - c0, buf = i & 1;
      if (!tc::mbar_wait(&acc_full[buf], (i >> 1) & 1, a.limit_ns, &abort_flag)) { fail(); ok = false; break; }
      tc::fence_after_sync();
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        if (p * 16 < ncol) {  // the same in the whole warp
          float v[16];
          tc::tmem_ld16(trow + buf * (uint32_t)E + p * 16, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[16 * p + j] += v[j];
        }
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&acc_empty[buf]);
    }
    const int t = tile * RT_M + m;
    if (ok && !abort_flag && t < a.T) {
      float* dst = a.S == 1 ? a.out + (size_t)t * E + h * ncol
                            : a.out + ((size_t)kp * a.T + t) * E + h * ncol;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        if (p * 16 < ncol) {
#pragma unroll
          for (int j = 0; j < 16; j += 4) {
            float4 o = make_float4(acc[16 * p + j], acc[16 * p + j + 1], acc[16 * p + j + 2], acc[16 * p + j + 3]);
            if (a.S == 1 && a.bias) {
              const float* b = a.bias + h * ncol + 16 * p + j;
              o.x += __ldg(b);
              o.y += __ldg(b + 1);
              o.z += __ldg(b + 2);
              o.w += __ldg(b + 3);
            }
            *reinterpret_cast<float4*>(dst + 16 * p + j) = o;
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, ncols);
  }
}

}  // namespace

bool router_tc_supported(int T, int H, int E) {
  return T > 512 && (E == 64 || E == 128) && H % RT_K == 0;
}

int router_tc_splits(int T, int H, int E) {
  const int tiles = (T + RT_M - 1) / RT_M;
  int S = sm_count() / tiles;
  S = imin(S, router_splits(T, E, H));  // the part buffer holds router_splits parts
  S = imin(S, H / RT_K / 8);            // at least 8 chunks per part
  return S < 1 ? 1 : S;
}

cudaError_t launch_router_tc(const uint16_t* x, const float* wr, const float* bias, float* out, int T, int H,
                             int E, int S, uint16_t* wsplit, int* status, uint64_t limit_ns, cudaStream_t s) {
  const size_t n = (size_t)E * H;
  count_launch(), k_router_wsplit<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(wr, n, wsplit);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  CUtensorMap mx, mw;
  if ((err = make_map(&mx, x, T, (uint64_t)H * 2, RT_M)) != cudaSuccess) return err;
  if ((err = make_map(&mw, wsplit, (uint64_t)3 * E, (uint64_t)H * 2, E)) != cudaSuccess) return err;
  const size_t smem = (size_t)RT_STAGES * rt_stage_bytes(E) + 1024;
  if ((err = cudaFuncSetAttribute((const void*)k_router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
      cudaSuccess)
    return err;
  RouterArgs a{T, H, E, S, bias, out, status, limit_ns};
  const int tiles = (T + RT_M - 1) / RT_M;
  count_launch(), k_router_tc<<<tiles * S, RT_THREADS, smem, s>>>(mx, mw, a);
  return cudaGetLastError();
}

}  // namespace moefp4
