// NVFP4 -> MXFP4 load-time conversion of routed-expert weights (the pages
// convert NVFP4 checkpoints to OCP MXFP4 before serving: AMD technical
// article "MiniMax-M3.1 on AMD Instinct GPUs", section "Enabling the MXFP4
// checkpoint with the AMD Quark"; vLLM PR #64273, section "Purpose").
//
// Each 32-element block: the values code x E4M3 scale x FP32 tensor scale are
// formed in FP64 (at most 31 significant bits: exact), then the OCP MXFP4
// rule: X = 2^(floor(log2 amax) - 2) clamped to [2^-127, 2^127] (amax = 0 ->
// 2^-127), codes = nearest E2M1 of v / X with ties to the even mantissa,
// |v / X| > 6 -> 6, a zero result is code 0.  Every decision is exact.
#include "common.cuh"
#include "kernels.h"

namespace moefp4 {
namespace {

__device__ __forceinline__ double e4m3_value(uint32_t b) {
  const int e = (b >> 3) & 15, m = b & 7;
  const double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
  return (b & 0x80) ? -v : v;
}

__device__ __forceinline__ double e2m1_value(uint32_t c) {
  const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  return (c & 8) ? -mag[c & 7] : mag[c & 7];
}

// Nearest E2M1 code of s (ties to the even mantissa, clamped to 6, +0 for zero).
__device__ __forceinline__ uint32_t e2m1_rne_f64(double s) {
  const double a = fabs(s);
  const uint32_t m = (a > 0.25) + (a >= 0.75) + (a > 1.25) + (a >= 1.75) + (a > 2.5) + (a >= 3.5) + (a > 5.0);
  return m | ((s < 0.0 && m) ? 8u : 0u);
}

// One thread per 32-element block of the rows of one weight matrix stack.
// Row r of matrix [E][R][K] uses tensor scale ts[e * 3 + proj(r)], where
// proj(r) = r < split ? p0 : p1 (W13: gate / up; W2: down / down).
__global__ void __launch_bounds__(256) k_nv_to_mx(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ s16,
                                                  const float* __restrict__ ts, int E, int R, int K, int split, int p0,
                                                  int p1, uint8_t* __restrict__ codes_out, uint8_t* __restrict__ s32) {
  const size_t nblk = (size_t)E * R * (K / 32);
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nblk) return;
  const size_t row = i / (K / 32);  // e * R + r
  const int b = (int)(i % (K / 32));
  const int e = (int)(row / R), r = (int)(row % R);
  const double t = (double)__ldg(ts + e * 3 + (r < split ? p0 : p1));
  const uint4 cw = __ldg(reinterpret_cast<const uint4*>(codes + row * (K / 2)) + b);
  const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
  const double sc0 = e4m3_value(__ldg(s16 + row * (K / 16) + 2 * b)) * t;
  const double sc1 = e4m3_value(__ldg(s16 + row * (K / 16) + 2 * b + 1)) * t;
  double v[32];
  double amax = 0.0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    v[j] = e2m1_value((w[j >> 3] >> (4 * (j & 7))) & 15u) * (j < 16 ? sc0 : sc1);
    amax = fmax(amax, fabs(v[j]));
  }
  int ex = -127;
  if (amax > 0.0) {
    int fe;
    frexp(amax, &fe);  // amax = f * 2^fe, f in [0.5, 1): floor(log2 amax) = fe - 1
    ex = max(-127, min(127, fe - 1 - 2));
  }
  uint32_t o[4] = {0, 0, 0, 0};
#pragma unroll
  for (int j = 0; j < 32; ++j) o[j >> 3] |= e2m1_rne_f64(ldexp(v[j], -ex)) << (4 * (j & 7));
  reinterpret_cast<uint4*>(codes_out + row * (K / 2))[b] = make_uint4(o[0], o[1], o[2], o[3]);
  s32[row * (K / 32) + b] = (uint8_t)(ex + 127);
}

cudaError_t launch_one(const uint8_t* c, const uint8_t* s, const float* ts, int E, int R, int K, int split, int p0,
                       int p1, uint8_t* co, uint8_t* so, cudaStream_t st) {
  const size_t n = (size_t)E * R * (K / 32);
  if (n == 0) return cudaSuccess;
  count_launch(), k_nv_to_mx<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(c, s, ts, E, R, K, split, p0, p1, co, so);
  return cudaGetLastError();
}

}  // namespace

namespace {

// MXFP8 -> BF16, one thread per 8 consecutive elements (their scale is the
// E8M0 byte of the 32-element block g / 4).  The E4M3 value (at most four
// significant bits, converted exactly through f16) times 2^(b - 127) is exact
// in FP32 (down to its subnormals; at or above 2^128 it overflows to inf, as
// BF16 would), so the one RNE conversion to BF16 is the only rounding, and
// it is exact wherever the value lies in BF16's normal range.  A NaN code or
// the E8M0 NaN byte 0xFF gives NaN.
__global__ void __launch_bounds__(256) k_mxfp8_to_bf16(const uint8_t* __restrict__ codes,
                                                       const uint8_t* __restrict__ scales, size_t ngroups,
                                                       uint16_t* __restrict__ out) {
  const size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= ngroups) return;
  const uint2 c = __ldg(reinterpret_cast<const uint2*>(codes) + g);
  const uint32_t sb = __ldg(scales + g / 4);
  const float sc = sb == 0xFFu ? __uint_as_float(0x7FC00000u) : e8m0_to_f32(sb);
  const uint32_t w[2] = {c.x, c.y};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = e4m3x2_to_f32x2(w[i >> 1] >> (16 * (i & 1)));
    o[i] = (uint32_t)f32_to_bf16_rn(f.x * sc) | ((uint32_t)f32_to_bf16_rn(f.y * sc) << 16);
  }
  reinterpret_cast<uint4*>(out)[g] = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

cudaError_t launch_mxfp8_to_bf16(const uint8_t* codes, const uint8_t* scales, size_t n, uint16_t* out,
                                 cudaStream_t s) {
  const size_t ngroups = n / 8;
  if (ngroups == 0) return cudaSuccess;
  count_launch(), k_mxfp8_to_bf16<<<(unsigned)((ngroups + 255) / 256), 256, 0, s>>>(codes, scales, ngroups, out);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_to_mxfp4(const Shape& sh, const ExpertsDev& ex, uint8_t* w13_out, uint8_t* w13s_out,
                                  uint8_t* w2_out, uint8_t* w2s_out, cudaStream_t s) {
  const int H = sh.H, I = sh.I, E = sh.E;
  cudaError_t err = launch_one(ex.w13, ex.w13s, ex.tscale, E, 2 * I, H, I, 0, 1, w13_out, w13s_out, s);
  if (err != cudaSuccess) return err;
  return launch_one(ex.w2, ex.w2s, ex.tscale, E, H, I, H, 2, 2, w2_out, w2s_out, s);
}

}  // namespace moefp4
