// Device helpers shared by the kernels of libmoefp4 (sm_103a).
//
// Number formats (model card "amd/MiniMax-M3.1-Flash-Quark-MXFP4", section
// "Model Overview": OCP MXFP4 weights and activations; AMD technical article
// "MiniMax-M3.1 on AMD Instinct GPUs", section "MiniMax-M3.1 at a glance":
// NVFP4 experts):
//   E2M1  1 sign, 2 exponent (bias 1), 1 mantissa bit: +-{0,.5,1,1.5,2,3,4,6}
//   E8M0  2^(b-127)
//   E4M3  OCP FP8 e4m3 ("fn")
// Element pairs are decoded with the sm_100-family conversion instructions
// (cvt.rn.f16x2.e2m1x2 / .e4m3x2), which are exact for these formats.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "layout.h"

namespace moefp4 {

constexpr uint32_t FULL = 0xffffffffu;

// ------------------------------------------------------------------ BF16

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ------------------------------------------------------------ scale bytes

// E8M0 byte -> float 2^(b-127).  b = 0 is 2^-127 (an FP32 subnormal); 0xFF
// (NaN in E8M0) is outside what the library produces or accepts.
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
  return b ? __uint_as_float(b << 23) : __uint_as_float(0x00400000u);
}

// Two E4M3 bytes (low byte first) -> two floats.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_bytes) {
  uint32_t h2;
  uint16_t in = (uint16_t)two_bytes;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

// -------------------------------------------------------------- E2M1 pairs

// One 32-bit word of packed E2M1 codes (8 elements) -> four f16x2 holding the
// exact element values; f16x2 i holds the two elements of byte i.
__device__ __forceinline__ void e2m1x8_to_h2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ float h2sum(uint32_t a) {
  float2 f = __half22float2(*reinterpret_cast<__half2*>(&a));
  return f.x + f.y;
}

// ------------------------------------------------------ MXFP4 quantisation

// Exponent of the OCP MX shared scale for a block with maximum magnitude amax:
// floor(log2(amax)) - 2, clamped to [-127, 127]; amax = 0 (or subnormal, whose
// floor(log2) is below -126) gives -127.
__device__ __forceinline__ int mx_scale_exp(float amax) {
  const int ef = (int)((__float_as_uint(amax) >> 23) & 0xff);
  return ef == 0 ? -127 : max(ef - 127 - 2, -127);
}

// 2^-e for e in [-127, 125], exactly.
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// E2M1 code of s (already divided by the block scale): nearest magnitude, ties
// to the even mantissa, clamped to 6; a zero result is the +0 code.
__device__ __forceinline__ uint32_t e2m1_rne(float s) {
  const float a = fabsf(s);
  uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
               (a >= 3.5f) + (a > 5.0f);
  return m | ((s < 0.0f && m) ? 8u : 0u);
}

// Eight E2M1 codes of v[i] * inv packed low nibble first (element i in bits
// 4i .. 4i+3), by the hardware's round-to-nearest-even, saturating E2M1
// conversion (two values per cvt): the same codes as e2m1_rne, except that
// the conversion keeps the sign of a value that rounds to zero, so those
// nibbles are cleared to the +0 code afterwards.
__device__ __forceinline__ uint32_t e2m1x8_rne(const float (&v)[8], float inv) {
  uint32_t packed;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(packed)
      : "f"(v[0] * inv), "f"(v[1] * inv), "f"(v[2] * inv), "f"(v[3] * inv), "f"(v[4] * inv), "f"(v[5] * inv),
        "f"(v[6] * inv), "f"(v[7] * inv));
  const uint32_t mag = packed & 0x77777777u;
  const uint32_t nonzero = (mag + 0x77777777u) & 0x88888888u;  // bit 3 of each nibble whose magnitude is not 0
  return packed & (0x77777777u | nonzero);
}

// Eight E4M3 codes of v[i] * inv, element i in byte i of the pair (lo, hi),
// by the hardware's round-to-nearest-even E4M3 conversion saturating at
// +-448 (two values per cvt); codes of magnitude 0 are cleared to +0.
__device__ __forceinline__ uint2 e4m3x8_rne(const float (&v)[8], float inv) {
  uint32_t lo, hi;
  asm("{\n\t.reg .b16 h0, h1, h2, h3;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h0, %3, %2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h1, %5, %4;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h2, %7, %6;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h3, %9, %8;\n\t"
      "mov.b32 %0, {h0, h1};\n\t"
      "mov.b32 %1, {h2, h3};\n\t}"
      : "=r"(lo), "=r"(hi)
      : "f"(v[0] * inv), "f"(v[1] * inv), "f"(v[2] * inv), "f"(v[3] * inv), "f"(v[4] * inv), "f"(v[5] * inv),
        "f"(v[6] * inv), "f"(v[7] * inv));
  auto clear_neg_zero = [](uint32_t w) {
    const uint32_t nonzero = ((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) & 0x80808080u;  // bit 7 of each nonzero byte
    return w & (0x7F7F7F7Fu | nonzero);
  };
  return make_uint2(clear_neg_zero(lo), clear_neg_zero(hi));
}

// One E4M3 code of v (the hardware's nearest-even conversion, saturating at
// +-448); a code of magnitude 0 is +0.
__device__ __forceinline__ uint32_t e4m3_rne1(float v) {
  uint32_t w;
  asm("{\n\t.reg .b16 h;\n\tcvt.rn.satfinite.e4m3x2.f32 h, %2, %1;\n\tcvt.u32.u16 %0, h;\n\t}"
      : "=r"(w)
      : "f"(v), "f"(0.0f));
  w &= 0xFFu;
  return (w & 0x7Fu) ? w : 0u;
}

// MXFP8 scale exponent of a 32-element block: X = 2^(floor(log2 amax) - 8),
// -127 for an all-zero block (or a subnormal amax).
__device__ __forceinline__ int mx8_scale_exp(float amax) {
  const int ef = (int)((__float_as_uint(amax) >> 23) & 0xff);
  return ef == 0 ? -127 : max(ef - 127 - 8, -127);
}

// MXFP4 codes of one 32-element BF16 block (16 bytes to dq, 16-byte aligned;
// xb 16-byte aligned) and its E8M0 byte, by one thread.  The same codes and
// scales as the standalone quantiser (mx_scale_exp, e2m1_rne).
__device__ __forceinline__ uint8_t quant32(const uint16_t* xb, uint8_t* dq) {
  const uint4* src = reinterpret_cast<const uint4*>(xb);
  uint4 raw[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) raw[j] = __ldg(src + j);
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w4[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w4[h])), fabsf(bf16_hi(w4[h]))));
  }
  const int ex = mx_scale_exp(amax);
  const float inv = pow2_neg(ex);
  uint32_t c[4];
#pragma unroll 1
  for (int j = 0; j < 4; ++j) {
    const uint32_t w4[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
    uint32_t word = 0;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      word |= e2m1_rne(bf16_lo(w4[h]) * inv) << (8 * h);
      word |= e2m1_rne(bf16_hi(w4[h]) * inv) << (8 * h + 4);
    }
    c[j] = word;
  }
  *reinterpret_cast<uint4*>(dq) = make_uint4(c[0], c[1], c[2], c[3]);
  return (uint8_t)(ex + 127);
}

// One thread quantises 8 consecutive BF16 values x[8g .. 8g+7] to MXFP8
// (E4M3, one E8M0 scale per 32: X = 2^(floor(log2 amax) - 8)); the 4 threads
// of a block share their maxima with two shuffles, as in quant8_values.
__device__ __forceinline__ void quant8_values_mx8(const uint4 q, size_t g, bool valid, uint8_t* __restrict__ codes,
                                                  uint8_t* __restrict__ scales) {
  float v[8];
  float amax = 0.0f;
  if (valid) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  if (!valid) return;
  const int ef = (int)((__float_as_uint(amax) >> 23) & 0xff);
  const int e = ef == 0 ? -127 : max(ef - 127 - 8, -127);
  reinterpret_cast<uint2*>(codes)[g] = e4m3x8_rne(v, pow2_neg(e));
  if ((g & 3) == 0) scales[g >> 2] = (uint8_t)(e + 127);
}

// One thread quantises 8 consecutive BF16 values x[8g .. 8g+7]; the 4 threads
// of a 32-element block (consecutive lanes, g = 4j .. 4j+3) share their maxima
// with two shuffles.  All 32 lanes of the warp must call it together; lanes
// with valid == false only join the shuffles.  Writes 4 code bytes and, from
// the first lane of the block, the E8M0 scale byte.
// quant8_values takes the 8 values already loaded (q = x[8g .. 8g+7]).
__device__ __forceinline__ void quant8_values(const uint4 q, size_t g, bool valid, uint8_t* __restrict__ codes,
                                              uint8_t* __restrict__ scales) {
  float v[8];
  float amax = 0.0f;
  if (valid) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  if (!valid) return;
  const int e = mx_scale_exp(amax);
  reinterpret_cast<uint32_t*>(codes)[g] = e2m1x8_rne(v, pow2_neg(e));
  if ((g & 3) == 0) scales[g >> 2] = (uint8_t)(e + 127);
}

__device__ __forceinline__ void quant8_group(const uint16_t* __restrict__ x, size_t g, bool valid,
                                             uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const uint4 q = valid ? *reinterpret_cast<const uint4*>(x + g * 8) : make_uint4(0, 0, 0, 0);
  quant8_values(q, g, valid, codes, scales);
}

// -------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

// The warp's largest of v >= 0 (finite): the bit patterns of non-negative
// floats order as the values, so one integer max reduction replaces five
// shuffle rounds.
__device__ __forceinline__ float warp_max_nonneg(float v) {
  return __uint_as_float(__reduce_max_sync(FULL, __float_as_uint(v)));
}

// Checked builds (compiled with MOEFP4_CHECKED=1) record a caller-given index
// that is out of range as MOE_ERR_INVALID_ARG in the status word; every build
// leaves such an index out (no access through it).
#ifndef MOEFP4_CHECKED
#define MOEFP4_CHECKED 0
#endif
__device__ __forceinline__ void report_bad_index(int* status) {
  if (MOEFP4_CHECKED && status) atomicCAS(status, 0, (int)MOE_DEV_INVALID);
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// SiLU for the batched GEMM epilogues, where it runs on every element of the
// accumulator: the fast exponential and division intrinsics, a few ulp from
// silu() for |g| < 88 (where h is later requantised or rounded to BF16), and
// 0 below (the approximate reciprocal of the infinite denominator is 0).
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// ------------------------------------------------------------- memory ops

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_relaxed(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A ticket arrival: releases the caller's stores (and, after a block
// barrier, its block's) and acquires those of every earlier arrival, in one
// atomic round trip instead of a fence followed by a relaxed atomic.
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait until *p >= target.  Bounded twice over: by limit_ns of wall-clock time
// and by an iteration cap; on expiry it records MOE_DEV_TIMEOUT in *status
// (first error wins) and returns false.  Also returns false at once when an
// earlier wait of the same launch already timed out.
__device__ __forceinline__ bool wait_at_least(const int* p, int target, int* status,
                                              uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  unsigned ns = 32;
  for (uint32_t it = 0; it < (1u << 24); ++it) {
    if (ld_acquire(p) >= target) return true;
    if (ld_acquire(status) == (int)MOE_DEV_TIMEOUT) return false;
    if (globaltimer_ns() - t0 > limit_ns) break;
    __nanosleep(ns);
    if (ns < 256) ns <<= 1;
  }
  atomicCAS(status, 0, (int)MOE_DEV_TIMEOUT);
  return false;
}

}  // namespace moefp4
