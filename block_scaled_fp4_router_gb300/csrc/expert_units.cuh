// Warp- and block-level building blocks of the expert FFNs (A5 - A8) used by
// both the unfused kernels and the fused single-launch decode.
//
// A weight row is streamed once from HBM with 16-byte loads: lane l takes the
// 16-byte chunks l, l+32, l+64, ... (for FP4 one chunk = 32 elements = one MX
// block; for BF16 one chunk = 8 elements), so a warp's load instruction covers
// 512 contiguous bytes.  The token activations the row is multiplied with sit
// in shared memory in the same chunk order, so the shared-memory reads of a
// warp are conflict-free.
#pragma once

#include "common.cuh"

namespace moefp4 {

// Decode one 16-byte chunk of E2M1 codes (32 elements) to 16 f16x2.
__device__ __forceinline__ void decode_chunk(const uint4& q, uint32_t (&h)[16]) {
  uint32_t t[4];
  e2m1x8_to_h2x4(q.x, t);
  h[0] = t[0]; h[1] = t[1]; h[2] = t[2]; h[3] = t[3];
  e2m1x8_to_h2x4(q.y, t);
  h[4] = t[0]; h[5] = t[1]; h[6] = t[2]; h[7] = t[3];
  e2m1x8_to_h2x4(q.z, t);
  h[8] = t[0]; h[9] = t[1]; h[10] = t[2]; h[11] = t[3];
  e2m1x8_to_h2x4(q.w, t);
  h[12] = t[0]; h[13] = t[1]; h[14] = t[2]; h[15] = t[3];
}

// sum_i e2m1(w_i) e2m1(x_i) over one chunk, w pre-decoded.  Exact (each f16
// lane of the two accumulators adds 8 products of magnitude <= 36 in steps of
// 1/4, so every partial sum is representable).
__device__ __forceinline__ float dot32_h(const uint32_t (&hw)[16], const uint4& x) {
  uint32_t hx[16];
  decode_chunk(x, hx);
  uint32_t a0 = 0, a1 = 0;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    a0 = hfma2u(hw[i], hx[i], a0);
    a1 = hfma2u(hw[i + 1], hx[i + 1], a1);
  }
  return h2sum(a0) + h2sum(a1);
}

// The two 16-element halves of a chunk separately (NVFP4 scales every 16).
__device__ __forceinline__ float2 dot16x2_h(const uint32_t (&hw)[16], const uint4& x) {
  uint32_t hx[16];
  decode_chunk(x, hx);
  uint32_t a0 = 0, a1 = 0, b0 = 0, b1 = 0;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    a0 = hfma2u(hw[i], hx[i], a0);
    a1 = hfma2u(hw[i + 1], hx[i + 1], a1);
    b0 = hfma2u(hw[8 + i], hx[8 + i], b0);
    b1 = hfma2u(hw[8 + i + 1], hx[8 + i + 1], b1);
  }
  return make_float2(h2sum(a0) + h2sum(a1), h2sum(b0) + h2sum(b1));
}

// One warp: partial dot products of one FP4 weight row (K elements, codes at
// wrow, scales at srow: E8M0 per 32 or E4M3 per 16) with nt <= NT MXFP4
// activation rows staged in shared memory: token t uses staged row
// r = tmap[t] (tmap == nullptr: r = t), codes at xq_s + r*xq_pitch and scale
// values (floats) at xsc_s + r*xsc_pitch.  acc[t] receives this lane's share;
// the caller reduces over the warp.
template <int NT, bool NV>
__device__ __forceinline__ void fp4_row_dot(const uint8_t* __restrict__ wrow,
                                            const uint8_t* __restrict__ srow, int K,
                                            const uint8_t* xq_s, int xq_pitch, const float* xsc_s,
                                            int xsc_pitch, const int* tmap, int nt, float (&acc)[NT]) {
  const int lane = threadIdx.x & 31;
  const int nch = K >> 5;
  for (int c0 = 0; c0 < nch; c0 += 128) {
    uint4 w[4];
    uint32_t sc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = c0 + i * 32 + lane;
      if (c < nch) {
        w[i] = ldg_stream(wrow + (size_t)c * 16);
        sc[i] = NV ? (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(srow) + c)
                   : (uint32_t)__ldg(srow + c);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = c0 + i * 32 + lane;
      if (c < nch) {
        uint32_t hw[16];
        decode_chunk(w[i], hw);
        float s0, s1 = 0.0f;
        if (NV) {
          const float2 f = e4m3x2_to_f32x2(sc[i]);
          s0 = f.x;
          s1 = f.y;
        } else {
          s0 = e8m0_to_f32(sc[i]);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < nt) {
            const int r = tmap ? tmap[t] : t;
            const uint4 xv = *reinterpret_cast<const uint4*>(xq_s + r * xq_pitch + c * 16);
            const float sx = xsc_s[r * xsc_pitch + c];
            if (NV) {
              const float2 d = dot16x2_h(hw, xv);
              acc[t] = fmaf(fmaf(d.x, s0, d.y * s1), sx, acc[t]);
            } else {
              acc[t] = fmaf(dot32_h(hw, xv), s0 * sx, acc[t]);
            }
          }
        }
      }
    }
  }
}

// One warp: partial dot products of one BF16 weight row (K elements) with
// nt <= NT BF16 activation rows staged in shared memory (x_s + t*x_pitch
// elements).
template <int NT>
__device__ __forceinline__ void bf16_row_dot(const uint16_t* __restrict__ wrow, int K,
                                             const uint16_t* x_s, int x_pitch, int nt,
                                             float (&acc)[NT]) {
  const int lane = threadIdx.x & 31;
  const int nch = K >> 3;
  for (int c0 = 0; c0 < nch; c0 += 128) {
    uint4 w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = c0 + i * 32 + lane;
      if (c < nch) w[i] = ldg_stream(wrow + (size_t)c * 8);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = c0 + i * 32 + lane;
      if (c < nch) {
        const uint32_t ww[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
        float wf[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          wf[2 * j] = bf16_lo(ww[j]);
          wf[2 * j + 1] = bf16_hi(ww[j]);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < nt) {
            const uint4 xv = *reinterpret_cast<const uint4*>(x_s + t * x_pitch + c * 8);
            float a = acc[t];
            a = fmaf(wf[0], bf16_lo(xv.x), a);
            a = fmaf(wf[1], bf16_hi(xv.x), a);
            a = fmaf(wf[2], bf16_lo(xv.y), a);
            a = fmaf(wf[3], bf16_hi(xv.y), a);
            a = fmaf(wf[4], bf16_lo(xv.z), a);
            a = fmaf(wf[5], bf16_hi(xv.z), a);
            a = fmaf(wf[6], bf16_lo(xv.w), a);
            a = fmaf(wf[7], bf16_hi(xv.w), a);
            acc[t] = a;
          }
        }
      }
    }
  }
}

// One warp, lane c holds G and U of column c of a 32-column block for one
// assignment: h = SiLU(G) * U, then OCP MXFP4 quantisation of the block
// (model card, section "Model Overview": routed-expert activations are
// MXFP4).  Writes 16 code bytes and one scale byte.
__device__ __forceinline__ void swiglu_quant_block(float g, float u, uint8_t* hq16, uint8_t* hs1) {
  const int lane = threadIdx.x & 31;
  const float h = silu(g) * u;
  const float amax = warp_max(fabsf(h));
  const int e = mx_scale_exp(amax);
  const uint32_t code = e2m1_rne(h * pow2_neg(e));
  const uint32_t hi = __shfl_down_sync(FULL, code, 1);
  if ((lane & 1) == 0) hq16[lane >> 1] = (uint8_t)(code | (hi << 4));
  if (lane == 0) *hs1 = (uint8_t)(e + 127);
}

// Stage MXFP4 activation rows into shared memory: codes (K/2 bytes per row)
// with 16-byte copies and scales converted to floats.  rows[i] gives the
// source row of staged row i.  All threads of the block take part.
__device__ __forceinline__ void stage_mx_rows(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                              int K, const int* rows, int n, uint8_t* q_s, float* s_s,
                                              bool coherent) {
  const int cpr = K / 32;  // 16-byte chunks per row == scales per row
  for (int i = threadIdx.x; i < n * cpr; i += blockDim.x) {
    const int r = i / cpr, c = i - r * cpr;
    const size_t src = (size_t)rows[r];
    const uint4* sp = reinterpret_cast<const uint4*>(q + src * (K / 2)) + c;
    uint4 v = coherent ? __ldcg(sp) : __ldg(sp);
    reinterpret_cast<uint4*>(q_s + (size_t)r * (K / 2))[c] = v;
    const uint8_t sb = coherent ? __ldcg(s + src * cpr + c) : __ldg(s + src * cpr + c);
    s_s[r * cpr + c] = e8m0_to_f32(sb);
  }
}

}  // namespace moefp4
