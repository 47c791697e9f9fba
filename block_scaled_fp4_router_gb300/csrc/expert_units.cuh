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

// ------------------------------------------------------- batched streams
//
// A warp streams a list of weight rows.  A row is read in 32-byte "pairs"
// (64 FP4 elements = two MX blocks, or 16 BF16 elements): lane l takes pairs
// l, l+32, ..., so one 256-bit load instruction of the warp covers 1 KB of
// contiguous bytes.  Before computing, every lane issues the loads of RB rows
// x PPL pairs (up to 8 x 32 B in flight per lane, 4 KB per warp); the scale
// bytes of a pair come with one coalesced 2- or 4-byte load.  The next work
// unit is meanwhile pulled into L2 by the block's bulk prefetch.  Per row the
// caller's sink receives the warp-reduced dot products (valid on every lane).

// One row of an FP4 stream: where its codes and scales are (Fp4Src), and
// which staged activation rows its tokens use (Fp4Tok: staged row of token t
// is tmap[t] if tmap, else tbase + t).  The two halves are asked for
// separately so that the addresses die once the loads are issued.
struct Fp4Src {
  const uint8_t* codes;
  const uint8_t* scales;
};

struct Fp4Tok {
  const int* tmap;
  int tbase;
  int nt;
};

__device__ __forceinline__ void ldg256(const void* p, uint32_t (&v)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "l"(p));
}

// Rows in flight per batch for a token bound MAXT (accumulators are RB x MAXT).
template <int MAXT, int RB>
struct BatchRows {
  static constexpr int value = MAXT == 1 ? RB : MAXT == 2 ? (RB > 1 ? RB / 2 : 1) : 1;
};

// Dot of one 32-element chunk (codes cw, pre-loaded) with staged activations.
template <int MAXT, bool NV>
__device__ __forceinline__ void fp4_chunk_acc(const uint4& cw, float s0, float s1, const Fp4Tok& r, int chunk,
                                              const uint8_t* xq_s, int xq_pitch, const float* xsc_s,
                                              int xsc_pitch, float (&acc)[MAXT]) {
  uint32_t hw[16];
  decode_chunk(cw, hw);
#pragma unroll
  for (int t = 0; t < MAXT; ++t) {
    if (t < r.nt) {
      const int row = r.tmap ? r.tmap[t] : r.tbase + t;
      const uint4 xv = *reinterpret_cast<const uint4*>(xq_s + row * xq_pitch + chunk * 16);
      const float sx = xsc_s[row * xsc_pitch + chunk];
      if (NV) {
        const float2 d = dot16x2_h(hw, xv);
        acc[t] = fmaf(fmaf(d.x, s0, d.y * s1), sx, acc[t]);
      } else {
        acc[t] = fmaf(dot32_h(hw, xv), s0 * sx, acc[t]);
      }
    }
  }
}

// srcfn(i) -> Fp4Src and tokfn(i) -> Fp4Tok for the warp's i-th row
// (0 <= i < nrows); sink(i, tok, acc).
template <int MAXT, bool NV, int RB, int PPL, class SrcFn, class TokFn, class Sink>
__device__ __forceinline__ void stream_fp4_rows(int nrows, int K, SrcFn srcfn, TokFn tokfn, const uint8_t* xq_s,
                                                int xq_pitch, const float* xsc_s, int xsc_pitch, Sink sink) {
  constexpr int R = BatchRows<MAXT, RB>::value;
  const int lane = threadIdx.x & 31;
  const int npair = K >> 6;
  const int G = (npair + 32 * PPL - 1) / (32 * PPL);
  for (int r0 = 0; r0 < nrows; r0 += R) {
    // keep each batch's loads after the previous batch's arithmetic: the
    // registers of two batches do not fit at once
    asm volatile("" ::: "memory");
    float acc[R][MAXT];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int t = 0; t < MAXT; ++t) acc[j][t] = 0.0f;
    for (int g = 0; g < G; ++g) {
      uint32_t w[R][PPL][8];
      uint32_t sc[R][PPL];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (r0 + j < nrows) {
          const Fp4Src r = srcfn(r0 + j);
#pragma unroll
          for (int i = 0; i < PPL; ++i) {
            const int p = (g * PPL + i) * 32 + lane;
            if (p < npair) {
              ldg256(r.codes + (size_t)p * 32, w[j][i]);
              sc[j][i] = NV ? __ldg(reinterpret_cast<const uint32_t*>(r.scales) + p)
                            : (uint32_t)__ldg(reinterpret_cast<const uint16_t*>(r.scales) + p);
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (r0 + j < nrows) {
          const Fp4Tok r = tokfn(r0 + j);
#pragma unroll
          for (int i = 0; i < PPL; ++i) {
            const int p = (g * PPL + i) * 32 + lane;
            if (p < npair) {
              const uint4 c0 = make_uint4(w[j][i][0], w[j][i][1], w[j][i][2], w[j][i][3]);
              const uint4 c1 = make_uint4(w[j][i][4], w[j][i][5], w[j][i][6], w[j][i][7]);
              float a0, a1, b0 = 0.0f, b1 = 0.0f;
              if (NV) {
                const float2 f0 = e4m3x2_to_f32x2(sc[j][i] & 0xffffu);
                const float2 f1 = e4m3x2_to_f32x2(sc[j][i] >> 16);
                a0 = f0.x; b0 = f0.y; a1 = f1.x; b1 = f1.y;
              } else {
                a0 = e8m0_to_f32(sc[j][i] & 0xffu);
                a1 = e8m0_to_f32(sc[j][i] >> 8);
              }
              fp4_chunk_acc<MAXT, NV>(c0, a0, b0, r, 2 * p, xq_s, xq_pitch, xsc_s, xsc_pitch, acc[j]);
              fp4_chunk_acc<MAXT, NV>(c1, a1, b1, r, 2 * p + 1, xq_s, xq_pitch, xsc_s, xsc_pitch, acc[j]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (r0 + j < nrows) {
#pragma unroll
        for (int t = 0; t < MAXT; ++t) acc[j][t] = warp_sum(acc[j][t]);
        sink(r0 + j, tokfn(r0 + j), acc[j]);
      }
    }
  }
}

// rowfn(i) -> const uint16_t* of the warp's i-th BF16 row; all rows use the
// same nt staged BF16 activation rows; sink(i, acc).
template <int MAXT, int RB, int PPL, class RowFn, class Sink>
__device__ __forceinline__ void stream_bf16_rows(int nrows, int K, RowFn rowfn, const uint16_t* x_s, int x_pitch,
                                                 int nt, Sink sink) {
  constexpr int R = BatchRows<MAXT, RB>::value;
  const int lane = threadIdx.x & 31;
  const int npair = K >> 4;
  const int G = (npair + 32 * PPL - 1) / (32 * PPL);
  for (int r0 = 0; r0 < nrows; r0 += R) {
    // keep each batch's loads after the previous batch's arithmetic: the
    // registers of two batches do not fit at once
    asm volatile("" ::: "memory");
    float acc[R][MAXT];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int t = 0; t < MAXT; ++t) acc[j][t] = 0.0f;
    for (int g = 0; g < G; ++g) {
      uint32_t w[R][PPL][8];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (r0 + j < nrows) {
          const uint16_t* row = rowfn(r0 + j);
#pragma unroll
          for (int i = 0; i < PPL; ++i) {
            const int p = (g * PPL + i) * 32 + lane;
            if (p < npair) ldg256(row + (size_t)p * 16, w[j][i]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (r0 + j < nrows) {
#pragma unroll
          for (int i = 0; i < PPL; ++i) {
            const int p = (g * PPL + i) * 32 + lane;
            if (p < npair) {
#pragma unroll
              for (int t = 0; t < MAXT; ++t) {
                if (t < nt) {
                  const uint4 x0 = *reinterpret_cast<const uint4*>(x_s + t * x_pitch + p * 16);
                  const uint4 x1 = *reinterpret_cast<const uint4*>(x_s + t * x_pitch + p * 16 + 8);
                  const uint32_t xx[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                  float a = acc[j][t];
#pragma unroll
                  for (int q = 0; q < 8; ++q) {
                    a = fmaf(bf16_lo(w[j][i][q]), bf16_lo(xx[q]), a);
                    a = fmaf(bf16_hi(w[j][i][q]), bf16_hi(xx[q]), a);
                  }
                  acc[j][t] = a;
                }
              }
            }
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      if (r0 + j < nrows) {
#pragma unroll
        for (int t = 0; t < MAXT; ++t) acc[j][t] = warp_sum(acc[j][t]);
        sink(r0 + j, acc[j]);
      }
    }
  }
}

// Asks the TMA engine to pull [p, p + bytes) from HBM into L2 (no registers,
// no completion to wait for).  p and bytes must be multiples of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
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
