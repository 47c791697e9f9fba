// A10 on tensor cores: the whole MoE layer for decode steps of 1-16 tokens in
// one launch, every contraction on tcgen05 (AMD technical article
// "MiniMax-M3.1 on AMD Instinct GPUs", section "What we Optimized": the "mono
// decode" path runs a pure decode step of at most 16 tokens as one fused MoE
// launch).
//
// A decode step streams every touched weight byte once, so the layer is
// bound by HBM.  The weights are the MMA's A operand (128 weight rows per
// MMA, moved by TMA through a shared-memory ring) and the 1-16 token rows are
// a 16-row B operand, so every SM keeps weights in flight without spending
// CUDA-core issue slots on FP4 decoding.
//
// Work units (one block per SM, cooperative launch, the same static
// round-robin list in every block):
//   SGU  shared gate/up:  128 gate + 128 up rows x a K part (BF16, kind::f16)
//   RGU  routed gate/up:  expert slot x 128 gate + 128 up rows x a K part (FP4)
//   SDN  shared down:     128 rows of H x a K part (BF16)
//   RDN  routed down:     128 rows of H x one expert slot (FP4, whole K)
// Split-K gate/up parts write FP32 partial sums; the block that delivers the
// last part of a tile (an atomic ticket) sums the parts in a fixed order and
// runs the tile's epilogue: SwiGLU to BF16 h (shared) or SwiGLU + MXFP4
// requantise (routed).  Down parts are counted; once all are stored, the
// weighted combine out = BF16(ys + sum_j w_j y_j), summed in a fixed order,
// runs as items of 128 columns x 4 tokens spread over all blocks.  Results
// are therefore bit-reproducible run to run.  With the shared expert folded
// into the FP4 table, every token has one more slot (the table's last
// expert, weight 1) and there are no SGU / SDN units.
//
// Warp roles: warp 0 issues TMA, warp 1 issues tcgen05.cp / tcgen05.mma,
// warps 2-5 are the epilogue (one TMEM lane = one weight row each).  Before
// their first unit the epilogue warps compute this block's router rows and
// its slice of the MXFP4 quantisation of x; once every block has done so they
// build the routing (top-k, sort by expert) in shared memory and release the
// producer and MMA warps onto the routed units.  There is no L2 prefetch
// beyond the stage ring: extra traffic measurably slows the latency-bound
// hand-offs more than it saves in streaming.
//
// Every wait is bounded (MOE_DEV_TIMEOUT in the status word); the last block
// out resets the counters, and each finishing block resets its ticket.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "routing.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moefp4 {
namespace {

constexpr int DT = 192;                 // threads: TMA warp, MMA warp, 4 epilogue warps
constexpr int EPI_THREADS = 128;
// A 4-stage ring, of which the host lets `depth` stages be in flight: two
// (~70-90 KB per SM, ~10-13 MB over the GPU) cover HBM's bandwidth-latency
// product for a 1-4 token step, where a deeper queue would only slow the
// latency-bound hand-offs between the steps; four for the larger steps,
// which stream hundreds of MB.
constexpr int DSTAGES = 4;
// byte offsets inside one stage (swizzled tiles on 1024-byte boundaries)
constexpr uint32_t ST_A0 = 0, ST_A1 = 16384;       // 128 rows x 128 B each
constexpr uint32_t ST_B0 = 32768, ST_B1 = 34816;   // 16 rows x 128 B each
// Scale blocks (512 B each): per 256-element K chunk and 128 rows, NBLK = 2
// for MXFP4 (E8M0 per 32) or 4 for NVFP4 (UE4M3 per 16).  Tile / half h of a
// stage keeps its blocks at ST_SFA / ST_SFB + h * NBLK * 512, and their TMEM
// copies at columns +4 NBLK h (A) and +4 NBLK (2 + h) (B) of the stage's
// 16 NBLK scale columns (stage s from column TM_SF + 16 NBLK s).
constexpr uint32_t ST_SFA = 36864;
template <bool NV> __host__ __device__ constexpr int nblk() { return NV ? 4 : 2; }
template <bool NV> __host__ __device__ constexpr uint32_t st_sfb() { return ST_SFA + 2 * 512 * nblk<NV>(); }
template <bool NV> __host__ __device__ constexpr uint32_t stage_bytes() { return st_sfb<NV>() + 2 * 512 * nblk<NV>(); }
constexpr uint32_t A_TILE = 16384, B_TILE = 2048;
// TMEM: NACC 32-column accumulators (the MMA runs up to NACC units ahead of
// the epilogue), then 16 NBLK scale columns per stage.
constexpr int NACC = 4;
template <bool NV> __host__ __device__ constexpr uint32_t tmem_cols() { return NV ? 512u : 256u; }
constexpr uint32_t TM_SF = 32 * NACC;
constexpr int MAXN = MAX_DECODE_T * MAX_TOPK;

enum UnitKind { U_SGU = 0, U_RGU = 1, U_SDN = 2, U_RDN = 3 };

struct DcArgs {
  int T, H, I, E, k;         // E experts in the table, k assignments per token
  int Er, kr;                // the router's experts and top-k (E - 1, k - 1 with the
                             // shared expert folded into the table as expert Er)
  int G;                     // blocks in the launch
  int s_sgu, s_rgu, s_sdn;   // split-K parts
  int n_sgu, n_sdn;          // unit counts that do not depend on the routing
  int nslot_max;             // min(T k, E): ticket slots
  int shared;
  int nv;                    // NVFP4 experts (UE4M3 scales per 16, FP32 tensor scales)
  int score;                 // SCORE_SOFTMAX (the bias is part of the logit) or SCORE_SIGMOID
  const uint8_t* w13s_mma;   // prepared routed weight scales
  const uint8_t* w2s_mma;
  const float* tscale;       // NVFP4: [E, 3] (gate, up, down)
  const float* wr;
  const float* bias;
  const uint16_t* x;
  uint16_t* out;
  int* ids_out;
  float* w_out;
  int* ctr;
  int* tickets;
  unsigned long long* logit64;  // [T, E]: (launch number << 32) | FP32 bits
  uint8_t* xq;               // [T, H/2]
  uint8_t* xs_mma;           // [H/128][512] E8M0 (MXFP4) or [H/64][512] UE4M3 (NVFP4)
  int* xshift;               // NVFP4: [16] per-row power of two of the UE4M3 x scales
  unsigned long long* rowmax;  // NVFP4: [T k] (launch << 32) | (largest h scale exponent + 256)
  uint8_t* hq;               // [T k, I/2] sorted-assignment rows
  uint8_t* hs_mma;           // [slots][I/128][512] E8M0 (MXFP4) or [slots][I/64][512] UE4M3 (NVFP4)
  uint8_t* hsc;              // NVFP4: E8M0 bytes of h [T k][I/32]
  int depth;                 // stages in flight (<= DSTAGES)
  uint16_t* h_shared;        // [T, I]
  float* gu_sh;              // [s_sgu][T][2I]
  float* gu_r;               // [s_rgu][T k][2I]
  float* ys;                 // [s_sdn][T][H]
  float* y_assign;           // [T k][H]
  uint64_t limit_ns;
};

struct DcMaps {
  CUtensorMap w13r, w2r, w13s, w2s;  // weights: boxes of 128 rows x 128 B
  CUtensorMap xq, x, hsh, hq;        // activations: boxes of 16 rows x 128 B
};

// Routing of the step, built by the epilogue warps of every block.
struct DcRouting {
  int ids[MAXN];
  float w[MAXN];
  int inv[MAXN];          // assignment t*k+j -> sorted position
  int tok[MAXN];          // sorted position -> token
  int sorted_e[MAXN];     // sorted position -> expert
  int slot_e[MAXN];       // slot -> expert (distinct experts, ascending)
  int slot_beg[MAXN + 1]; // slot -> first sorted position
  int wcount[EPI_THREADS / 32];
  int n_slots;
};

struct Unit {
  int kind;
  int tile;   // 128-row tile: of I (gate/up) or of H (down)
  int part;   // split-K part
  int slot;   // routed units
  int st0, st1;
};

__device__ __forceinline__ int units_total(const DcArgs& a, int n_slots) {
  return a.n_sgu + n_slots * (a.I / 128) * a.s_rgu + a.n_sdn + n_slots * (a.H / 128);
}

// Part p of `stages` stages split into s near-equal parts.
__device__ __forceinline__ void part_range(int stages, int s, int p, int& st0, int& st1) {
  st0 = p * stages / s;
  st1 = (p + 1) * stages / s;
}

// v-th shared down unit: 128-row tile of H, K part over stages of two chunks.
__device__ __forceinline__ Unit sdn_unit(const DcArgs& a, int v) {
  Unit U{};
  U.kind = U_SDN;
  U.tile = v / a.s_sdn;
  U.part = v % a.s_sdn;
  part_range((a.I / 64 + 1) / 2, a.s_sdn, U.part, U.st0, U.st1);
  return U;
}

// v-th routed down unit: 128-row tile of H x expert slot, whole K.
__device__ __forceinline__ Unit rdn_unit(const DcArgs& a, int n_slots, int v) {
  Unit U{};
  U.kind = U_RDN;
  U.tile = v / n_slots;
  U.slot = v % n_slots;
  U.st0 = 0;
  U.st1 = (a.I / 256 + 1) / 2;
  return U;
}

__device__ Unit unit_at(const DcArgs& a, int n_slots, int u) {
  Unit U{};
  const int nbI = a.I / 128;
  if (u < a.n_sgu) {
    U.kind = U_SGU;
    U.tile = u / a.s_sgu;
    U.part = u % a.s_sgu;
    part_range(a.H / 64, a.s_sgu, U.part, U.st0, U.st1);
    return U;
  }
  u -= a.n_sgu;
  const int n_rgu = n_slots * nbI * a.s_rgu;
  if (u < n_rgu) {
    U.kind = U_RGU;
    U.slot = u / (nbI * a.s_rgu);
    U.tile = (u / a.s_rgu) % nbI;
    U.part = u % a.s_rgu;
    part_range(a.H / 256, a.s_rgu, U.part, U.st0, U.st1);
    return U;
  }
  u -= n_rgu;
  if (u < a.n_sdn) return sdn_unit(a, u);
  return rdn_unit(a, n_slots, u - a.n_sdn);
}

__device__ __forceinline__ void epi_sync() { tc::named_sync(1, EPI_THREADS); }

// sum over p < S <= MAXS of src[p * stride], in ascending p, every load issued first.
template <int MAXS = DC_MAX_SPLIT>
__device__ __forceinline__ float sum_parts(const float* src, size_t stride, int S) {
  float v[MAXS];
#pragma unroll
  for (int p = 0; p < MAXS; ++p) v[p] = p < S ? __ldcg(src + p * stride) : 0.0f;
  float s = 0.0f;
#pragma unroll
  for (int p = 0; p < MAXS; ++p)
    if (p < S) s += v[p];
  return s;
}

// v[base + t] for a runtime t < 16 without indexing registers dynamically.
__device__ __forceinline__ float pick16(const float (&v)[32], int base, int t) {
  float r = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) r = i == t ? v[base + i] : r;
  return r;
}

// ----------------------------------------------------- epilogue-warp prologue

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Router row e for all tokens (FP32 weights and accumulation), 128 threads.
// Tokens go in groups of 8; within a group every load of a pass (4 x 8
// elements per thread) is in flight before the FMAs, since these loads
// compete with the weight streams for HBM.
__device__ void router_row(const DcArgs& a, int e, int et, float (*red_s)[MAX_DECODE_T], uint32_t epoch) {
  const int T = a.T, H = a.H;
  const int w = et >> 5, lane = et & 31;
  constexpr int PASS = EPI_THREADS * 8;
  const float* wrow = a.wr + (size_t)e * H;
  constexpr int TG = 8;
  for (int t0 = 0; t0 < T; t0 += TG) {
    float acc[TG];
#pragma unroll
    for (int tt = 0; tt < TG; ++tt) acc[tt] = 0.0f;
    for (int k0 = et * 8; k0 < H; k0 += 4 * PASS) {
      uint4 wv[8];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int kk = k0 + c * PASS;
        wv[2 * c] = kk < H ? __ldg(reinterpret_cast<const uint4*>(wrow + kk)) : make_uint4(0, 0, 0, 0);
        wv[2 * c + 1] = kk < H ? __ldg(reinterpret_cast<const uint4*>(wrow + kk + 4)) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int tt = 0; tt < TG; ++tt) {
        if (t0 + tt < T) {
          const uint16_t* xr = a.x + (size_t)(t0 + tt) * H;
          uint4 xv[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int kk = k0 + c * PASS;
            xv[c] = kk < H ? __ldg(reinterpret_cast<const uint4*>(xr + kk)) : make_uint4(0, 0, 0, 0);
          }
          float s = acc[tt];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 q = xv[c], wa = wv[2 * c], wb = wv[2 * c + 1];
            s = fmaf(bf16_lo(q.x), __uint_as_float(wa.x), s);
            s = fmaf(bf16_hi(q.x), __uint_as_float(wa.y), s);
            s = fmaf(bf16_lo(q.y), __uint_as_float(wa.z), s);
            s = fmaf(bf16_hi(q.y), __uint_as_float(wa.w), s);
            s = fmaf(bf16_lo(q.z), __uint_as_float(wb.x), s);
            s = fmaf(bf16_hi(q.z), __uint_as_float(wb.y), s);
            s = fmaf(bf16_lo(q.w), __uint_as_float(wb.z), s);
            s = fmaf(bf16_hi(q.w), __uint_as_float(wb.w), s);
          }
          acc[tt] = s;
        }
      }
    }
#pragma unroll
    for (int tt = 0; tt < TG; ++tt) {
      const float v = warp_sum(acc[tt]);
      if (lane == 0 && t0 + tt < T) red_s[w][t0 + tt] = v;
    }
  }
  epi_sync();
  if (et < T) {
    float s = red_s[0][et];
    for (int ww = 1; ww < EPI_THREADS / 32; ++ww) s += red_s[ww][et];
    if (a.bias && a.score == SCORE_SOFTMAX) s += a.bias[e];
    // one 64-bit store carries the value and this launch's number: a reader
    // that sees the number has the value, with no fence or counter between
    st_relaxed_u64(a.logit64 + (size_t)et * a.Er + e, ((unsigned long long)epoch << 32) | __float_as_uint(s));
  }
  epi_sync();
}

// MXFP4 quantisation of one 32-element block i = (token row t < 16, block b
// of H/32): 16 code bytes of xq and byte b % 4 of the MMA-layout scale word
// of row t in group b / 4 (word 4t of that group's 512-byte block).  Rows
// t >= T get a zero scale byte.  Same arithmetic as the standalone quantiser.
__device__ void quant_block(const DcArgs& a, int i) {
  const int nb = a.H / 32;
  const int t = i / nb, b = i % nb;
  uint8_t sb = 0;
  if (t < a.T) {
    const uint4* src = reinterpret_cast<const uint4*>(a.x + (size_t)t * a.H + b * 32);
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
    *reinterpret_cast<uint4*>(a.xq + (size_t)t * (a.H / 2) + b * 16) = make_uint4(c[0], c[1], c[2], c[3]);
    sb = (uint8_t)(ex + 127);
  }
  a.xs_mma[(size_t)(b / 4) * 512 + t * 16 + (b % 4)] = sb;
}

// One warp reads token t's E logits once every one carries this launch's
// number (bounded wait; false on timeout).  Lane l gets experts l, l+32, ...
__device__ bool wait_logit_row(const DcArgs& a, int t, uint32_t epoch, float (&v)[8]) {
  const int lane = threadIdx.x & 31;
  const unsigned long long* row = a.logit64 + (size_t)t * a.Er;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    bool mine = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      v[i] = 0.0f;
      if (e < a.Er) {
        const unsigned long long w = ld_relaxed_u64(row + e);
        mine &= (uint32_t)(w >> 32) == epoch;
        v[i] = __uint_as_float((uint32_t)w);
      }
    }
    if (__all_sync(FULL, mine)) return true;
    if (__shfl_sync(FULL, (int)(globaltimer_ns() - t0 > a.limit_ns), 0)) return false;
    __nanosleep(32);
  }
}

// 2^p as a UE4M3 byte: normal for p >= -6, subnormal down to 2^-9, 0 below
// (p <= 8 always: the row shift puts the largest block scale at 2^8).
__device__ __forceinline__ uint32_t ue4m3_pow2(int p) {
  if (p < -9) return 0u;
  if (p < -6) return 1u << (p + 9);
  return (uint32_t)(p + 7) << 3;
}

// 2^c as a float (c >= -149).
__device__ __forceinline__ float pow2f(int c) {
  return c >= -126 ? __uint_as_float((uint32_t)(c + 127) << 23) : __uint_as_float(1u << (c + 149));
}

// NVFP4 experts: one warp quantises token row t < 16 to MXFP4 (the same codes
// and E8M0 exponents as the standalone quantiser) and writes the scales for
// the UE4M3 MMA: each 32-block's 2^e twice (two 16-blocks) as 2^(e - c_t),
// c_t = (largest e of the row) - 8, and c_t to xshift[t]; the epilogue
// multiplies the row's products by 2^c_t.  A block more than 2^17 below the
// row's largest block scale falls under UE4M3's range and is dropped.  Rows
// t >= T get zero scale words.  Lane l takes blocks l, l+32, ... in batches
// of 4 with all their loads in flight; the exponents wait in e_s (H <= 8192).
__device__ void quant_row_nv(const DcArgs& a, int t, uint8_t* e_s) {
  const int lane = threadIdx.x & 31, nb = a.H / 32;
  if (t >= a.T) {
    for (int kb = lane; kb < a.H / 64; kb += 32) *reinterpret_cast<uint32_t*>(a.xs_mma + (size_t)kb * 512 + t * 16) = 0u;
    return;
  }
  const uint16_t* xr = a.x + (size_t)t * a.H;
  int emax = -127;
  for (int b0 = lane; b0 < nb; b0 += 4 * 32) {
    uint4 raw[16];  // 4 blocks: every load issued before any is used
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int b = b0 + 32 * (i >> 2);
      raw[i] = b < nb ? __ldg(reinterpret_cast<const uint4*>(xr + b * 32) + (i & 3)) : make_uint4(0, 0, 0, 0);
    }
    // compact loops: this runs once per launch, where instruction fetch is slow
#pragma unroll 1
    for (int j = 0; j < 4; ++j) {
      const int b = b0 + 32 * j;
      if (b >= nb) break;
      float amax = 0.0f;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        const uint4 w = raw[4 * j + q];
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(w.x)), fabsf(bf16_hi(w.x))), fmaxf(fabsf(bf16_lo(w.y)), fabsf(bf16_hi(w.y)))));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(w.z)), fabsf(bf16_hi(w.z))), fmaxf(fabsf(bf16_lo(w.w)), fabsf(bf16_hi(w.w)))));
      }
      const int ex = mx_scale_exp(amax);
      const float inv = pow2_neg(ex);
      uint32_t* dst = reinterpret_cast<uint32_t*>(a.xq + (size_t)t * (a.H / 2) + b * 16);
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        const uint4 w = raw[4 * j + q];
        const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
        uint32_t word = 0;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          word |= e2m1_rne(bf16_lo(w4[h]) * inv) << (8 * h);
          word |= e2m1_rne(bf16_hi(w4[h]) * inv) << (8 * h + 4);
        }
        dst[q] = word;
      }
      e_s[b] = (uint8_t)(ex + 127);
      emax = max(emax, ex);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) emax = max(emax, __shfl_xor_sync(FULL, emax, o));
  const int c = emax - 8;
  if (lane == 0) a.xshift[t] = c;
  __syncwarp();
  // bytes 2(b&1), 2(b&1)+1 of the word of row t in 64-element chunk b/2
  for (int b = lane; b < nb; b += 32) {
    const uint32_t u = ue4m3_pow2((int)e_s[b] - 127 - c);
    *reinterpret_cast<uint16_t*>(a.xs_mma + (size_t)(b / 2) * 512 + t * 16 + 2 * (b & 1)) = (uint16_t)(u | (u << 8));
  }
}

// Top-k of every token (one epilogue warp per token), then the stable sort
// of the T*k <= 128 assignments by expert (each assignment counts the ones
// that precede it) and the distinct-expert slots (runs of one expert in the
// sorted order, numbered with a ballot).  128 epilogue threads, et = 0..127.
// *failed is set (by some thread) when a logit row never arrived.
__device__ void build_routing(const DcArgs& a, DcRouting& R, int et, uint32_t epoch, int* failed) {
  const int T = a.T, k = a.k, kr = a.kr, n = T * k;
  const int w = et >> 5, lane = et & 31;
  for (int t = w; t < T; t += EPI_THREADS / 32) {
    float v[8];
    if (!wait_logit_row(a, t, epoch, v)) {
      if (lane == 0) *failed = 1;
      continue;
    }
    int sel[MAX_TOPK];
    float wt[MAX_TOPK];
    route_row(v, a.Er, kr, a.score, a.bias, sel, wt);
#pragma unroll
    for (int j = 0; j < MAX_TOPK; ++j)
      if (j == lane && j < kr) {
        R.ids[t * k + j] = sel[j];
        R.w[t * k + j] = wt[j];
      }
    if (lane == 0 && kr < k) {  // the shared expert folded into the table: expert Er, weight 1
      R.ids[t * k + kr] = a.Er;
      R.w[t * k + kr] = 1.0f;
    }
  }
  epi_sync();
  if (*failed) return;  // the same answer in every thread after the barrier
  if (et < n) {
    const int e = R.ids[et];
    int pos = 0;
    for (int b = 0; b < n; ++b) {
      const int eb = R.ids[b];
      pos += (eb < e) | ((eb == e) & (b < et));
    }
    R.inv[et] = pos;
    R.tok[pos] = et / k;
    R.sorted_e[pos] = e;
  }
  epi_sync();
  const bool start = et < n && (et == 0 || R.sorted_e[et] != R.sorted_e[et - 1]);
  const unsigned mask = __ballot_sync(FULL, start);
  if (lane == 0) R.wcount[w] = __popc(mask);
  epi_sync();
  int base = 0;
  for (int ww = 0; ww < w; ++ww) base += R.wcount[ww];
  if (start) {
    const int slot = base + __popc(mask & ((1u << lane) - 1u));
    R.slot_e[slot] = R.sorted_e[et];
    R.slot_beg[slot] = et;
  }
  if (et == 0) {
    int total = 0;
    for (int ww = 0; ww < EPI_THREADS / 32; ++ww) total += R.wcount[ww];
    R.n_slots = total;
    R.slot_beg[total] = n;
  }
  epi_sync();
}

// Halves of a stage that a unit uses: gate/up units one K chunk (two weight
// tiles, one activation tile), down units two K chunks (the second may be
// past the end of K).
__device__ __forceinline__ int stage_halves(const DcArgs& a, const Unit& U, int st) {
  if (U.kind == U_SDN) return 2 * st + 1 < a.I / 64 ? 2 : 1;
  if (U.kind == U_RDN) return 2 * st + 1 < a.I / 256 ? 2 : 1;
  return 2;
}

// Scale bytes per 128 rows and 256-element K chunk.
template <bool NV> __device__ __forceinline__ constexpr uint32_t sf_chunk() { return 512u * nblk<NV>(); }

// Bytes one stage of a unit brings in (the mbarrier transaction count).
template <bool NV>
__device__ __forceinline__ uint32_t stage_tx(const DcArgs& a, const Unit& U, int st) {
  const uint32_t h = stage_halves(a, U, st);
  switch (U.kind) {
    case U_SGU: return 2 * A_TILE + B_TILE;
    case U_RGU: return 2 * A_TILE + B_TILE + 3 * sf_chunk<NV>();
    case U_SDN: return h * (A_TILE + B_TILE);
    default: return h * (A_TILE + B_TILE + 2 * sf_chunk<NV>());
  }
}

// TMA / bulk copies of the weight tiles (and their scales) of stage st.
template <bool NV>
__device__ __forceinline__ void issue_weights(const DcArgs& a, const DcMaps& m, const Unit& U, int st, int e,
                                              uint8_t* sp, uint64_t* fb) {
  const int nbI = a.I / 128, nbH = a.H / 128;
  if (U.kind == U_SGU) {
    tc::tma_load_2d(sp + ST_A0, &m.w13s, st * 128, 128 * U.tile, fb);
    tc::tma_load_2d(sp + ST_A1, &m.w13s, st * 128, a.I + 128 * U.tile, fb);
  } else if (U.kind == U_RGU) {
    const int row = e * 2 * a.I + 128 * U.tile;
    const uint32_t sfc = sf_chunk<NV>();
    const size_t bpr = (size_t)a.H / 256 * (sfc / 512);  // scale blocks per 128-row tile
    const size_t rt = (size_t)e * (2 * nbI) + U.tile;    // gate row tile; the up tile is nbI further
    tc::tma_load_2d(sp + ST_A0, &m.w13r, st * 128, row, fb);
    tc::tma_load_2d(sp + ST_A1, &m.w13r, st * 128, row + a.I, fb);
    tc::bulk_load(sp + ST_SFA, a.w13s_mma + rt * bpr * 512 + (size_t)st * sfc, sfc, fb);
    tc::bulk_load(sp + ST_SFA + sfc, a.w13s_mma + (rt + nbI) * bpr * 512 + (size_t)st * sfc, sfc, fb);
  } else if (U.kind == U_SDN) {
    for (int h = 0; h < stage_halves(a, U, st); ++h)
      tc::tma_load_2d(sp + (h ? ST_A1 : ST_A0), &m.w2s, (2 * st + h) * 128, 128 * U.tile, fb);
  } else {
    const int halves = stage_halves(a, U, st);
    for (int h = 0; h < halves; ++h)
      tc::tma_load_2d(sp + (h ? ST_A1 : ST_A0), &m.w2r, (2 * st + h) * 128, e * a.H + 128 * U.tile, fb);
    const uint32_t sfc = sf_chunk<NV>();
    const size_t bpr = (size_t)a.I / 256 * (sfc / 512);
    tc::bulk_load(sp + ST_SFA, a.w2s_mma + ((size_t)e * nbH + U.tile) * bpr * 512 + (size_t)2 * st * sfc, halves * sfc, fb);
  }
}

// TMA / bulk copies of the activation tiles (and their scales) of stage st.
template <bool NV>
__device__ __forceinline__ void issue_acts(const DcArgs& a, const DcMaps& m, const Unit& U, int st, int beg,
                                           uint8_t* sp, uint64_t* fb) {
  if (U.kind == U_SGU) {
    tc::tma_load_2d(sp + ST_B0, &m.x, st * 128, 0, fb);
  } else if (U.kind == U_RGU) {
    tc::tma_load_2d(sp + ST_B0, &m.xq, st * 128, 0, fb);
    tc::bulk_load(sp + st_sfb<NV>(), a.xs_mma + (size_t)st * sf_chunk<NV>(), sf_chunk<NV>(), fb);
  } else if (U.kind == U_SDN) {
    for (int h = 0; h < stage_halves(a, U, st); ++h)
      tc::tma_load_2d(sp + (h ? ST_B1 : ST_B0), &m.hsh, (2 * st + h) * 128, 0, fb);
  } else {
    const int halves = stage_halves(a, U, st);
    for (int h = 0; h < halves; ++h)
      tc::tma_load_2d(sp + (h ? ST_B1 : ST_B0), &m.hq, (2 * st + h) * 128, beg, fb);
    const size_t bpr = (size_t)a.I / 256 * nblk<NV>();  // scale blocks of one slot
    tc::bulk_load(sp + st_sfb<NV>(), a.hs_mma + (size_t)U.slot * bpr * 512 + (size_t)2 * st * sf_chunk<NV>(),
                  halves * sf_chunk<NV>(), fb);
  }
}

// Row shift c of sorted h row p (NVFP4), final once every routed h tile is done.
__device__ __forceinline__ int h_row_shift(const DcArgs& a, int p);

// NVFP4: the UE4M3 scale blocks of slot s's h rows (sorted positions beg ..
// beg+cnt-1) for the down MMA, [I/64][512 B], from their E8M0 bytes and the
// row shift 2^c (c = the row's largest exponent - 8).  128 threads; thread
// et writes word et of every block (row et/4 when et % 4 == 0, else zero).
__device__ void convert_h_scales_nv(const DcArgs& a, int slot, int beg, int cnt, int et) {
  const int nb = a.I / 32, r = et >> 2;
  const bool real = (et & 3) == 0 && r < cnt;
  const int c = real ? h_row_shift(a, beg + r) : 0;
  const uint8_t* hsr = a.hsc + (size_t)(beg + (real ? r : 0)) * nb;
  uint32_t* dst = reinterpret_cast<uint32_t*>(a.hs_mma) + (size_t)slot * (a.I / 64) * 128 + et;
  for (int g = 0; g < a.I / 64; ++g) {
    uint32_t word = 0;
    if (real) {
      const uint32_t u0 = ue4m3_pow2((int)__ldcg(hsr + 2 * g) - 127 - c);
      const uint32_t u1 = ue4m3_pow2((int)__ldcg(hsr + 2 * g + 1) - 127 - c);
      word = u0 | (u0 << 8) | (u1 << 16) | (u1 << 24);
    }
    dst[(size_t)g * 128] = word;
  }
}

__device__ __forceinline__ int h_row_shift(const DcArgs& a, int p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(a.rowmax + p) : "memory");
  return (int)(uint32_t)v - 256 - 8;
}

// One FP4 MMA (M = 128, N = 16, K = 64, the kk-th of a 256-element chunk)
// with the chunk's A / B scale tiles at TMEM columns sfa / sfb: MXFP4 reads
// byte pair (kk & 1) of the 128-element group kk / 2, NVFP4 the whole word of
// 64-element chunk kk.
template <bool NV>
__device__ __forceinline__ void fp4_mma(uint32_t d, uint64_t ad, uint64_t bd, int kk, uint32_t sfa, uint32_t sfb,
                                        uint32_t accum) {
  if (NV) {
    tc::mma_nvf4(d, ad, bd, tc::idesc_nvf4(128, 16), sfa + 4 * kk, sfb + 4 * kk, accum);
  } else {
    const int grp = kk >> 1, id = (kk & 1) * 2;
    tc::mma_mxf4(d, ad, bd, tc::idesc_mxf4(128, 16, id, id), sfa + 4 * grp, sfb + 4 * grp, accum);
  }
}

// ------------------------------------------------------------------ kernel

template <bool NV>
__global__ void __launch_bounds__(DT, 1) k_decode_tc(const __grid_constant__ DcMaps maps, const DcArgs a) {
  constexpr uint32_t STAGE_BYTES = stage_bytes<NV>();
  constexpr uint32_t ST_SFB = st_sfb<NV>();
  constexpr int NB = nblk<NV>();
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[DSTAGES], empty[DSTAGES], acc_full[NACC], acc_empty[NACC], drain, routing_ready;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag, s_ok, s_last, s_fail;
  __shared__ uint32_t s_epoch;
  __shared__ DcRouting R;
  __shared__ float red_s[EPI_THREADS / 32][MAX_DECODE_T];
  __shared__ __align__(4) uint8_t s_hsb[MAX_DECODE_T * 4];
  __shared__ uint8_t s_qe[EPI_THREADS / 32][256];  // NVFP4 quantiser: a row's block exponents
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nbI = a.I / 128, nbH = a.H / 128;
  int* status = a.ctr + C_STATUS;

  if (threadIdx.x == 0) {
    for (int s = 0; s < DSTAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NACC; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], EPI_THREADS);
    }
    tc::mbar_init(&drain, 1);
    tc::mbar_init(&routing_ready, 1);
    tc::mbar_fence_init();
    abort_flag = 0;
    s_fail = 0;
    // Launch number: never 0 (the tag of zero-filled words), so after 2^32
    // launches it skips from 0xFFFFFFFF to 1.
    const uint32_t ep = (uint32_t)ld_acquire(a.ctr + C_DC_EPOCH) + 1u;
    s_epoch = ep == 0u ? 1u : ep;
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, tmem_cols<NV>());
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  auto fail = [&]() {
    atomicCAS(status, 0, (int)MOE_DEV_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const int never = 0;
      uint32_t stage = 0, phase = 0, issued = 0, last_parity = 0, gi = 0;
      // Stage gi may be issued once stage gi - depth has been consumed (which
      // also frees slot gi % DSTAGES: depth <= DSTAGES, consumption in order).
      auto claim = [&]() -> bool {
        if (gi < (uint32_t)a.depth) return true;
        const uint32_t j = gi - (uint32_t)a.depth;
        return tc::mbar_wait(&empty[j % DSTAGES], (j / DSTAGES) & 1, a.limit_ns, &abort_flag);
      };
      int n_slots = -1;
      bool hsh_ok = false, hr_ok = false;
      tc::prefetch_tensormap(&maps.w13r);
      tc::prefetch_tensormap(&maps.w2r);
      tc::prefetch_tensormap(&maps.xq);
      tc::prefetch_tensormap(&maps.hq);
      if (a.shared) {
        tc::prefetch_tensormap(&maps.w13s);
        tc::prefetch_tensormap(&maps.w2s);
        tc::prefetch_tensormap(&maps.x);
        tc::prefetch_tensormap(&maps.hsh);
      }
      for (int u = blockIdx.x;; u += a.G) {
        if (u >= a.n_sgu && n_slots < 0) {
          if (!tc::mbar_wait(&routing_ready, 0, a.limit_ns, &abort_flag)) { fail(); break; }
          n_slots = R.n_slots;
          // x was quantised by plain stores of other blocks
          if (!wait_at_least(a.ctr + C_DC_READY, a.G, status, a.limit_ns)) { fail(); break; }
          tc::fence_proxy_async_global();
        }
        if (u >= units_total(a, n_slots < 0 ? 0 : n_slots)) break;
        const Unit U = unit_at(a, n_slots < 0 ? 0 : n_slots, u);
        int e = 0, beg = 0;
        if (U.kind == U_RGU || U.kind == U_RDN) {
          e = R.slot_e[U.slot];
          beg = R.slot_beg[U.slot];
        }
        // Down units read h that other blocks write.  While it is not there
        // yet, the unit's weight tiles already go into the ring (up to its
        // depth); their h tiles follow once the dependency is met.
        int npre = 0;
        uint32_t pre_stage[DSTAGES];
        const bool dep_sdn = U.kind == U_SDN && !hsh_ok, dep_rdn = U.kind == U_RDN && !hr_ok;
        if (dep_sdn || dep_rdn) {
          int* cnt = a.ctr + (dep_sdn ? C_DC_HSH : C_DC_HR);
          const int target = dep_sdn ? nbI : (NV ? n_slots : n_slots * nbI);
          if (ld_acquire(cnt) < target) {
            npre = imin(U.st1 - U.st0, a.depth);
            bool ok = true;
            for (int j = 0; j < npre; ++j) {
              if (!claim()) { fail(); ok = false; break; }
              tc::mbar_expect_tx(&full[stage], stage_tx<NV>(a, U, U.st0 + j));
              issue_weights<NV>(a, maps, U, U.st0 + j, e, dsm + stage * STAGE_BYTES, &full[stage]);
              pre_stage[j] = stage;
              issued |= 1u << stage;
              last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
              ++gi;
              if (++stage == DSTAGES) {
                stage = 0;
                phase ^= 1;
              }
            }
            if (!ok) break;
            if (!wait_at_least(cnt, target, status, a.limit_ns)) { fail(); break; }
          }
          if (dep_sdn) hsh_ok = true; else hr_ok = true;
          tc::fence_proxy_async_global();
        }
        for (int j = 0; j < npre; ++j)
          issue_acts<NV>(a, maps, U, U.st0 + j, beg, dsm + pre_stage[j] * STAGE_BYTES, &full[pre_stage[j]]);
        bool ok = true;
        for (int st = U.st0 + npre; st < U.st1; ++st) {
          if (!claim()) { fail(); ok = false; break; }
          uint8_t* sp = dsm + stage * STAGE_BYTES;
          tc::mbar_expect_tx(&full[stage], stage_tx<NV>(a, U, st));
          issue_weights<NV>(a, maps, U, st, e, sp, &full[stage]);
          issue_acts<NV>(a, maps, U, st, beg, sp, &full[stage]);
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          ++gi;
          if (++stage == DSTAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      // copies still in flight must land before the block's shared memory goes away
      for (int s = 0; s < DSTAGES; ++s)
        if ((issued >> s & 1) && !tc::mbar_wait(&full[s], last_parity >> s & 1, a.limit_ns, &never)) fail();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const int never = 0;
      const uint32_t id_bf = tc::idesc_bf16(128, 16);
      uint32_t stage = 0, phase = 0;
      int n_slots = -1, i = 0;
      for (int u = blockIdx.x;; u += a.G, ++i) {
        if (u >= a.n_sgu && n_slots < 0) {
          if (!tc::mbar_wait(&routing_ready, 0, a.limit_ns, &abort_flag)) { fail(); break; }
          n_slots = R.n_slots;
        }
        if (u >= units_total(a, n_slots < 0 ? 0 : n_slots)) break;
        const Unit U = unit_at(a, n_slots < 0 ? 0 : n_slots, u);
        const int buf = i % NACC;
        const uint32_t use = (uint32_t)(i / NACC);
        if (!tc::mbar_wait(&acc_empty[buf], (use & 1) ^ 1, a.limit_ns, &abort_flag)) { fail(); break; }
        tc::fence_after_sync();
        const uint32_t acc = tmem + 32 * buf;
        bool ok = true;
        for (int st = U.st0; st < U.st1; ++st) {
          if (!tc::mbar_wait(&full[stage], phase, a.limit_ns, &abort_flag)) { fail(); ok = false; break; }
          tc::fence_after_sync();
          const uint32_t sa = tc::smem_u32(dsm + stage * STAGE_BYTES);
          const uint32_t tsf = tmem + TM_SF + 16 * NB * stage;
          const bool first = st == U.st0;
          if (U.kind == U_SGU) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = tc::desc_sw128(sa + ST_B0 + 32 * kk);
              const uint32_t accum = (first && kk == 0) ? 0u : 1u;
              tc::mma_bf16(acc, tc::desc_sw128(sa + ST_A0 + 32 * kk), bd, id_bf, accum);
              tc::mma_bf16(acc + 16, tc::desc_sw128(sa + ST_A1 + 32 * kk), bd, id_bf, accum);
            }
          } else if (U.kind == U_RGU) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              tc::sf_copy(tsf + 4 * b, tc::desc_sf(sa + ST_SFA + 512 * b));
              tc::sf_copy(tsf + 4 * NB + 4 * b, tc::desc_sf(sa + ST_SFA + 512 * (NB + b)));
              tc::sf_copy(tsf + 8 * NB + 4 * b, tc::desc_sf(sa + ST_SFB + 512 * b));
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = tc::desc_sw128(sa + ST_B0 + 32 * kk);
              const uint32_t accum = (first && kk == 0) ? 0u : 1u;
              fp4_mma<NV>(acc, tc::desc_sw128(sa + ST_A0 + 32 * kk), bd, kk, tsf, tsf + 8 * NB, accum);
              fp4_mma<NV>(acc + 16, tc::desc_sw128(sa + ST_A1 + 32 * kk), bd, kk, tsf + 4 * NB, tsf + 8 * NB, accum);
            }
          } else if (U.kind == U_SDN) {
            const int halves = stage_halves(a, U, st);
            for (int h = 0; h < halves; ++h) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t accum = (first && h == 0 && kk == 0) ? 0u : 1u;
                tc::mma_bf16(acc, tc::desc_sw128(sa + (h ? ST_A1 : ST_A0) + 32 * kk),
                             tc::desc_sw128(sa + (h ? ST_B1 : ST_B0) + 32 * kk), id_bf, accum);
              }
            }
          } else {
            const int halves = stage_halves(a, U, st);
            for (int h = 0; h < halves; ++h)
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                tc::sf_copy(tsf + 4 * NB * h + 4 * b, tc::desc_sf(sa + ST_SFA + 512 * (NB * h + b)));
                tc::sf_copy(tsf + 4 * NB * (2 + h) + 4 * b, tc::desc_sf(sa + ST_SFB + 512 * (NB * h + b)));
              }
            for (int h = 0; h < halves; ++h) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t accum = (first && h == 0 && kk == 0) ? 0u : 1u;
                fp4_mma<NV>(acc, tc::desc_sw128(sa + (h ? ST_A1 : ST_A0) + 32 * kk),
                            tc::desc_sw128(sa + (h ? ST_B1 : ST_B0) + 32 * kk), kk, tsf + 4 * NB * h,
                            tsf + 4 * NB * (2 + h), accum);
              }
            }
          }
          tc::mma_commit(&empty[stage]);
          if (++stage == DSTAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(&acc_full[buf]);
      }
      // every MMA issued must finish before TMEM is released
      tc::mma_commit(&drain);
      if (!tc::mbar_wait(&drain, 0, a.limit_ns, &never)) fail();
    }
  } else {
    // -------------------------------------------------- epilogue warps
    const int et = threadIdx.x - 64;
    const int q = warp & 3;                 // TMEM lane quadrant this warp may read
    const int m = q * 32 + lane;            // weight row within the 128-row tile
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    const int T = a.T, H = a.H, I = a.I, k = a.k, n = T * k;

    const uint32_t epoch = s_epoch;
    for (int e = blockIdx.x; e < a.Er; e += a.G) router_row(a, e, et, red_s, epoch);
    // the router rows go to the first E blocks, the quantisation to the last ones
    if (NV) {
      const int t = (a.G - 1 - blockIdx.x) * (EPI_THREADS / 32) + (et >> 5);
      if (t < MAX_DECODE_T) quant_row_nv(a, t, s_qe[et >> 5]);
    } else {
      const int nqb = MAX_DECODE_T * (H / 32);
      for (int i = (a.G - 1 - blockIdx.x) * EPI_THREADS + et; i < nqb; i += a.G * EPI_THREADS) quant_block(a, i);
    }
    tc::fence_proxy_async_global();
    epi_sync();  // orders every thread's stores before thread 0's release
    if (et == 0) red_release_add(a.ctr + C_DC_READY, 1);
    build_routing(a, R, et, epoch, &s_fail);
    if (s_fail) {
      if (et == 0) fail();
    } else {
      if (et == 0) tc::mbar_arrive(&routing_ready);
      if (blockIdx.x == 0 && et < n && et % a.k < a.kr) {  // the router's top-k, [T][kr]
        const int o = et / a.k * a.kr + et % a.k;
        if (a.ids_out) a.ids_out[o] = R.ids[et];
        if (a.w_out) a.w_out[o] = R.w[et];
      }
      const int n_slots = R.n_slots;
      const int total = units_total(a, n_slots);
      const int dn_total = nbH * ((a.shared ? a.s_sdn : 0) + n_slots);  // down parts over all tiles
      int i = 0;
      for (int u = blockIdx.x; u < total; u += a.G, ++i) {
        const Unit U = unit_at(a, n_slots, u);
        const int buf = i % NACC;
        const uint32_t use = (uint32_t)(i / NACC);
        if (et == 0) {
          s_ok = tc::mbar_wait(&acc_full[buf], use & 1, a.limit_ns, &abort_flag);
          if (!s_ok) fail();
        }
        epi_sync();
        if (!s_ok) break;
        tc::fence_after_sync();
        float v[32];
        tc::tmem_ld32(trow + 32 * buf, v);
        tc::fence_before_sync();
        tc::mbar_arrive(&acc_empty[buf]);

        int beg = 0, cnt = 0;
        if (U.kind == U_RGU || U.kind == U_RDN) {
          beg = R.slot_beg[U.slot];
          cnt = R.slot_beg[U.slot + 1] - beg;
        }
        int ticket, target;
        if (U.kind == U_SGU) {
          float* dst = a.gu_sh + (size_t)U.part * T * 2 * I + 128 * U.tile + m;
#pragma unroll
          for (int t = 0; t < MAX_DECODE_T; ++t)
            if (t < T) {
              dst[(size_t)t * 2 * I] = v[t];
              dst[(size_t)t * 2 * I + I] = v[16 + t];
            }
          ticket = U.tile;
          target = a.s_sgu;
        } else if (U.kind == U_RGU) {
          // B held every token row: slot row c is the column of its token
          // (NVFP4: times the expert's gate / up tensor scale and 2^c_t)
          float* dst = a.gu_r + ((size_t)U.part * n + beg) * 2 * I + 128 * U.tile + m;
          float sg = 1.0f, su = 1.0f;
          if (NV) {
            const int e = R.slot_e[U.slot];
            sg = __ldg(a.tscale + 3 * e);
            su = __ldg(a.tscale + 3 * e + 1);
          }
          for (int c = 0; c < cnt; ++c) {
            const int t = R.tok[beg + c];
            const float f = NV ? pow2f(__ldcg(a.xshift + t)) : 1.0f;
            dst[(size_t)c * 2 * I] = pick16(v, 0, t) * (sg * f);
            dst[(size_t)c * 2 * I + I] = pick16(v, 16, t) * (su * f);
          }
          ticket = nbI + U.slot * nbI + U.tile;
          target = a.s_rgu;
        } else if (U.kind == U_SDN) {
          float* dst = a.ys + (size_t)U.part * T * H + 128 * U.tile + m;
#pragma unroll
          for (int t = 0; t < MAX_DECODE_T; ++t)
            if (t < T) dst[(size_t)t * H] = v[t];
          ticket = -1;
          target = 0;
        } else {
          // B held the slot's sorted rows: column c is sorted position beg + c
          // (NVFP4: times the expert's down tensor scale and 2^c of the h row)
          float* dst = a.y_assign + (size_t)beg * H + 128 * U.tile + m;
          const float sd = NV ? __ldg(a.tscale + 3 * R.slot_e[U.slot] + 2) : 1.0f;
#pragma unroll
          for (int c = 0; c < MAX_DECODE_T; ++c)
            if (c < cnt) dst[(size_t)c * H] = NV ? v[c] * (sd * pow2f(h_row_shift(a, beg + c))) : v[c];
          ticket = -1;
          target = 0;
        }
        if (ticket < 0) {
          // a down part: counted without waiting; the combine runs after the unit list
          epi_sync();
          if (et == 0) red_release_add(a.ctr + C_DC_DN, 1);
          continue;
        }
        // split-K arrival: the block that brings the last part finishes the
        // tile (a tile of one part needs no ticket: its own stores precede)
        if (target > 1) {
          epi_sync();
          if (et == 0) {
            __threadfence();
            const int old = atomicAdd(a.tickets + ticket, 1);
            s_last = old == target - 1;
            if (s_last) {
              a.tickets[ticket] = 0;
              __threadfence();
            }
          }
          epi_sync();
          if (!s_last) continue;
        }
        if (U.kind == U_SGU) {
          const float* src = a.gu_sh + 128 * U.tile + m;
          const size_t stride = (size_t)T * 2 * I;
          for (int t0 = 0; t0 < T; t0 += 2) {  // two tokens' loads in flight together
            float g[2], up[2];
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
              const int t = imin(t0 + tt, T - 1);
              g[tt] = sum_parts(src + (size_t)t * 2 * I, stride, a.s_sgu);
              up[tt] = sum_parts(src + (size_t)t * 2 * I + I, stride, a.s_sgu);
            }
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
              if (t0 + tt < T) a.h_shared[(size_t)(t0 + tt) * I + 128 * U.tile + m] = f32_to_bf16_rn(silu(g[tt]) * up[tt]);
          }
          tc::fence_proxy_async_global();
          epi_sync();
          if (et == 0) red_release_add(a.ctr + C_DC_HSH, 1);
        } else if (U.kind == U_RGU) {
          // h = SiLU(G) U requantised to MXFP4: warp q holds one 32-column block
          const float* src = a.gu_r + (size_t)beg * 2 * I + 128 * U.tile + m;
          const size_t stride = (size_t)n * 2 * I;
          for (int c = 0; c < cnt; ++c) {
            const float g = sum_parts(src + (size_t)c * 2 * I, stride, a.s_rgu);
            const float up = sum_parts(src + (size_t)c * 2 * I + I, stride, a.s_rgu);
            const float h = silu(g) * up;
            const int ex = mx_scale_exp(warp_max(fabsf(h)));
            uint32_t wv = e2m1_rne(h * pow2_neg(ex)) << (4 * (lane & 7));
            wv |= __shfl_xor_sync(FULL, wv, 1);
            wv |= __shfl_xor_sync(FULL, wv, 2);
            wv |= __shfl_xor_sync(FULL, wv, 4);
            if ((lane & 7) == 0)
              *reinterpret_cast<uint32_t*>(a.hq + (size_t)(beg + c) * (I / 2) + 64 * U.tile + 16 * q + 4 * (lane >> 3)) = wv;
            if (lane == 0) {
              if (NV) {
                // E8M0 byte of the block and the row's largest exponent so far
                a.hsc[(size_t)(beg + c) * (I / 32) + 4 * U.tile + q] = (uint8_t)(ex + 127);
                atomicMax(a.rowmax + beg + c, ((unsigned long long)epoch << 32) | (unsigned long long)(ex + 256));
              } else {
                s_hsb[c * 4 + q] = (uint8_t)(ex + 127);
              }
            }
          }
          epi_sync();
          if (!NV) {
            // the slot's scale block for this 128-column group: word 4c holds row c
            const uint32_t word =
                ((et & 3) == 0 && (et >> 2) < cnt) ? reinterpret_cast<const uint32_t*>(s_hsb)[et >> 2] : 0u;
            reinterpret_cast<uint32_t*>(a.hs_mma)[((size_t)U.slot * nbI + U.tile) * 128 + et] = word;
            tc::fence_proxy_async_global();
            epi_sync();
            if (et == 0) red_release_add(a.ctr + C_DC_HR, 1);
          } else {
            // NVFP4: the slot's last finished tile knows every row's largest
            // exponent and writes the slot's UE4M3 scale blocks for the down MMA
            if (et == 0) {
              __threadfence();
              const int old = atomicAdd(a.tickets + nbI * (1 + a.nslot_max) + nbH + U.slot, 1);
              s_last = old == nbI - 1;
              if (s_last) {
                a.tickets[nbI * (1 + a.nslot_max) + nbH + U.slot] = 0;
                __threadfence();
              }
            }
            epi_sync();
            if (s_last) {
              convert_h_scales_nv(a, U.slot, beg, cnt, et);
              tc::fence_proxy_async_global();
              epi_sync();
              if (et == 0) red_release_add(a.ctr + C_DC_HR, 1);
            }
          }
        }
      }
      // out = BF16(ys + sum_j w_j y_j), summed in a fixed order, once every
      // down part is stored.  Items (128 columns of H x 4 tokens) are spread
      // over all blocks, so a block's items cost one load round trip each
      // (on 32 blocks a 16-token step took four in a row).
      const int n_items = nbH * ((T + 3) / 4);
      if ((int)blockIdx.x < n_items) {
        if (et == 0) {
          s_ok = wait_at_least(a.ctr + C_DC_DN, dn_total, status, a.limit_ns);
          if (!s_ok) fail();
        }
        epi_sync();
      }
      for (int item = blockIdx.x; item < n_items && s_ok; item += a.G) {
        const int col = 128 * (item % nbH) + m;
        {
          const int t0 = 4 * (item / nbH);  // four tokens' loads in flight together
          float y[4][MAX_TOPK], ysh[4];
#pragma unroll
          for (int tt = 0; tt < 4; ++tt) {
            const int t = imin(t0 + tt, T - 1);
#pragma unroll
            for (int j = 0; j < MAX_TOPK; ++j)
              y[tt][j] = j < k ? __ldcg(a.y_assign + (size_t)R.inv[t * k + j] * H + col) : 0.0f;
            ysh[tt] = a.shared ? sum_parts<4>(a.ys + (size_t)t * H + col, (size_t)T * H, a.s_sdn) : 0.0f;
          }
#pragma unroll
          for (int tt = 0; tt < 4; ++tt) {
            const int t = t0 + tt;
            if (t < T) {
              float acc = ysh[tt];
#pragma unroll
              for (int j = 0; j < MAX_TOPK; ++j)
                if (j < k) acc = fmaf(R.w[t * k + j], y[tt][j], acc);
              a.out[(size_t)t * H + col] = f32_to_bf16_rn(acc);
            }
          }
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, tmem_cols<NV>());
  }
  // The last block out resets the launch's counters for the next call and
  // clears the NVFP4 row exponents (atomicMax words: a word tagged with an
  // older launch number than the next launch's would otherwise win it).
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.ctr + C_DC_EXIT, 1) == a.G - 1;
  }
  __syncthreads();
  if (s_last) {
    if (a.nv)
      for (int i = threadIdx.x; i < MAXN; i += blockDim.x) a.rowmax[i] = 0ull;
    if (threadIdx.x == 0) {
      a.ctr[C_DC_READY] = 0;
      a.ctr[C_DC_HSH] = 0;
      a.ctr[C_DC_HR] = 0;
      a.ctr[C_DC_EXIT] = 0;
      a.ctr[C_DC_DN] = 0;
      a.ctr[C_DC_EPOCH] = (int)s_epoch;
    }
    __threadfence();
  }
}

}  // namespace

bool fused_decode_tc_supported(const Shape& sh, const ExpertsDev& ex) {
  return ex.w13s_mma && ex.w2s_mma && sh.T >= 1 && sh.T <= MAX_DECODE_T && sh.H % 256 == 0 && sh.I % 256 == 0 &&
         (!ex.nv || sh.H <= 8192);  // the NVFP4 quantiser keeps a row's 32-block exponents in shared memory
}

cudaError_t launch_fused_decode_tc(const Shape& sh, const ExpertsDev& ex, const SharedDev& shd, const float* wr,
                                   const float* bias, const uint16_t* x, uint16_t* out, int* ids_out, float* w_out,
                                   void* ws, uint64_t wait_limit_ns, cudaStream_t s, int fold, int score) {
  if (sh.T == 0) return cudaSuccess;
  if (!fused_decode_tc_supported(sh, ex)) return cudaErrorInvalidValue;
  const int T = sh.T, H = sh.H, I = sh.I, E = sh.E, k = sh.k, n = T * k;
  const WsLayout L = ws_layout(T, H, I, E, k);
  uint8_t* base = static_cast<uint8_t*>(ws);
  const bool nv = ex.nv != 0;
  // One block per SM: the stage ring leaves no room for a second block,
  // whose TMA stream would share the SM's copy engine.
  const size_t smem = (size_t)DSTAGES * (nv ? stage_bytes<true>() : stage_bytes<false>()) + 1024;
  static_assert(DSTAGES * stage_bytes<false>() + 1024 > 114 * 1024, "the ring must keep one block per SM");
  auto kern = nv ? k_decode_tc<true> : k_decode_tc<false>;
  cudaError_t err = cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, DT, smem)) != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // one block per SM: every block holds a 200 KB stage ring and a TMEM allocation
  const int G = imin(sm_count(), DC_MAX_GRID);
  const bool shared = shd.w13 != nullptr;
  const DcSplits sp = dc_splits(T, H, I, E, k, G);

  DcArgs a{};
  a.T = T;
  a.H = H;
  a.I = I;
  a.E = E;
  a.k = k;
  a.Er = E - fold;
  a.kr = k - fold;
  a.G = G;
  a.s_sgu = sp.sgu;
  a.s_rgu = sp.rgu;
  a.s_sdn = sp.sdn;
  a.n_sgu = shared ? (I / 128) * sp.sgu : 0;
  a.n_sdn = shared ? (H / 128) * sp.sdn : 0;
  a.nslot_max = imin(n, E);
  a.shared = shared ? 1 : 0;
  a.nv = ex.nv;
  a.score = score;
  a.w13s_mma = ex.w13s_mma;
  a.w2s_mma = ex.w2s_mma;
  a.tscale = ex.tscale;
  a.wr = wr;
  a.bias = bias;
  a.x = x;
  a.out = out;
  a.ids_out = ids_out;
  a.w_out = w_out;
  a.ctr = reinterpret_cast<int*>(base + L.counters);
  a.tickets = reinterpret_cast<int*>(base + L.dc_tickets);
  a.logit64 = reinterpret_cast<unsigned long long*>(base + L.dc_logit64);
  a.xq = base + L.xq;
  a.xs_mma = base + L.dc_xs;
  a.xshift = reinterpret_cast<int*>(base + L.dc_xshift);
  a.hsc = base + L.dc_hsc;
  a.depth = a.nslot_max >= 16 ? 4 : 2;
  a.rowmax = reinterpret_cast<unsigned long long*>(base + L.dc_rowmax);
  a.hq = base + L.hq;
  a.hs_mma = base + L.dc_hs;
  a.h_shared = reinterpret_cast<uint16_t*>(base + L.h_shared);
  a.gu_sh = reinterpret_cast<float*>(base + L.dc_gu_sh);
  a.gu_r = reinterpret_cast<float*>(base + L.dc_gu_r);
  a.ys = reinterpret_cast<float*>(base + L.dc_ys);
  a.y_assign = reinterpret_cast<float*>(base + L.y_assign);
  a.limit_ns = wait_limit_ns;

  DcMaps m;
  memset(&m, 0, sizeof(m));
  if ((err = make_map(&m.w13r, ex.w13, (uint64_t)E * 2 * I, H / 2)) != cudaSuccess) return err;
  if ((err = make_map(&m.w2r, ex.w2, (uint64_t)E * H, I / 2)) != cudaSuccess) return err;
  if ((err = make_map(&m.xq, a.xq, T, H / 2, 16)) != cudaSuccess) return err;
  if ((err = make_map(&m.hq, a.hq, n, I / 2, 16)) != cudaSuccess) return err;
  if (shared) {
    if ((err = make_map(&m.w13s, shd.w13, (uint64_t)2 * I, (uint64_t)2 * H)) != cudaSuccess) return err;
    if ((err = make_map(&m.w2s, shd.w2, H, (uint64_t)2 * I)) != cudaSuccess) return err;
    if ((err = make_map(&m.x, x, T, (uint64_t)2 * H, 16)) != cudaSuccess) return err;
    if ((err = make_map(&m.hsh, a.h_shared, T, (uint64_t)2 * I, 16)) != cudaSuccess) return err;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(DT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // blocks wait on one another: all must be resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return count_launch(), cudaLaunchKernelEx(&cfg, kern, m, a);
}

}  // namespace moefp4
