// Tensor-core (tcgen05) GEMMs of the batched path: the routed expert
// gate/up and down projections on block-scaled FP4 (kind::mxf4, E8M0 scales
// per 32) and the BF16 shared expert (kind::f16), with the SwiGLU + MXFP4
// requantise epilogue fused into the gate/up GEMM (AMD technical article
// "MiniMax-M3.1 on AMD Instinct GPUs", section "What we Optimized": the
// MXFP4 fused MoE; model card "amd/MiniMax-M3.1-Flash-Quark-MXFP4", section
// "Model Overview": MXFP4 weights and activations).
//
// One persistent kernel per GEMM, warp-specialised (576 threads):
//   warp 0      TMA producer: 2D swizzled tiles of A and B and 1D bulk copies
//               of their scale blocks into a 4-stage shared-memory ring;
//   warp 1      MMA issuer: copies the stage's scale blocks into TMEM with
//               tcgen05.cp and issues 4 MMAs per 256-element (FP4) / 64-element
//               (BF16) K stage into a 128 x 256 FP32 accumulator in TMEM;
//               tcgen05.commit frees the stage and signals the epilogue;
//   warps 2-17  epilogue: four warps per TMEM lane quadrant, each taking one
//               quarter of the tile's columns; a warp copies its columns from
//               TMEM to registers and frees the accumulator before the
//               SwiGLU / requantise arithmetic and the stores, so the next
//               tile's MMAs overlap them.
// Tiles are 128 rows of A (tokens) x 256 rows of B (weight rows); for the
// gate/up GEMMs the 256 B rows are 128 gate rows and the 128 matching up rows,
// so each thread holds G and U of the same 128 columns.
//
// Grouped (routed) GEMMs run on a per-expert padded row order: expert e's
// assignments occupy rows [poff[e], poff[e] + count[e]) of a buffer whose
// expert blocks start at multiples of 128, so a tile never spans experts.
// Dense (shared-expert) GEMMs may split K into parts written to separate FP32
// outputs that small kernels sum in order (few tokens: too few tiles for the
// SMs).  With a few tokens per expert the routed GEMMs swap operands instead
// (k_tc_gemm_wa below: weights as A, 64-row token windows as B).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moefp4 {

namespace {

constexpr int BM = 128;           // A rows per tile
constexpr int BN = 256;           // B rows per tile (accumulator columns)
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 16;
constexpr int TC_THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t A_BYTES = BM * 128;       // 16 KB: 128 rows x 128 B
constexpr uint32_t B_BYTES = BN * 128;       // 32 KB
constexpr uint32_t SFA_BYTES = 2 * 512;      // two K groups of 128 elements
constexpr uint32_t SFB_BYTES = 2 * 2 * 512;  // two 128-row B blocks x two K groups
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_TMEM_BASE = 256;       // scale slots after the 256 accumulator columns

enum Kind { KIND_FP4 = 0, KIND_BF16 = 1, KIND_FP8 = 2 };
enum Epi { EPI_SWIGLU_MX = 0, EPI_STORE_F32 = 1, EPI_SWIGLU_BF16 = 2, EPI_SWIGLU_MX8 = 3, EPI_COMBINE_RED = 4 };

// out[0..1] += {a, b}: one vector FP32 reduction at the L2 (8-byte aligned).
__device__ __forceinline__ void red_add_f32x2(float* out, float a, float b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(out), "f"(a), "f"(b) : "memory");
}

// Shared-memory stride of one stage (FP8 stages keep the FP4 layout and fill
// half of each scale slot: one K group of 128 per stage).
__host__ __device__ constexpr uint32_t stage_bytes(int kind) {
  return kind == KIND_BF16 ? A_BYTES + B_BYTES : A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
}
// Bytes a stage's copies deliver (the mbarrier transaction count).
__host__ __device__ constexpr uint32_t stage_tx(int kind) {
  return kind == KIND_FP8 ? A_BYTES + B_BYTES + 512 + 1024 : stage_bytes(kind);
}

}  // namespace

// One 128-row tile of A: which expert, its first row in the padded order and
// in the sorted-assignment order, and how many of its rows are real.
struct MTile {
  int e;
  int prow0;
  int srow0;
  int rows;
};

// --------------------------------------------------------------- tile list

// One block: padded expert offsets and the list of row windows (tiles of
// `win` = 128 or 64 rows; each expert's rows are rounded up to `win`).
__global__ void __launch_bounds__(256) k_build_mtiles(const int* __restrict__ offsets, int E, int win,
                                                      int* __restrict__ poff, MTile* __restrict__ tiles,
                                                      int* __restrict__ num_tiles) {
  __shared__ int s_poff[MAX_E + 1];
  __shared__ int s_pad[MAX_E];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {  // the offsets are read in parallel
    const int cnt = offsets[e + 1] - offsets[e];
    s_pad[e] = (cnt + win - 1) / win * win;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int p = 0;
    for (int e = 0; e < E; ++e) {
      s_poff[e] = p;
      p += s_pad[e];
    }
    s_poff[E] = p;
    *num_tiles = p / win;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) poff[e] = s_poff[e];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int cnt = offsets[e + 1] - offsets[e];
    for (int m = 0; m * win < cnt; ++m) {
      MTile t;
      t.e = e;
      t.prow0 = s_poff[e] + m * win;
      t.srow0 = offsets[e] + m * win;
      t.rows = min(win, cnt - m * win);
      tiles[t.prow0 / win] = t;
    }
  }
}

// One block per GR consecutive padded rows (one window: GR divides `win`):
// copy the MXFP4 activation row of each row's assignment there (zeros for
// padding rows) and scatter its scale bytes into the MMA scale layout.  The
// GR rows' index and data loads are issued together.  Scale layout of a
// matrix of windows of `win` rows and K elements: block (window, K/128 group)
// of 512 bytes, word (i, j) at byte 16 i + 4 j holding the 4 scale bytes of
// window row 32 j + i (with 64-row windows words j = 2, 3 are unused).  With
// rows16 set, rows past the window's real rows rounded up to 16 are skipped
// (nothing reads them).
constexpr int GR = 4;
__global__ void __launch_bounds__(128) k_gather_mx_rows(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                                        int K, int k_top, const int* __restrict__ perm,
                                                        const MTile* __restrict__ tiles, const int* __restrict__ num_tiles,
                                                        int win, int rows16, uint8_t* __restrict__ q_out,
                                                        uint32_t* __restrict__ sf_out, int n_assign,
                                                        int* __restrict__ status) {
  const int r0 = blockIdx.x * GR;
  if (r0 >= *num_tiles * win) return;
  const MTile t = tiles[r0 / win];
  const int lim = rows16 ? ((t.rows + 15) & ~15) : win;  // rows of the window that are written
  int src[GR];
#pragma unroll
  for (int i = 0; i < GR; ++i) {
    const int m = r0 % win + i;
    const int a = m < t.rows ? perm[t.srow0 + m] : -1;
    if (m < t.rows && (a < 0 || a >= n_assign)) report_bad_index(status);
    src[i] = (a >= 0 && a < n_assign) ? a / k_top : -1;  // out-of-range assignments read as zeros
  }
  const int cpr = K / 32;  // 16-byte chunks per row
  for (int c = threadIdx.x; c < cpr; c += blockDim.x) {
    uint4 v[GR];
#pragma unroll
    for (int i = 0; i < GR; ++i)
      v[i] = src[i] >= 0 ? __ldg(reinterpret_cast<const uint4*>(q + (size_t)src[i] * (K / 2)) + c)
                         : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < GR; ++i)
      if (r0 % win + i < lim) reinterpret_cast<uint4*>(q_out + (size_t)(r0 + i) * (K / 2))[c] = v[i];
  }
  const int groups = K / 128;
  for (int x = threadIdx.x; x < GR * groups; x += blockDim.x) {
    const int i = x / groups, g = x % groups;
    const int m = r0 % win + i;
    if (m >= lim) continue;
    const uint32_t w = src[i] >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(s + (size_t)src[i] * (K / 32)) + g) : 0u;
    sf_out[((size_t)((r0 + i) / win) * groups + g) * 128 + (m % 32) * 4 + m / 32] = w;
  }
}

// Re-lays canonical scale bytes [E][R][K/32] into the MMA scale layout
// [E][R/128][K/128][512 B].  One thread per 4-byte word.
__global__ void __launch_bounds__(256) k_relayout_weight_sf(const uint8_t* __restrict__ s, int E, int R, int K,
                                                            uint32_t* __restrict__ out) {
  const size_t words = (size_t)E * R * (K / 128);
  const size_t w = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= words) return;
  const int groups = K / 128;
  const size_t row = w / groups;  // global row (e * R + r)
  const int g = (int)(w % groups);
  const int m = (int)(row % BM);
  const size_t tile = row / BM;   // (e * R + r) / 128: R is a multiple of 128
  const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(s + row * (K / 32)) + g);
  out[(tile * groups + g) * 128 + (m % 32) * 4 + (m / 32)] = v;
}

cudaError_t launch_relayout_weight_sf(const uint8_t* s, int E, int R, int K, uint8_t* out, cudaStream_t st) {
  const size_t words = (size_t)E * R * (K / 128);
  if (words == 0) return cudaSuccess;
  count_launch(), k_relayout_weight_sf<<<(unsigned)((words + 255) / 256), 256, 0, st>>>(s, E, R, K, reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError();
}

// ------------------------------------------------------------------ GEMM

namespace {

struct GemmArgs {
  int K;                   // reduction length in elements
  int n_tiles;             // B tiles per A tile
  const int* num_mt;       // grouped: device count of A tiles
  int num_mt_dense;        // dense: count of A tiles
  int rows_dense;          // dense: rows of A
  const MTile* mt;         // grouped: A tiles
  int b_rows_per_expert;   // grouped: rows of B per expert (0 for dense)
  int b_up_off;            // gate/up GEMMs: row offset of the up block (I)
  const uint8_t* sfa;      // FP4: A scales, MMA layout
  const uint8_t* sfb;      // FP4: B scales, MMA layout [E][R/128][K/128][512]
  int sfb_rtiles;          // FP4: R/128 of B per expert
  // epilogue outputs
  uint8_t* hq;             // EPI_SWIGLU_MX: codes [padded rows][I/2]
  uint32_t* hs;            // EPI_SWIGLU_MX: scales, MMA layout over I
  int h_cols;              // I (SwiGLU epilogues)
  uint16_t* h_bf16;        // EPI_SWIGLU_BF16: [rows][I]
  float* out;              // EPI_STORE_F32: [rows][ldo] (split-K: part p at out + p * part_stride)
  int ldo;
  int ksplit;              // dense: K parts per output tile (0 or 1: none)
  size_t part_stride;
  // EPI_COMBINE_RED: out[token][col] += topk_w[a] * y for sorted row p with
  // assignment a = perm[p], token a / k_top (out is FP32 [T][ldo])
  const int* perm;
  const float* topk_w;
  int k_top;
  int n_major;             // tiles ordered B tile first (every A tile of one output column slice in turn)
  // EPI_STORE_F32 (one K part) / EPI_COMBINE_RED: out laid out by 256-column
  // slices, [ldo / 256][slice_rows][256], when slice_rows > 0
  int slice_rows;
  int* status;
  uint64_t limit_ns;
};

__device__ __forceinline__ int ksplit_of(const GemmArgs& g) { return g.ksplit > 1 ? g.ksplit : 1; }

// A tile / B tile of work item t (num_mt A tiles).
__device__ __forceinline__ int mti_of(const GemmArgs& g, int t, int num_mt) {
  t /= ksplit_of(g);
  return g.n_major ? t % num_mt : t / g.n_tiles;
}
__device__ __forceinline__ int nt_of(const GemmArgs& g, int t, int num_mt) {
  t /= ksplit_of(g);
  return g.n_major ? t / num_mt : t % g.n_tiles;
}

// Tile t: A tile mti, B tile nt and K part kp (split-K dense GEMMs).
// A grouped caller may pass the tile's MTile, loaded ahead (pre).
__device__ __forceinline__ void tile_coords(const GemmArgs& g, bool grouped, int t, int num_mt, int& a_row, int& e,
                                            int& rows, int& srow0, int& nt, int& mti, int& kp,
                                            const MTile* pre = nullptr) {
  kp = t % ksplit_of(g);
  mti = mti_of(g, t, num_mt);
  nt = nt_of(g, t, num_mt);
  if (grouped) {
    const MTile m = pre ? *pre : g.mt[mti];
    a_row = m.prow0;
    e = m.e;
    rows = m.rows;
    srow0 = m.srow0;
  } else {
    a_row = mti * BM;
    e = 0;
    rows = min(BM, g.rows_dense - a_row);
    srow0 = a_row;
  }
}

template <int KIND, int EPI, bool GROUPED>
__global__ void __launch_bounds__(TC_THREADS, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB, GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[STAGES], empty[STAGES], acc_full, acc_empty, drain;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  constexpr uint32_t SB = stage_bytes(KIND);
  constexpr bool SWIGLU = EPI == EPI_SWIGLU_MX || EPI == EPI_SWIGLU_BF16 || EPI == EPI_SWIGLU_MX8;
  static_assert(EPI != EPI_COMBINE_RED || GROUPED, "the combine epilogue needs the routed tile list");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(&acc_full, 1);
    tc::mbar_init(&acc_empty, 32 * EPI_WARPS);
    tc::mbar_init(&drain, 1);
    tc::mbar_fence_init();
    abort_flag = 0;
    tc::prefetch_tensormap(&mapA);
    tc::prefetch_tensormap(&mapB);
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const int num_mt = GROUPED ? *g.num_mt : g.num_mt_dense;
  const int total = num_mt * g.n_tiles * ksplit_of(g);
  const int nks = g.K / (KIND == KIND_FP4 ? 256 : KIND == KIND_FP8 ? 128 : 64);
  const int kgroups = g.K / 128;  // FP4 scale groups per row

  auto fail = [&]() {
    atomicCAS(g.status, 0, (int)MOE_DEV_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };

  if (warp == 0 && lane == 0) {
    // ---------------- producer
    uint32_t stage = 0, phase = 0, issued = 0, last_parity = 0;
    // grouped: each tile's MTile is loaded a tile ahead, off the stream's critical path
    auto mt_of = [&](int t) { return GROUPED && t < total ? g.mt[mti_of(g, t, num_mt)] : MTile{}; };
    MTile mn = mt_of(blockIdx.x);
    for (int t = blockIdx.x; t < total && !abort_flag; t += gridDim.x) {
      int a_row, e, rows, srow0, nt, mti, kp;
      const MTile m = mn;
      tile_coords(g, GROUPED, t, num_mt, a_row, e, rows, srow0, nt, mti, kp, &m);
      mn = mt_of(t + gridDim.x);
      const int b_base = e * g.b_rows_per_expert;
      const int b0 = SWIGLU ? b_base + nt * (BN / 2) : b_base + nt * BN;
      const int b1 = SWIGLU ? b0 + g.b_up_off : b0 + BN / 2;
      const int ks1 = (kp + 1) * nks / ksplit_of(g);
      for (int ks = kp * nks / ksplit_of(g); ks < ks1; ++ks) {
        if (!tc::mbar_wait(&empty[stage], phase ^ 1, g.limit_ns, &abort_flag)) { fail(); break; }
        uint8_t* sa = dsm + stage * SB;
        uint8_t* sb = sa + A_BYTES;
        issued |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        tc::mbar_expect_tx(&full[stage], stage_tx(KIND));
        tc::tma_load_2d(sa, &mapA, ks * 128, a_row, &full[stage]);
        if (GROUPED && EPI == EPI_COMBINE_RED) {
          // the routed down weights with an evict-first L2 policy, so that the
          // accumulator slice the combine reduces into stays in L2 (measured
          // ~4 us of ~500 at 8192 tokens; the same on the gate/up weights lost)
          const uint64_t pol = tc::l2_evict_first();
          tc::tma_load_2d_hint(sb, &mapB, ks * 128, b0, &full[stage], pol);
          tc::tma_load_2d_hint(sb + B_BYTES / 2, &mapB, ks * 128, b1, &full[stage], pol);
        } else {
          tc::tma_load_2d(sb, &mapB, ks * 128, b0, &full[stage]);
          tc::tma_load_2d(sb + B_BYTES / 2, &mapB, ks * 128, b1, &full[stage]);
        }
        if (KIND == KIND_FP4) {
          uint8_t* ssa = sb + B_BYTES;
          uint8_t* ssb = ssa + SFA_BYTES;
          const int a_tile = a_row / BM;
          tc::bulk_load(ssa, g.sfa + ((size_t)a_tile * kgroups + 2 * ks) * 512, 1024, &full[stage]);
          const size_t rt0 = (size_t)e * g.sfb_rtiles + (b0 - b_base) / BM;
          const size_t rt1 = (size_t)e * g.sfb_rtiles + (b1 - b_base) / BM;
          tc::bulk_load(ssb, g.sfb + (rt0 * kgroups + 2 * ks) * 512, 1024, &full[stage]);
          tc::bulk_load(ssb + 1024, g.sfb + (rt1 * kgroups + 2 * ks) * 512, 1024, &full[stage]);
        } else if (KIND == KIND_FP8) {  // one K group (128 elements) per stage
          uint8_t* ssa = sb + B_BYTES;
          uint8_t* ssb = ssa + SFA_BYTES;
          const int a_tile = a_row / BM;
          tc::bulk_load(ssa, g.sfa + ((size_t)a_tile * kgroups + ks) * 512, 512, &full[stage]);
          const size_t rt0 = (size_t)e * g.sfb_rtiles + (b0 - b_base) / BM;
          const size_t rt1 = (size_t)e * g.sfb_rtiles + (b1 - b_base) / BM;
          tc::bulk_load(ssb, g.sfb + (rt0 * kgroups + ks) * 512, 512, &full[stage]);
          tc::bulk_load(ssb + 512, g.sfb + (rt1 * kgroups + ks) * 512, 512, &full[stage]);
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    // no copy of this block may still be landing in its shared memory when it
    // exits (after an abort the consumer may not have waited for them): wait,
    // bounded but regardless of the abort flag, for the last copy of each stage
    const int never = 0;
    for (int s2 = 0; s2 < STAGES; ++s2)
      if ((issued >> s2 & 1) && !tc::mbar_wait(&full[s2], last_parity >> s2 & 1, g.limit_ns, &never)) fail();
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    uint32_t stage = 0, phase = 0, acc_phase = 0;
    const uint32_t idesc_bf = tc::idesc_bf16(BM, BN);
    for (int t = blockIdx.x; t < total && !abort_flag; t += gridDim.x) {
      if (!tc::mbar_wait(&acc_empty, acc_phase ^ 1, g.limit_ns, &abort_flag)) { fail(); break; }
      tc::fence_after_sync();
      bool ok = true;
      const int kp = t % ksplit_of(g);
      const int ks0 = kp * nks / ksplit_of(g), ks1 = (kp + 1) * nks / ksplit_of(g);
      for (int ks = ks0; ks < ks1; ++ks) {
        if (!tc::mbar_wait(&full[stage], phase, g.limit_ns, &abort_flag)) { fail(); ok = false; break; }
        tc::fence_after_sync();
        const uint32_t sa = tc::smem_u32(dsm + stage * SB);
        const uint32_t sb = sa + A_BYTES;
        if (KIND == KIND_FP4) {
          const uint32_t ssa = sb + B_BYTES, ssb = ssa + SFA_BYTES;
          const uint32_t ta = tmem + SF_TMEM_BASE + stage * 24;  // 8 columns of A scales, 16 of B
          const uint32_t tb = ta + 8;
          tc::sf_copy(ta + 0, tc::desc_sf(ssa));
          tc::sf_copy(ta + 4, tc::desc_sf(ssa + 512));
          tc::sf_copy(tb + 0, tc::desc_sf(ssb));            // B rows 0..127, group 0
          tc::sf_copy(tb + 4, tc::desc_sf(ssb + 1024));     // B rows 128..255, group 0
          tc::sf_copy(tb + 8, tc::desc_sf(ssb + 512));      // B rows 0..127, group 1
          tc::sf_copy(tb + 12, tc::desc_sf(ssb + 1536));    // B rows 128..255, group 1
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int grp = kk >> 1, id = (kk & 1) * 2;
            tc::mma_mxf4(tmem, tc::desc_sw128(sa + kk * 32), tc::desc_sw128(sb + kk * 32),
                         tc::idesc_mxf4(BM, BN, id, id), ta + 4 * grp, tb + 8 * grp, (ks != ks0) | (kk != 0));
          }
        } else if (KIND == KIND_FP8) {
          const uint32_t ssa = sb + B_BYTES, ssb = ssa + SFA_BYTES;
          const uint32_t ta = tmem + SF_TMEM_BASE + stage * 24;  // 4 columns of A scales, 8 of B
          const uint32_t tb = ta + 8;
          tc::sf_copy(ta, tc::desc_sf(ssa));
          tc::sf_copy(tb + 0, tc::desc_sf(ssb));        // B rows 0..127
          tc::sf_copy(tb + 4, tc::desc_sf(ssb + 512));  // B rows 128..255
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 32 per MMA: scale byte kk of each row's word
            tc::mma_mxf8(tmem, tc::desc_sw128(sa + kk * 32), tc::desc_sw128(sb + kk * 32),
                         tc::idesc_mxf8(BM, BN, kk, kk), ta, tb, (ks != ks0) | (kk != 0));
        } else {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16(tmem, tc::desc_sw128(sa + kk * 32), tc::desc_sw128(sb + kk * 32), idesc_bf,
                         (ks != ks0) | (kk != 0));
        }
        tc::mma_commit(&empty[stage]);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      tc::mma_commit(&acc_full);
      acc_phase ^= 1;
    }
    // wait (bounded, regardless of the abort flag) for every MMA this thread
    // issued before TMEM is released
    const int never = 0;
    tc::mma_commit(&drain);
    if (!tc::mbar_wait(&drain, 0, g.limit_ns, &never)) fail();
  } else if (warp >= 2) {
    // ---------------- epilogue: thread <-> accumulator row m, column quarter cq
    const int q = warp & 3;          // TMEM lane quadrant this warp may read
    const int cq = (warp - 2) >> 2;  // column quarter: 32 h columns, or 64 output columns
    const int m = q * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total && !abort_flag; t += gridDim.x) {
      int a_row, e, rows, srow0, nt, mti, kp;
      tile_coords(g, GROUPED, t, num_mt, a_row, e, rows, srow0, nt, mti, kp);
      // the combine's assignment and routing weight of this thread's four
      // rows, loaded while the tile's MMAs still run
      int ra[4] = {0, 0, 0, 0};
      float rw[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (EPI == EPI_COMBINE_RED) {
        const int r0 = q * 32 + (lane >> 2);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
          if (r0 + 8 * hh < rows) ra[hh] = __ldg(g.perm + srow0 + r0 + 8 * hh);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh)
          if (r0 + 8 * hh < rows) rw[hh] = __ldg(g.topk_w + ra[hh]);
      }
      if (!tc::mbar_wait(&acc_full, acc_phase, g.limit_ns, &abort_flag)) { fail(); break; }
      tc::fence_after_sync();
      float va[32], vb[32];
      if (SWIGLU) {
        tc::tmem_ld32(trow + cq * 32, va);        // G, h columns 32cq ..
        tc::tmem_ld32(trow + 128 + cq * 32, vb);  // U, the same columns
      } else {
        // rows 32q + {0..15} and 32q + {16..31}, columns 64cq .. 64cq + 63
        tc::tmem_ld16x256_x8(trow + cq * 64, va);
        tc::tmem_ld16x256_x8(trow + (16u << 16) + cq * 64, vb);
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&acc_empty);  // the accumulator is free for the next tile
      acc_phase ^= 1;
      if (EPI == EPI_SWIGLU_MX) {
        // h = SiLU(G) U for 32 columns, requantised to MXFP4 (one block); every
        // padded row is written (padding rows quantise zeros).
        const int r = a_row + m;
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          va[i] = silu_fast(va[i]) * vb[i];
          amax = fmaxf(amax, fabsf(va[i]));
        }
        const int ex = mx_scale_exp(amax);
        const float inv = pow2_neg(ex);
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = e2m1x8_rne(*reinterpret_cast<const float(*)[8]>(&va[8 * j]), inv);
        *reinterpret_cast<uint4*>(g.hq + (size_t)r * (g.h_cols / 2) + (nt * 128 + cq * 32) / 2) =
            make_uint4(w[0], w[1], w[2], w[3]);
        const int hgroups = g.h_cols / 128;
        // byte cq of the MMA-layout scale word of row m in group nt
        reinterpret_cast<uint8_t*>(g.hs)[(((size_t)(r / BM) * hgroups + nt) * 128 + (m % 32) * 4 + (m / 32)) * 4 + cq] =
            (uint8_t)(ex + 127);
      } else if (EPI == EPI_SWIGLU_MX8) {
        // h = SiLU(G) U for 32 columns, requantised to MXFP8 (E4M3, one E8M0
        // scale per 32); rows past the tile's real rows are not written.
        if (m < rows) {
          const int r = a_row + m;
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            va[i] = silu_fast(va[i]) * vb[i];
            amax = fmaxf(amax, fabsf(va[i]));
          }
          const int ef = (int)((__float_as_uint(amax) >> 23) & 0xff);
          const int ex = ef == 0 ? -127 : max(ef - 127 - 8, -127);
          const float inv = pow2_neg(ex);
          uint8_t* dst = g.hq + (size_t)r * g.h_cols + nt * 128 + cq * 32;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            const float (&v8)[8] = *reinterpret_cast<const float(*)[8]>(&va[i]);
            *reinterpret_cast<uint2*>(dst + i) = e4m3x8_rne(v8, inv);
          }
          const int hgroups = g.h_cols / 128;
          reinterpret_cast<uint8_t*>(g.hs)[(((size_t)(r / BM) * hgroups + nt) * 128 + (m % 32) * 4 + (m / 32)) * 4 + cq] =
              (uint8_t)(ex + 127);
        }
      } else if (EPI == EPI_SWIGLU_BF16) {
        if (m < rows) {
          uint16_t* dst = g.h_bf16 + (size_t)(srow0 + m) * g.h_cols + nt * 128 + cq * 32;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 o;
            o.x = f32_to_bf16_rn(silu_fast(va[i + 0]) * vb[i + 0]) | ((uint32_t)f32_to_bf16_rn(silu_fast(va[i + 1]) * vb[i + 1]) << 16);
            o.y = f32_to_bf16_rn(silu_fast(va[i + 2]) * vb[i + 2]) | ((uint32_t)f32_to_bf16_rn(silu_fast(va[i + 3]) * vb[i + 3]) << 16);
            o.z = f32_to_bf16_rn(silu_fast(va[i + 4]) * vb[i + 4]) | ((uint32_t)f32_to_bf16_rn(silu_fast(va[i + 5]) * vb[i + 5]) << 16);
            o.w = f32_to_bf16_rn(silu_fast(va[i + 6]) * vb[i + 6]) | ((uint32_t)f32_to_bf16_rn(silu_fast(va[i + 7]) * vb[i + 7]) << 16);
            *reinterpret_cast<uint4*>(dst + i) = o;
          }
        }
      } else if (EPI == EPI_COMBINE_RED) {
        // A9 fused: each real row's 64 columns, times its routing weight, are
        // added into its token's FP32 output row by vector reductions (four
        // threads share a row: every warp reduction covers whole sectors)
        const int r0 = q * 32 + (lane >> 2);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const int r = r0 + 8 * hh;  // hh: lanes +0, +8 (first load), +16, +24 (second)
          if (r < rows) {
            const size_t tok = (size_t)(ra[hh] / g.k_top);
            float* dst = (g.slice_rows ? g.out + ((size_t)nt * g.slice_rows + tok) * BN
                                       : g.out + tok * g.ldo + nt * BN) + cq * 64 + 2 * (lane & 3);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float* v = hh < 2 ? va : vb;
              const int o = 4 * j + 2 * (hh & 1);
              red_add_f32x2(dst + 8 * j, rw[hh] * v[o], rw[hh] * v[o + 1]);
            }
          }
        }
      } else {
        // Four threads share a row, so each warp store fills eight whole
        // 32-byte sectors (a row-per-thread store fills 32 half sectors).
        const int r0 = q * 32 + (lane >> 2);
        const bool sl = g.slice_rows > 0;
        float* base = (sl ? g.out + ((size_t)nt * g.slice_rows + srow0) * BN
                          : g.out + kp * g.part_stride + (size_t)srow0 * g.ldo + nt * BN) + cq * 64 + 2 * (lane & 3);
        const size_t rstride = sl ? (size_t)BN : (size_t)g.ldo;
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const int r = r0 + 8 * hh;  // hh: lanes +0, +8 (first load), +16, +24 (second)
          if (r < rows) {
            float* dst = base + (size_t)r * rstride;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float* v = hh < 2 ? va : vb;
              const int o = 4 * j + 2 * (hh & 1);
              *reinterpret_cast<float2*>(dst + 8 * j) = make_float2(v[o], v[o + 1]);
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
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------- weights-as-A grouped GEMM
//
// With a few tokens per expert (batched decode) the routed GEMMs above would
// carry up to 127 padding rows in every 128-row token tile.  This variant
// swaps the operands: 128 weight rows are the MMA's A (M = 128) and the
// expert's tokens are B, a window of up to WA_WIN rows of the per-expert
// padded order (N = the window's real rows rounded up to 16, moved as 16-row
// TMA boxes), so an SM streams weights and little else.  TMEM lane = weight
// row, column = token.  Two accumulator buffers of 128 columns (gate 0..63
// and up 64..127, or down 0..63) let the next tile's MMAs overlap the
// epilogue.  Epilogues:
//   EPI_SWIGLU_MX  lane = h column; the 32 lanes of a warp are one MXFP4
//                  block of h for each token: amax and the packed codes by
//                  warp shuffles, h rows written in the padded window order
//                  with their scales in the MMA layout of 64-row windows;
//   EPI_STORE_F32  lane = output column; each warp store writes one token's
//                  32 consecutive FP32 outputs (a whole 128-byte line).
// GemmArgs here: sfa = the token operand's scale blocks (per window), sfb =
// the weights' ([E][R/128][K/128][512]), b_rows_per_expert / sfb_rtiles /
// b_up_off describe the weights, n_tiles = 128-row weight tiles per window.

constexpr int WA_WIN = 64;
constexpr uint32_t WA_B_BYTES = WA_WIN * 128;
constexpr uint32_t WA_ACC_COLS = 128;
constexpr uint32_t WA_SF_BASE = 2 * WA_ACC_COLS;
template <int NA> __host__ __device__ constexpr uint32_t wa_stage_bytes() {
  return NA * A_BYTES + WA_B_BYTES + NA * 1024 + 1024;
}
// 172 / 156 KB of stages per SM (deeper rings, 5 / 8 stages, measured no faster)
template <int NA> __host__ __device__ constexpr int wa_stages() { return NA == 2 ? 4 : 6; }

template <int EPI>
__global__ void __launch_bounds__(TC_THREADS, 1)
    k_tc_gemm_wa(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapX, GemmArgs g) {
  constexpr bool SWIGLU = EPI == EPI_SWIGLU_MX;
  constexpr int NA = SWIGLU ? 2 : 1;  // weight tiles per stage: gate + up, or down
  constexpr int NS = wa_stages<NA>();
  constexpr uint32_t SB = wa_stage_bytes<NA>();
  constexpr uint32_t OFF_B = NA * A_BYTES, OFF_SFA = OFF_B + WA_B_BYTES, OFF_SFB = OFF_SFA + NA * 1024;
  constexpr uint32_t SF_COLS = 8 * NA + 8;  // TMEM scale columns per stage
  static_assert(WA_SF_BASE + NS * SF_COLS <= TMEM_COLS, "TMEM columns");
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[NS], empty[NS], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], 32 * EPI_WARPS);
    }
    tc::mbar_init(&drain, 1);
    tc::mbar_fence_init();
    abort_flag = 0;
    tc::prefetch_tensormap(&mapW);
    tc::prefetch_tensormap(&mapX);
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const int total = *g.num_mt * g.n_tiles;
  const int nks = g.K / 256;
  const int kgroups = g.K / 128;

  auto fail = [&]() {
    atomicCAS(g.status, 0, (int)MOE_DEV_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };

  if (warp == 0 && lane == 0) {
    // ---------------- producer
    uint32_t stage = 0, phase = 0, issued = 0, last_parity = 0;
    MTile mn = (int)blockIdx.x < total ? g.mt[blockIdx.x / g.n_tiles] : MTile{};
    for (int t = blockIdx.x; t < total && !abort_flag; t += gridDim.x) {
      const int nt = t % g.n_tiles;
      const MTile m = mn;
      // the next tile's window, loaded a tile ahead so its latency overlaps the stream
      if (t + (int)gridDim.x < total) mn = g.mt[(t + gridDim.x) / g.n_tiles];
      const int nb = (m.rows + 15) >> 4;  // 16-row token boxes
      const int wr0 = m.e * g.b_rows_per_expert + nt * BM;
      const size_t rt0 = (size_t)m.e * g.sfb_rtiles + nt;
      const size_t rt1 = rt0 + g.b_up_off / BM;
      const size_t win = (size_t)(m.prow0 / WA_WIN);
      const uint32_t bytes = NA * (A_BYTES + 1024) + (uint32_t)nb * 2048 + 1024;
      for (int ks = 0; ks < nks; ++ks) {
        if (!tc::mbar_wait(&empty[stage], phase ^ 1, g.limit_ns, &abort_flag)) { fail(); break; }
        uint8_t* st = dsm + stage * SB;
        issued |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        tc::mbar_expect_tx(&full[stage], bytes);
        tc::tma_load_2d(st, &mapW, ks * 128, wr0, &full[stage]);
        if (SWIGLU) tc::tma_load_2d(st + A_BYTES, &mapW, ks * 128, wr0 + g.b_up_off, &full[stage]);
        for (int b = 0; b < nb; ++b)
          tc::tma_load_2d(st + OFF_B + b * 2048, &mapX, ks * 128, m.prow0 + 16 * b, &full[stage]);
        tc::bulk_load(st + OFF_SFA, g.sfb + (rt0 * kgroups + 2 * ks) * 512, 1024, &full[stage]);
        if (SWIGLU) tc::bulk_load(st + OFF_SFA + 1024, g.sfb + (rt1 * kgroups + 2 * ks) * 512, 1024, &full[stage]);
        tc::bulk_load(st + OFF_SFB, g.sfa + (win * kgroups + 2 * ks) * 512, 1024, &full[stage]);
        if (++stage == NS) { stage = 0; phase ^= 1; }
      }
    }
    // the last copy of each stage has landed before the block may exit
    const int never = 0;
    for (int s2 = 0; s2 < NS; ++s2)
      if ((issued >> s2 & 1) && !tc::mbar_wait(&full[s2], last_parity >> s2 & 1, g.limit_ns, &never)) fail();
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    uint32_t stage = 0, phase = 0;
    int it = 0;
    int rows_n = (int)blockIdx.x < total ? g.mt[blockIdx.x / g.n_tiles].rows : 0;
    for (int t = blockIdx.x; t < total && !abort_flag; t += gridDim.x, ++it) {
      const int buf = it & 1;
      const int N = (rows_n + 15) & ~15;
      if (t + (int)gridDim.x < total) rows_n = g.mt[(t + gridDim.x) / g.n_tiles].rows;  // a tile ahead
      if (!tc::mbar_wait(&acc_empty[buf], ((it >> 1) & 1) ^ 1, g.limit_ns, &abort_flag)) { fail(); break; }
      tc::fence_after_sync();
      const uint32_t acc = tmem + buf * WA_ACC_COLS;
      bool ok = true;
      for (int ks = 0; ks < nks; ++ks) {
        if (!tc::mbar_wait(&full[stage], phase, g.limit_ns, &abort_flag)) { fail(); ok = false; break; }
        tc::fence_after_sync();
        const uint32_t sa = tc::smem_u32(dsm + stage * SB);
        const uint32_t sb = sa + OFF_B, ssa = sa + OFF_SFA, ssb = sa + OFF_SFB;
        // weight tile a's scales at columns tsf + 8a (+4 for the second K group), the tokens' at tsf + 8 NA
        const uint32_t tsf = tmem + WA_SF_BASE + stage * SF_COLS;
        tc::sf_copy(tsf + 0, tc::desc_sf(ssa));
        tc::sf_copy(tsf + 4, tc::desc_sf(ssa + 512));
        if (SWIGLU) {
          tc::sf_copy(tsf + 8, tc::desc_sf(ssa + 1024));
          tc::sf_copy(tsf + 12, tc::desc_sf(ssa + 1536));
        }
        tc::sf_copy(tsf + 8 * NA, tc::desc_sf(ssb));
        tc::sf_copy(tsf + 8 * NA + 4, tc::desc_sf(ssb + 512));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int grp = kk >> 1, id = (kk & 1) * 2;
          const uint32_t idesc = tc::idesc_mxf4(BM, N, id, id);
          const uint64_t bdesc = tc::desc_sw128(sb + kk * 32);
          tc::mma_mxf4(acc, tc::desc_sw128(sa + kk * 32), bdesc, idesc, tsf + 4 * grp, tsf + 8 * NA + 4 * grp,
                       (ks | kk) != 0);
          if (SWIGLU)
            tc::mma_mxf4(acc + 64, tc::desc_sw128(sa + A_BYTES + kk * 32), bdesc, idesc, tsf + 8 + 4 * grp,
                         tsf + 8 * NA + 4 * grp, (ks | kk) != 0);
        }
        tc::mma_commit(&empty[stage]);
        if (++stage == NS) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      tc::mma_commit(&acc_full[buf]);
    }
    const int never = 0;
    tc::mma_commit(&drain);
    if (!tc::mbar_wait(&drain, 0, g.limit_ns, &never)) fail();
  } else if (warp >= 2) {
    // ---------------- epilogue: lane <-> weight row 32q + lane, token columns 16cq .. 16cq + 15
    const int q = warp & 3;
    const int cq = (warp - 2) >> 2;
    const int j0 = 16 * cq;
    const uint32_t tlane = tmem + ((uint32_t)(q * 32) << 16);
    int it = 0;
    MTile mn = (int)blockIdx.x < total ? g.mt[blockIdx.x / g.n_tiles] : MTile{};
    for (int t = blockIdx.x; t < total && !abort_flag; t += gridDim.x, ++it) {
      const int buf = it & 1;
      const int nt = t % g.n_tiles;
      const MTile m = mn;
      if (t + (int)gridDim.x < total) mn = g.mt[(t + gridDim.x) / g.n_tiles];  // a tile ahead
      if (!tc::mbar_wait(&acc_full[buf], (it >> 1) & 1, g.limit_ns, &abort_flag)) { fail(); break; }
      tc::fence_after_sync();
      const bool active = j0 < ((m.rows + 15) & ~15);  // the same in the whole warp
      float va[16], vb[16];
      if (active) {
        tc::tmem_ld16(tlane + buf * WA_ACC_COLS + j0, va);
        if (SWIGLU) tc::tmem_ld16(tlane + buf * WA_ACC_COLS + 64 + j0, vb);
      }
      tc::fence_before_sync();
      tc::mbar_arrive(&acc_empty[buf]);  // the accumulator is free for the tile after next
      if (!active) continue;
      if (EPI == EPI_SWIGLU_MX) {
        const int c0 = nt * BM + q * 32;  // this warp's MXFP4 block of h columns
        const int hgroups = g.h_cols / 128;
        uint8_t* hs = reinterpret_cast<uint8_t*>(g.hs) + ((size_t)(m.prow0 / WA_WIN) * hgroups + nt) * 512;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float h = silu_fast(va[j]) * vb[j];
          float amax = fabsf(h);
#pragma unroll
          for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          const int ex = mx_scale_exp(amax);
          uint32_t v = e2m1_rne(h * pow2_neg(ex)) << (4 * (lane & 7));
          v |= __shfl_xor_sync(0xffffffffu, v, 1);
          v |= __shfl_xor_sync(0xffffffffu, v, 2);
          v |= __shfl_xor_sync(0xffffffffu, v, 4);
          const int r = j0 + j;  // window row
          if ((lane & 7) == 0)
            *reinterpret_cast<uint32_t*>(g.hq + (size_t)(m.prow0 + r) * (g.h_cols / 2) + c0 / 2 + lane / 2) = v;
          if (lane == 0) hs[((r % 32) * 4 + r / 32) * 4 + q] = (uint8_t)(ex + 127);
        }
      } else {
        float* dst = g.out + (size_t)(m.srow0 + j0) * g.ldo + nt * BM + q * 32 + lane;
        const int nj = min(16, m.rows - j0);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < nj) dst[(size_t)j * g.ldo] = va[j];
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

// --------------------------------------------------------- h inspection

// One block per (padded tile, 128 rows): the requantised h of each real row,
// codes and unscrambled scales, to its sorted-assignment position; or, when
// h was left in sorted order, a plain copy.
__global__ void __launch_bounds__(128) k_copy_h(int n, int I, const int* __restrict__ hpath,
                                                const uint8_t* __restrict__ hq_sorted, const uint8_t* __restrict__ hs_sorted,
                                                const MTile* __restrict__ tiles, const int* __restrict__ num_tiles,
                                                const uint8_t* __restrict__ hq_perm, const uint32_t* __restrict__ hs_mma,
                                                uint8_t* __restrict__ hq_out, uint8_t* __restrict__ hs_out) {
  const int m = threadIdx.x;
  const int groups = I / 128;
  const int path = *hpath & 0xff;  // written by a byte-wise memset
  if (path == 0) {
    const int p = blockIdx.x * 128 + m;
    if (p >= n) return;
    for (int c = 0; c < I / 32; ++c)
      reinterpret_cast<uint4*>(hq_out + (size_t)p * (I / 2))[c] = reinterpret_cast<const uint4*>(hq_sorted + (size_t)p * (I / 2))[c];
    for (int c = 0; c < I / 32; ++c) hs_out[(size_t)p * (I / 32) + c] = hs_sorted[(size_t)p * (I / 32) + c];
    return;
  }
  // h in the padded order: windows of 128 rows (hpath 1) or 64 (hpath 2)
  const int win = path == 2 ? 64 : 128;
  if ((int)blockIdx.x >= *num_tiles) return;
  const MTile t = tiles[blockIdx.x];
  if (m >= t.rows) return;
  const int r = t.prow0 + m, p = t.srow0 + m;
  for (int c = 0; c < I / 32; ++c)
    reinterpret_cast<uint4*>(hq_out + (size_t)p * (I / 2))[c] = reinterpret_cast<const uint4*>(hq_perm + (size_t)r * (I / 2))[c];
  for (int g = 0; g < groups; ++g) {
    const uint32_t w = hs_mma[((size_t)(r / win) * groups + g) * 128 + (m % 32) * 4 + (m / 32)];
    for (int b = 0; b < 4; ++b) hs_out[(size_t)p * (I / 32) + 4 * g + b] = (uint8_t)(w >> (8 * b));
  }
}

cudaError_t launch_copy_h(const Shape& sh, const int* hpath, const uint8_t* hq_sorted, const uint8_t* hs_sorted,
                          const TcWorkspace& w, uint8_t* hq_out, uint8_t* hs_out, cudaStream_t s) {
  const int n = sh.T * sh.k;
  if (n == 0) return cudaSuccess;
  const int blocks = tc_routed_enabled(n) ? max(max(tc_padded_rows(n, sh.E) / BM, tc_padded_rows_win(n, sh.E, 64) / 64),
                                                (n + 127) / 128)
                                          : (n + 127) / 128;
  count_launch(), k_copy_h<<<blocks, 128, 0, s>>>(n, sh.I, hpath, hq_sorted, hs_sorted, reinterpret_cast<const MTile*>(w.mtiles),
                                  w.num_mt, w.hq_perm, reinterpret_cast<const uint32_t*>(w.hs_mma), hq_out, hs_out);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ host

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

cudaError_t make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

namespace {

template <int KIND, int EPI, bool GROUPED>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& g, int max_tiles, cudaStream_t s) {
  const size_t smem = (size_t)STAGES * stage_bytes(KIND) + 1024;
  const void* fn = (const void*)k_tc_gemm<KIND, EPI, GROUPED>;
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = max(1, min(max_tiles, sm_count()));
  count_launch(), k_tc_gemm<KIND, EPI, GROUPED><<<grid, TC_THREADS, smem, s>>>(a, b, g);
  return cudaGetLastError();
}

template <int EPI>
cudaError_t launch_gemm_wa(const CUtensorMap& w, const CUtensorMap& x, const GemmArgs& g, int max_tiles,
                           cudaStream_t s) {
  constexpr int NA = EPI == EPI_SWIGLU_MX ? 2 : 1;
  const size_t smem = (size_t)wa_stages<NA>() * wa_stage_bytes<NA>() + 1024;
  const void* fn = (const void*)k_tc_gemm_wa<EPI>;
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = max(1, min(max_tiles, sm_count()));
  count_launch(), k_tc_gemm_wa<EPI><<<grid, TC_THREADS, smem, s>>>(w, x, g);
  return cudaGetLastError();
}

}  // namespace

bool tc_weights_as_a(int n, int E, int mode) {
  return mode == TC_GEMM_WEIGHTS_AS_A || (mode == TC_GEMM_AUTO && n <= WA_MAX_AVG_ROWS * E);
}

cudaError_t launch_expert_ffn_tc(const Shape& sh, const ExpertsDev& ex, const TcWorkspace& w, const uint8_t* xq,
                                 const uint8_t* xs, const int* offsets, const int* perm, float* y_assign,
                                 int* status, uint64_t limit_ns, bool wa, cudaStream_t s, const CombineArgs* comb) {
  const int H = sh.H, I = sh.I, E = sh.E;
  const int n = sh.T * sh.k;
  if (n == 0) return cudaSuccess;
  if (comb && wa) return cudaErrorInvalidValue;  // the fused combine exists for 128-token tiles as A
  const int win = wa ? WA_WIN : BM;
  const int rmax = tc_padded_rows_win(n, E, win);
  cudaError_t err;
  count_launch(), k_build_mtiles<<<1, 256, 0, s>>>(offsets, E, win, w.poff, reinterpret_cast<MTile*>(w.mtiles), w.num_mt);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  count_launch(), k_gather_mx_rows<<<rmax / GR, 128, 0, s>>>(xq, xs, H, sh.k, perm, reinterpret_cast<const MTile*>(w.mtiles),
                                             w.num_mt, win, wa ? 1 : 0, w.xq_perm,
                                             reinterpret_cast<uint32_t*>(w.xs_mma), n, status);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const uint8_t* w13s_mma = ex.w13s_mma;
  const uint8_t* w2s_mma = ex.w2s_mma;
  if (!w13s_mma || !w2s_mma) {  // not prepared at load time: re-lay the scales for this call
    if ((err = launch_relayout_weight_sf(ex.w13s, E, 2 * I, H, w.w13s_mma, s)) != cudaSuccess) return err;
    if ((err = launch_relayout_weight_sf(ex.w2s, E, H, I, w.w2s_mma, s)) != cudaSuccess) return err;
    w13s_mma = w.w13s_mma;
    w2s_mma = w.w2s_mma;
  }
  const int max_mt = rmax / win;
  CUtensorMap ma, mb;
  record_mark(MARK_ROUTED_GEMM_BEGIN, s);
  if (wa) {
    // gate/up: A = W13 [E*2I][H/2], B = gathered activations [rmax][H/2] in 16-row boxes
    if ((err = make_map(&ma, ex.w13, (uint64_t)E * 2 * I, H / 2)) != cudaSuccess) return err;
    if ((err = make_map(&mb, w.xq_perm, rmax, H / 2, 16)) != cudaSuccess) return err;
    GemmArgs g1{};
    g1.K = H;
    g1.n_tiles = I / BM;
    g1.num_mt = w.num_mt;
    g1.mt = reinterpret_cast<const MTile*>(w.mtiles);
    g1.b_rows_per_expert = 2 * I;
    g1.b_up_off = I;
    g1.sfa = w.xs_mma;
    g1.sfb = w13s_mma;
    g1.sfb_rtiles = 2 * I / BM;
    g1.hq = w.hq_perm;
    g1.hs = reinterpret_cast<uint32_t*>(w.hs_mma);
    g1.h_cols = I;
    g1.status = status;
    g1.limit_ns = limit_ns;
    if ((err = launch_gemm_wa<EPI_SWIGLU_MX>(ma, mb, g1, max_mt * g1.n_tiles, s)) != cudaSuccess) return err;
    // down: A = W2 [E*H][I/2], B = requantised h [rmax][I/2]
    if ((err = make_map(&ma, ex.w2, (uint64_t)E * H, I / 2)) != cudaSuccess) return err;
    if ((err = make_map(&mb, w.hq_perm, rmax, I / 2, 16)) != cudaSuccess) return err;
    GemmArgs g2{};
    g2.K = I;
    g2.n_tiles = H / BM;
    g2.num_mt = w.num_mt;
    g2.mt = reinterpret_cast<const MTile*>(w.mtiles);
    g2.b_rows_per_expert = H;
    g2.sfa = w.hs_mma;
    g2.sfb = w2s_mma;
    g2.sfb_rtiles = H / BM;
    g2.out = y_assign;
    g2.ldo = H;
    g2.status = status;
    g2.limit_ns = limit_ns;
    if ((err = launch_gemm_wa<EPI_STORE_F32>(ma, mb, g2, max_mt * g2.n_tiles, s)) != cudaSuccess) return err;
    record_mark(MARK_ROUTED_GEMM_END, s);
    return cudaSuccess;
  }
  // gate/up: A = gathered activations [rmax][H/2], B = W13 [E*2I][H/2]
  if ((err = make_map(&ma, w.xq_perm, rmax, H / 2)) != cudaSuccess) return err;
  if ((err = make_map(&mb, ex.w13, (uint64_t)E * 2 * I, H / 2)) != cudaSuccess) return err;
  GemmArgs g1{};
  g1.K = H;
  g1.n_tiles = I / 128;
  g1.num_mt = w.num_mt;
  g1.mt = reinterpret_cast<const MTile*>(w.mtiles);
  g1.b_rows_per_expert = 2 * I;
  g1.b_up_off = I;
  g1.sfa = w.xs_mma;
  g1.sfb = w13s_mma;
  g1.sfb_rtiles = 2 * I / 128;
  g1.hq = w.hq_perm;
  g1.hs = reinterpret_cast<uint32_t*>(w.hs_mma);
  g1.h_cols = I;
  g1.status = status;
  g1.limit_ns = limit_ns;
  if ((err = launch_gemm<KIND_FP4, EPI_SWIGLU_MX, true>(ma, mb, g1, max_mt * g1.n_tiles, s)) != cudaSuccess) return err;
  // down: A = requantised h [rmax][I/2], B = W2 [E*H][I/2]
  if ((err = make_map(&ma, w.hq_perm, rmax, I / 2)) != cudaSuccess) return err;
  if ((err = make_map(&mb, ex.w2, (uint64_t)E * H, I / 2)) != cudaSuccess) return err;
  GemmArgs g2{};
  g2.K = I;
  g2.n_tiles = H / BN;
  g2.num_mt = w.num_mt;
  g2.mt = reinterpret_cast<const MTile*>(w.mtiles);
  g2.b_rows_per_expert = H;
  g2.sfa = w.hs_mma;
  g2.sfb = w2s_mma;
  g2.sfb_rtiles = H / 128;
  g2.out = y_assign;
  g2.ldo = H;
  g2.status = status;
  g2.limit_ns = limit_ns;
  if (comb) {
    // the combine in the epilogue: tiles of one 256-column slice of the
    // output in turn, so that slice of the FP32 accumulator (T x 1 KB) stays
    // in L2 while every expert adds into it
    g2.out = comb->acc;
    g2.perm = perm;
    g2.topk_w = comb->topk_w;
    g2.k_top = sh.k;
    g2.n_major = 1;
    g2.slice_rows = comb->slice_rows;
    err = launch_gemm<KIND_FP4, EPI_COMBINE_RED, true>(ma, mb, g2, max_mt * g2.n_tiles, s);
  } else {
    err = launch_gemm<KIND_FP4, EPI_STORE_F32, true>(ma, mb, g2, max_mt * g2.n_tiles, s);
  }
  if (err != cudaSuccess) return err;
  record_mark(MARK_ROUTED_GEMM_END, s);
  return cudaSuccess;
}

namespace {

// out[t][c] = BF16(acc at (t, c)), four consecutive columns per thread; acc
// row-major [T][H] or (slice_rows = T) by 256-column slices [H/256][T][256].
__global__ void __launch_bounds__(256) k_acc_to_bf16(const float* __restrict__ acc, size_t n4, int H, int slice_rows,
                                                     uint16_t* __restrict__ out) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  size_t src = i;
  if (slice_rows) {
    const size_t t = i / (H / 4), c = (i % (H / 4)) * 4;
    src = ((c / 256) * slice_rows + t) * 64 + (c % 256) / 4;
  }
  const float4 v = __ldcs(reinterpret_cast<const float4*>(acc) + src);
  uint2 o;
  o.x = (uint32_t)f32_to_bf16_rn(v.x) | ((uint32_t)f32_to_bf16_rn(v.y) << 16);
  o.y = (uint32_t)f32_to_bf16_rn(v.z) | ((uint32_t)f32_to_bf16_rn(v.w) << 16);
  reinterpret_cast<uint2*>(out)[i] = o;
}

}  // namespace

cudaError_t launch_acc_to_bf16(const float* acc, int T, int H, int slice_rows, uint16_t* out, cudaStream_t s) {
  const size_t n4 = (size_t)T * H / 4;
  if (n4 == 0) return cudaSuccess;
  count_launch(), k_acc_to_bf16<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(acc, n4, H, slice_rows, out);
  return cudaGetLastError();
}

namespace {

// Split-K finishers of the shared expert (parts summed in ascending order).
// h[t][c] = BF16(SiLU(G) U), G and U the sums of parts [S][T][2I] at columns
// c and I + c; four columns per thread.
__global__ void __launch_bounds__(256) k_swiglu_parts(const float* __restrict__ parts, int S, int T, int I,
                                                      uint16_t* __restrict__ h) {
  const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i >= (size_t)T * I) return;
  const size_t t = i / I, c = i % I;
  const size_t stride = (size_t)T * 2 * I;
  const float* pg = parts + t * 2 * I + c;
  float4 gs = *reinterpret_cast<const float4*>(pg), us = *reinterpret_cast<const float4*>(pg + I);
  for (int p = 1; p < S; ++p) {
    const float4 a = *reinterpret_cast<const float4*>(pg + p * stride);
    const float4 b = *reinterpret_cast<const float4*>(pg + p * stride + I);
    gs.x += a.x; gs.y += a.y; gs.z += a.z; gs.w += a.w;
    us.x += b.x; us.y += b.y; us.z += b.z; us.w += b.w;
  }
  uint2 o;
  o.x = f32_to_bf16_rn(silu(gs.x) * us.x) | ((uint32_t)f32_to_bf16_rn(silu(gs.y) * us.y) << 16);
  o.y = f32_to_bf16_rn(silu(gs.z) * us.z) | ((uint32_t)f32_to_bf16_rn(silu(gs.w) * us.w) << 16);
  *reinterpret_cast<uint2*>(h + i) = o;
}

// out[i] = sum of parts [S][n] at i, four elements per thread; with
// slice_rows = T the parts are [S][T][H] and out is laid out by 256-column
// slices, [H/256][T][256].
__global__ void __launch_bounds__(256) k_sum_parts(const float* __restrict__ parts, int S, size_t n, int H,
                                                   int slice_rows, float* __restrict__ out) {
  const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i >= n) return;
  float4 v = *reinterpret_cast<const float4*>(parts + i);
  for (int p = 1; p < S; ++p) {
    const float4 a = *reinterpret_cast<const float4*>(parts + p * n + i);
    v.x += a.x; v.y += a.y; v.z += a.z; v.w += a.w;
  }
  size_t dst = i;
  if (slice_rows) {
    const size_t t = i / H, c = i % H;
    dst = ((c / 256) * slice_rows + t) * 256 + c % 256;
  }
  *reinterpret_cast<float4*>(out + dst) = v;
}

}  // namespace

cudaError_t launch_shared_mxfp8_tc(const Shape& sh, const Shared8Dev& sh8, const uint16_t* x, const Shared8Ws& w,
                                   float* y_shared, int* status, uint64_t limit_ns, cudaStream_t s, int slice_rows) {
  const int T = sh.T, H = sh.H, I = sh.I;
  if (T == 0) return cudaSuccess;
  const int mt = (T + BM - 1) / BM;
  const int tpad = mt * BM;
  cudaError_t err;
  // the token (MXFP8, scales into the MMA layout over 128-row tiles; padding
  // rows' scales are never used) and the weights' scales in the MMA layout
  if ((err = launch_quant_mxfp8(x, T, H, w.xq, w.xs, s)) != cudaSuccess) return err;
  if ((err = launch_relayout_weight_sf(w.xs, 1, tpad, H, w.xs_mma, s)) != cudaSuccess) return err;
  // the weights' scales: prepared at load time, else re-laid for this call
  const uint8_t* w13s_mma = sh8.w13s_mma;
  const uint8_t* w2s_mma = sh8.w2s_mma;
  if (!w13s_mma || !w2s_mma) {
    if ((err = launch_relayout_weight_sf(sh8.w13s, 1, 2 * I, H, w.w13s_mma, s)) != cudaSuccess) return err;
    if ((err = launch_relayout_weight_sf(sh8.w2s, 1, H, I, w.w2s_mma, s)) != cudaSuccess) return err;
    w13s_mma = w.w13s_mma;
    w2s_mma = w.w2s_mma;
  }
  CUtensorMap ma, mb;
  // gate/up: A = xq [T][H] E4M3, B = W13 [2I][H] E4M3; SwiGLU + MXFP8 requantise
  if ((err = make_map(&ma, w.xq, T, H)) != cudaSuccess) return err;
  if ((err = make_map(&mb, sh8.w13, (uint64_t)2 * I, H)) != cudaSuccess) return err;
  GemmArgs g1{};
  g1.K = H;
  g1.n_tiles = I / 128;
  g1.num_mt_dense = mt;
  g1.rows_dense = T;
  g1.b_up_off = I;
  g1.sfa = w.xs_mma;
  g1.sfb = w13s_mma;
  g1.sfb_rtiles = 2 * I / BM;
  g1.hq = w.hq;
  g1.hs = reinterpret_cast<uint32_t*>(w.hs_mma);
  g1.h_cols = I;
  g1.status = status;
  g1.limit_ns = limit_ns;
  if ((err = launch_gemm<KIND_FP8, EPI_SWIGLU_MX8, false>(ma, mb, g1, mt * g1.n_tiles, s)) != cudaSuccess) return err;
  // down: A = hq [T][I] E4M3, B = W2 [H][I] E4M3 -> y_shared FP32
  if ((err = make_map(&ma, w.hq, T, I)) != cudaSuccess) return err;
  if ((err = make_map(&mb, sh8.w2, H, I)) != cudaSuccess) return err;
  GemmArgs g2{};
  g2.K = I;
  g2.n_tiles = H / BN;
  g2.num_mt_dense = mt;
  g2.rows_dense = T;
  g2.sfa = w.hs_mma;
  g2.sfb = w2s_mma;
  g2.sfb_rtiles = H / BM;
  g2.out = y_shared;
  g2.ldo = H;
  g2.slice_rows = slice_rows;
  g2.status = status;
  g2.limit_ns = limit_ns;
  return launch_gemm<KIND_FP8, EPI_STORE_F32, false>(ma, mb, g2, mt * g2.n_tiles, s);
}

cudaError_t launch_shared_tc(const Shape& sh, const SharedDev& shd, const uint16_t* x, uint16_t* h_shared,
                             float* y_shared, float* parts, int* status, uint64_t limit_ns, cudaStream_t s,
                             int slice_rows) {
  const int T = sh.T, H = sh.H, I = sh.I;
  if (T == 0) return cudaSuccess;
  const int mt = (T + BM - 1) / BM;
  CUtensorMap ma, mb;
  cudaError_t err;
  // Few tokens: the 128 x 256 tiles alone would leave most SMs idle, so K is
  // split and small kernels finish (the same parts for every T: the choice
  // depends on the shape only).
  const int s1 = shared_ksplit(shared_tiles_gu(T, I), H / 64);
  const int s2 = shared_ksplit(shared_tiles_dn(T, H), I / 64);
  if (s1 > 1) {
    if ((err = make_map(&ma, x, T, (uint64_t)H * 2)) != cudaSuccess) return err;
    if ((err = make_map(&mb, shd.w13, (uint64_t)2 * I, (uint64_t)H * 2)) != cudaSuccess) return err;
    GemmArgs g1{};
    g1.K = H;
    g1.n_tiles = 2 * I / BN;
    g1.num_mt_dense = mt;
    g1.rows_dense = T;
    g1.out = parts;
    g1.ldo = 2 * I;
    g1.ksplit = s1;
    g1.part_stride = (size_t)T * 2 * I;
    g1.status = status;
    g1.limit_ns = limit_ns;
    if ((err = launch_gemm<KIND_BF16, EPI_STORE_F32, false>(ma, mb, g1, mt * g1.n_tiles * s1, s)) != cudaSuccess)
      return err;
    const size_t n4 = (size_t)T * I / 4;
    count_launch(), k_swiglu_parts<<<(unsigned)((n4 + 255) / 256), 256, 0, s>>>(parts, s1, T, I, h_shared);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  } else {
    if ((err = make_map(&ma, x, T, (uint64_t)H * 2)) != cudaSuccess) return err;
    if ((err = make_map(&mb, shd.w13, (uint64_t)2 * I, (uint64_t)H * 2)) != cudaSuccess) return err;
    GemmArgs g1{};
    g1.K = H;
    g1.n_tiles = I / 128;
    g1.num_mt_dense = mt;
    g1.rows_dense = T;
    g1.b_up_off = I;
    g1.h_bf16 = h_shared;
    g1.h_cols = I;
    g1.status = status;
    g1.limit_ns = limit_ns;
    if ((err = launch_gemm<KIND_BF16, EPI_SWIGLU_BF16, false>(ma, mb, g1, mt * g1.n_tiles, s)) != cudaSuccess)
      return err;
  }
  if ((err = make_map(&ma, h_shared, T, (uint64_t)I * 2)) != cudaSuccess) return err;
  if ((err = make_map(&mb, shd.w2, H, (uint64_t)I * 2)) != cudaSuccess) return err;
  GemmArgs g2{};
  g2.K = I;
  g2.n_tiles = H / BN;
  g2.num_mt_dense = mt;
  g2.rows_dense = T;
  g2.out = s2 > 1 ? parts : y_shared;
  g2.ldo = H;
  g2.slice_rows = s2 > 1 ? 0 : slice_rows;
  g2.ksplit = s2;
  g2.part_stride = (size_t)T * H;
  g2.status = status;
  g2.limit_ns = limit_ns;
  if ((err = launch_gemm<KIND_BF16, EPI_STORE_F32, false>(ma, mb, g2, mt * g2.n_tiles * s2, s)) != cudaSuccess)
    return err;
  if (s2 > 1) {
    const size_t n = (size_t)T * H;
    count_launch(), k_sum_parts<<<(unsigned)((n / 4 + 255) / 256), 256, 0, s>>>(parts, s2, n, H, slice_rows,
                                                                               y_shared);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace moefp4
