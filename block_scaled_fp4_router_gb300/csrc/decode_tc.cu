// A10 on tensor cores: the whole MoE layer for decode steps of 1-16 tokens in
// one launch, every contraction on tcgen05 (AMD technical article
// "MiniMax-M3.1 on AMD Instinct GPUs", section "What we Optimized": the "mono
// decode" path runs a pure decode step of at most 16 tokens as one fused MoE
// launch), and the same launch for wider steps of 17-128 tokens (the
// article's section "What's next": wider mono steps).
//
// A decode step streams every touched weight byte once, so the layer is
// bound by HBM.  The weights are the MMA's A operand (128 weight rows per
// MMA, moved by TMA through a shared-memory ring) and the 1-16 token rows are
// a 16-row B operand, so every SM keeps weights in flight without spending
// CUDA-core issue slots on FP4 decoding.
//
// Work units (one block per SM, cooperative launch; one unit list, the same
// in every block, handed out round-robin or, for 16-token-class steps,
// dynamically in increasing order -- see UQ):
//   SGU  shared gate/up:  128 gate + 128 up rows x a K part (BF16 kind::f16,
//                         or MXFP8 kind::mxf8f6f4)
//   RGU  routed gate/up:  expert slot x 128 gate + 128 up rows x a K part (FP4)
//   SDN  shared down:     128 rows of H x a K part (BF16 or MXFP8)
//   RDN  routed down:     2 x 128 rows of H x one expert slot (FP4, whole
//                         K; both tiles share the slot's h tile)
// Split-K gate/up parts write FP32 partial sums; the block that delivers the
// last part of a tile (an atomic ticket) sums the parts in a fixed order (a
// tile of one part takes them from its registers) and runs the tile's
// epilogue: SwiGLU to BF16 h, or MXFP8 h (shared), or SwiGLU + MXFP4
// requantise (routed).  A routed down unit waits only for its own slot's h.
// Down parts are counted; once all are stored, the weighted combine
// out = BF16(ys + sum_j w_j y_j), summed in a fixed order, runs as items of
// 128 columns x 4 (wide steps 32 or 16) tokens spread over all blocks, their
// rows brought into the idle ring by bulk copies.  Results are therefore
// bit-reproducible run to run.  With the shared expert folded into the FP4
// table, every token has one more slot (the table's last expert, weight 1)
// and there are no SGU / SDN units.
//
// Warp roles: warp 0 issues TMA, warp 1 issues tcgen05.cp / tcgen05.mma,
// warps 2-5 are the epilogue (one TMEM lane = one weight row each).  Before
// their first unit the epilogue warps compute this block's router rows and
// its slice of the MXFP4 quantisation of x; once every block has done so they
// build the routing (top-k, sort by expert) in shared memory and release the
// producer and MMA warps onto the routed units.  Routed weights load with an
// evict-first L2 policy, so the small hand-off data (partials, h, y) stays in
// L2; steps of up to 16 tokens prefetch nothing beyond the stage ring (extra
// traffic measurably slows their latency-bound hand-offs).
//
// Wide steps (17-128 tokens, the W instantiations) keep the 16-row B
// operand: the shared expert runs per 16-token chunk (SGU / SDN units per
// chunk), and the routed experts per slot, a run of at most 16 sorted
// assignments of one expert.  The router runs as split-K items, each block
// computes the top-k of its own tokens and publishes it tagged with the
// launch number, and every block then sorts all T k assignments by expert
// (per-warp histograms and scans) in shared memory.  x is quantised in token
// order while the router parts land and copied into sorted order once the
// routing is known, so a slot's activation rows are one 16-row TMA box; the
// routed gate/up units stream their weight tiles into the ring while they
// wait for it, and the first experts' gate/up weights are prefetched into L2
// during the routing when the step touches about every expert.
//
// Every wait is bounded (MOE_DEV_TIMEOUT in the status word); the last block
// out resets the counters, and each finishing block resets its ticket.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "moefp4.h"
#include "routing.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace moefp4 {
namespace {

// Trace builds (MOEFP4_TRACE=1): each block stamps %globaltimer at its phase
// boundaries of the last launch, read back by moe_debug_decode_trace.
enum DcTraceEvent {
  TR_START = 0,        // the block's TMEM is allocated
  TR_ROUTER = 1,       // router rows or parts (wide steps: and x in token order) done
  TR_ROUTING = 2,      // routing table built
  TR_X = 3,            // x quantised (steps up to 16 tokens) or copied into sorted order (wide steps)
  TR_X_SEEN = 4,       // producer: the quantised x of every block seen (wide steps)
  TR_HSH_SEEN = 5,     // producer: the shared expert's h seen
  TR_H_SEEN = 6,       // producer: every slot's routed h seen
  TR_PRODUCER = 7,     // producer: every copy issued
  TR_UNITS = 8,        // epilogue: every unit of the block done
  TR_DOWN_SEEN = 9,    // epilogue: every down part stored
  TR_END = 10,         // epilogue: combine done
  TR_LAST_UNIT = 11,   // + unit kind: the block's last unit of that kind finished
};
// Per expert slot (the first DC_TRACE_SLOTS): earliest and latest hand-out
// of its routed gate/up units, latest gate/up unit done, h ready, earliest
// and latest hand-out of its down units, latest down unit stored, and
// (expert << 8 | rows).  Earliest times are kept as ~t under atomicMax, so
// that zeroed entries mean "not reached".
enum DcSlotEvent { TS_RGU_FIRST = 0, TS_RGU_LAST, TS_RGU_DONE, TS_H, TS_RDN_FIRST, TS_RDN_LAST, TS_RDN_DONE, TS_INFO };
#if MOEFP4_TRACE
constexpr int DC_TRACE_EVENTS = 16;
constexpr int DC_TRACE_SLOTS = 320;
__device__ unsigned long long g_dc_trace[DC_MAX_GRID][DC_TRACE_EVENTS];
__device__ unsigned long long g_dc_slot_trace[DC_TRACE_SLOTS][8];
#define DC_TRACE(ev) (g_dc_trace[blockIdx.x][(ev)] = globaltimer_ns())
#define DC_SLOT_FIRST(s, ev) \
  ((s) < DC_TRACE_SLOTS ? (void)atomicMax(&g_dc_slot_trace[(s)][(ev)], ~globaltimer_ns()) : (void)0)
#define DC_SLOT_LAST(s, ev) \
  ((s) < DC_TRACE_SLOTS ? (void)atomicMax(&g_dc_slot_trace[(s)][(ev)], globaltimer_ns()) : (void)0)
#define DC_SLOT_SET(s, ev, v) ((s) < DC_TRACE_SLOTS ? (void)(g_dc_slot_trace[(s)][(ev)] = (v)) : (void)0)
#else
#define DC_TRACE(ev) ((void)0)
#define DC_SLOT_FIRST(s, ev) ((void)0)
#define DC_SLOT_LAST(s, ev) ((void)0)
#define DC_SLOT_SET(s, ev, v) ((void)0)
#endif

constexpr int DT = 192;                 // threads: TMA warp, MMA warp, 4 epilogue warps
constexpr int EPI_THREADS = 128;
// A 4-stage ring, of which the host lets `depth` stages be in flight: two
// for a step of up to 15 assignments (its shared units stream while the
// routing is computed, and a deeper queue slows the latency-bound hand-offs),
// four for the larger steps.  Routed down units put up to four of their
// weight stages (of six at I = 1536) into the ring before they wait for
// their slot's h.
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
// Units go round-robin (unit u to block u mod G), or, in steps of up to 16
// tokens whose routed gate/up units fill more than one round of blocks (the
// DYN instantiations), dynamically: each block's first
// unit is blockIdx.x, the later ones come from a launch-wide counter in
// increasing order, and the producer passes them to the MMA and epilogue
// warps through a ring of UQ entries.  Measured on GB300: dynamic 130-133 us
// against 137-141 us round-robin for 16 NVFP4 tokens (the four-versus-three
// gate/up units per block no longer decide the end), but slower for one
// token, for the 16-token small layer and for 128 tokens, where the
// round-robin list is already balanced and the hand-off costs.
constexpr int UQ = 16;
template <bool NV> __host__ __device__ constexpr uint32_t tmem_cols() { return NV ? 512u : 256u; }
constexpr uint32_t TM_SF = 32 * NACC;
// assignments and expert slots of a step (W: wide steps of up to 128 tokens)
template <bool W> __host__ __device__ constexpr int maxn() { return (W ? MAX_WIDE_T : MAX_DECODE_T) * MAX_TOPK; }
template <bool W> __host__ __device__ constexpr int maxslot() {
  return W ? MAX_E + 1 + MAX_WIDE_T * MAX_TOPK / 16 : MAX_DECODE_T * MAX_TOPK;
}
template <bool W> __host__ __device__ constexpr int maxt() { return W ? MAX_WIDE_T : MAX_DECODE_T; }
constexpr int EH = MAX_E + 2;  // per-expert table stride (the table holds up to MAX_E + 1 experts)
constexpr int DC_SDN_MAX = 4;  // shared down parts (dc_splits caps them at 4)

enum UnitKind { U_SGU = 0, U_RGU = 1, U_SDN = 2, U_RDN = 3 };

struct DcArgs {
  int T, H, I, E, k;         // E experts in the table, k assignments per token
  int Er, kr;                // the router's experts and top-k (E - 1, k - 1 with the
                             // shared expert folded into the table as expert Er)
  int G;                     // blocks in the launch
  int s_sgu, s_rgu, s_sdn;   // split-K parts
  int n_sgu, n_sdn;          // unit counts that do not depend on the routing
  int nslot_max;             // slots a step can have (dc_nslot_max)
  int nck;                   // 16-token chunks of the shared expert's units (1 up to 16 tokens)
  int tk_rgu, tk_nv, tk_slot;  // ticket offsets: routed gate/up tiles, NVFP4 per-slot scale blocks,
                               // per-slot counters of finished routed h
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
  unsigned long long* logit64;  // steps of up to 16 tokens: [T, Er] (launch number << 32) | FP32 bits
  uint8_t* xq;               // [T, H/2]; wide steps: [T k, H/2] in sorted-assignment order
  uint8_t* xs_mma;           // [H/128][512] E8M0 (MXFP4) or [H/64][512] UE4M3 (NVFP4); wide steps:
                             // one such set per slot
  int* xshift;               // NVFP4: [16] per-row power of two of the UE4M3 x scales; wide steps: [T k]
  unsigned long long* topk64;  // wide steps: [2][T kr] (launch number << 32) | expert id, | weight bits
  float* rpart;              // wide steps: [H/256][T][Er] router partial sums
  int pf_experts;            // wide steps: experts whose gate/up weights go to L2 during the routing
  int sh8;                   // the shared expert in MXFP8 (E4M3 codes, UE8M0 scales per 32)
  const uint8_t* w13s8_mma;  // its prepared scales: [2I/128][H/128][512 B], [H/128][I/128][512 B]
  const uint8_t* w2s8_mma;
  uint8_t* x8;               // MXFP8 shared expert: x codes [T, H]; scales [16-token chunks][H/128][512 B]
  uint8_t* x8s;
  uint8_t* h8s;              // h's scales [16-token chunks][I/128][512 B] (codes [T, I] in h_shared)
  uint8_t* xq_tok;           // wide steps: [T, H/2] x codes in token order (before the routing)
  uint8_t* xe_tok;           // wide steps: [T, H/32] their E8M0 exponent bytes
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

// Routing of the step, built by the epilogue warps of every block (16-byte
// aligned: before it is built, wide steps stage x in its storage as float4).
template <bool W>
struct __align__(16) DcRouting {
  int ids[maxn<W>()];
  float w[maxn<W>()];
  int inv[maxn<W>()];          // assignment t*k+j -> sorted position
  int tok[maxn<W>()];          // sorted position -> token
  int sorted_e[maxn<W>()];     // sorted position -> expert
  int slot_e[maxslot<W>()];    // slot -> expert (ascending)
  int slot_beg[maxslot<W>() + 1];  // slot -> first sorted position
  int wcount[EPI_THREADS / 32];
  int n_slots;
  // wide steps: per-warp expert histograms (then bases), expert offsets and
  // first slots in the sorted order
  int whist[W ? 4 * EH : 1];
  int eoff[W ? EH : 1];
  int soff[W ? EH : 1];
};

struct Unit {
  int kind;
  int tile;   // 128-row tile: of I (gate/up) or of H (down)
  int part;   // split-K part
  int slot;   // routed units
  int chunk;  // shared units: 16-token chunk
  int st0, st1;
};

__device__ __forceinline__ int units_total(const DcArgs& a, int n_slots) {
  return a.n_sgu + n_slots * (a.I / 128) * a.s_rgu + a.n_sdn + n_slots * (a.H / 256);
}

// Part p of `stages` stages split into s near-equal parts.
__device__ __forceinline__ void part_range(int stages, int s, int p, int& st0, int& st1) {
  st0 = p * stages / s;
  st1 = (p + 1) * stages / s;
}

// v-th shared down unit: 128-row tile of H, K part over stages of two
// chunks, 16-token chunk (the chunks of one tile and part are neighbours in
// the list, so their weight tiles are read from HBM about once).
__device__ __forceinline__ Unit sdn_unit(const DcArgs& a, int v) {
  Unit U{};
  U.kind = U_SDN;
  U.chunk = v % a.nck;
  v /= a.nck;
  U.tile = v / a.s_sdn;
  U.part = v % a.s_sdn;
  part_range((a.I / (a.sh8 ? 128 : 64) + 1) / 2, a.s_sdn, U.part, U.st0, U.st1);
  return U;
}

// v-th routed down unit: a pair of 128-row tiles of H (rows 256 tile ..
// 256 tile + 255) x expert slot, whole K, one 256-element K chunk per stage,
// in slot order (slots finish their gate/up in about that order, and each
// down unit waits only for its own slot's h).  The pair shares one h tile
// per stage, as the gate/up units share their x tile.
__device__ __forceinline__ Unit rdn_unit(const DcArgs& a, int v) {
  Unit U{};
  U.kind = U_RDN;
  U.slot = v / (a.H / 256);
  U.tile = v % (a.H / 256);
  U.st0 = 0;
  U.st1 = a.I / 256;
  return U;
}

__device__ Unit unit_at(const DcArgs& a, int n_slots, int u) {
  Unit U{};
  const int nbI = a.I / 128;
  if (u < a.n_sgu) {
    U.kind = U_SGU;
    U.chunk = u % a.nck;
    u /= a.nck;
    U.tile = u / a.s_sgu;
    U.part = u % a.s_sgu;
    part_range(a.H / (a.sh8 ? 128 : 64), a.s_sgu, U.part, U.st0, U.st1);  // K stages of 128 bytes per row
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
  return rdn_unit(a, u - a.n_sdn);
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
template <int MT>
__device__ void router_row(const DcArgs& a, int e, int et, float (*red_s)[MT], uint32_t epoch) {
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

// Wide steps: the router as split-K items (16-token group g, 256-element K
// part q), so that no block streams more than one group's x.  The epilogue
// warps stage x[16g .. 16g+15][256q .. 256q+255] in shared memory (xs, 16 KB
// as FP32) and thread et computes experts et, et + 128, ... over the part,
// each logit part four FP32 chains of 64 products added pairwise, stored to
// rpart[q][t][e].  Every block counts itself on C_DC_RT once its items are
// stored; the top-k adds a token's parts in q order.
__device__ void router_w(const DcArgs& a, int et, float* xs) {
  const int T = a.T, H = a.H, Er = a.Er, KP = H / 256, items = (T + 15) / 16 * KP;
  for (int item = blockIdx.x; item < items; item += a.G) {
    const int g = item / KP, q = item % KP;
    for (int i = et; i < 16 * 32; i += EPI_THREADS) {  // 16 rows x 32 groups of 8 BF16
      const int r = i >> 5, c = i & 31, t = 16 * g + r;
      const uint4 v = t < T ? __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * H + 256 * q) + c)
                            : make_uint4(0, 0, 0, 0);
      float4* d = reinterpret_cast<float4*>(xs + r * 256 + 8 * c);
      d[0] = make_float4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y));
      d[1] = make_float4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w));
    }
    epi_sync();
    for (int e = et; e < Er; e += EPI_THREADS) {
      // four FP32 chains per token (k = 0, 1, 2, 3 mod 4), 64 products each,
      // added pairwise at the end: the accuracy of the batched router's
      // 128-element chains or better
      float4 acc[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) acc[t] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      const float4* wrow = reinterpret_cast<const float4*>(a.wr + (size_t)e * H + 256 * q);
#pragma unroll 1
      for (int k0 = 0; k0 < 64; k0 += 16) {
        float4 wv[16];  // 64 weights in flight, then 16 tokens x 64 FMAs
#pragma unroll
        for (int j = 0; j < 16; ++j) wv[j] = __ldg(wrow + k0 + j);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const float4 xv = *reinterpret_cast<const float4*>(xs + t * 256 + 4 * (k0 + j));
            acc[t].x = fmaf(xv.x, wv[j].x, acc[t].x);
            acc[t].y = fmaf(xv.y, wv[j].y, acc[t].y);
            acc[t].z = fmaf(xv.z, wv[j].z, acc[t].z);
            acc[t].w = fmaf(xv.w, wv[j].w, acc[t].w);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < 16; ++t)
        if (16 * g + t < T)
          a.rpart[((size_t)q * T + 16 * g + t) * Er + e] = (acc[t].x + acc[t].y) + (acc[t].z + acc[t].w);
    }
    epi_sync();  // xs is restaged by the next item
  }
  if (et == 0) red_release_add(a.ctr + C_DC_RT, 1);  // after the barrier: every thread's parts
}

// Wide steps: token t's logits to lg[e] (thread et: experts et, et + 128),
// the parts added in q order (up to 32 parts' loads in flight), the softmax
// bias added last.
__device__ void logits_w(const DcArgs& a, int t, int et, float* lg) {
  const int KP = a.H / 256;
  const size_t stride = (size_t)a.T * a.Er;
  for (int e = et; e < a.Er; e += EPI_THREADS) {
    const float* src = a.rpart + (size_t)t * a.Er + e;
    float v = 0.0f;
    for (int q0 = 0; q0 < KP; q0 += 32) {
      float p[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) p[q] = q0 + q < KP ? __ldcg(src + (q0 + q) * stride) : 0.0f;
#pragma unroll
      for (int q = 0; q < 32; ++q)
        if (q0 + q < KP) v += p[q];
    }
    if (a.bias && a.score == SCORE_SOFTMAX) v += __ldg(a.bias + e);
    lg[e] = v;
  }
}


// MXFP8 codes of one 32-element BF16 block (32 bytes to dq) and its E8M0
// byte, the rule of the standalone MXFP8 quantiser.
__device__ __forceinline__ uint8_t quant32_mx8(const uint16_t* xb, uint8_t* dq) {
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
  const int ex = mx8_scale_exp(amax);
  const float inv = pow2_neg(ex);
#pragma unroll 1
  for (int j = 0; j < 4; ++j) {
    const float v[8] = {bf16_lo(raw[j].x), bf16_hi(raw[j].x), bf16_lo(raw[j].y), bf16_hi(raw[j].y),
                        bf16_lo(raw[j].z), bf16_hi(raw[j].z), bf16_lo(raw[j].w), bf16_hi(raw[j].w)};
    reinterpret_cast<uint2*>(dq)[j] = e4m3x8_rne(v, inv);
  }
  return (uint8_t)(ex + 127);
}

// MXFP8 shared expert: x to x8 (token rows, 32-element block per item) and
// its scale bytes in the MMA layout of the 16-row B tiles, [chunk][H/128]
// [512 B], row t % 16; the rows past T of the last chunk get zero scales.
__device__ void quant_x8(const DcArgs& a, int et) {
  const int nb = a.H / 32, rows = 16 * a.nck;
  for (int i = blockIdx.x * EPI_THREADS + et; i < rows * nb; i += a.G * EPI_THREADS) {
    const int t = i / nb, b = i % nb;
    uint8_t sb = 0;
    if (t < a.T) sb = quant32_mx8(a.x + (size_t)t * a.H + b * 32, a.x8 + (size_t)t * a.H + b * 32);
    a.x8s[((size_t)(t >> 4) * (a.H / 128) + b / 4) * 512 + (t & 15) * 16 + (b % 4)] = sb;
  }
}

// MXFP4 quantisation of one 32-element block i = (token row t < 16, block b
// of H/32): 16 code bytes of xq and byte b % 4 of the MMA-layout scale word
// of row t in group b / 4 (word 4t of that group's 512-byte block).  Rows
// t >= T get a zero scale byte.
__device__ void quant_block(const DcArgs& a, int i) {
  const int nb = a.H / 32;
  const int t = i / nb, b = i % nb;
  uint8_t sb = 0;
  if (t < a.T) sb = quant32(a.x + (size_t)t * a.H + b * 32, a.xq + (size_t)t * (a.H / 2) + b * 16);
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

// NVFP4 experts: one warp quantises token row t to MXFP4 (the same codes and
// E8M0 exponents as the standalone quantiser), the codes to xrow, and writes
// row `row` of the scale blocks at xs for the UE4M3 MMA: each 32-block's 2^e
// twice (two 16-blocks) as 2^(e - c_t), c_t = (largest e of the row) - 8, and
// c_t to *shift; the epilogue multiplies the row's products by 2^c_t.  A
// block more than 2^17 below the row's largest block scale falls under
// UE4M3's range and is dropped.  Lane l takes blocks l, l+32, ... in batches
// of 4 with all their loads in flight; the exponents wait in e_s (H <= 8192).
__device__ void quant_row_nv_to(const DcArgs& a, int t, uint8_t* xrow, uint8_t* xs, int row, int* shift,
                                uint8_t* e_s, uint8_t* e8_out = nullptr) {
  const int lane = threadIdx.x & 31, nb = a.H / 32;
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
      uint32_t* dst = reinterpret_cast<uint32_t*>(xrow + b * 16);
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
      if (e8_out) e8_out[b] = (uint8_t)(ex + 127);
      emax = max(emax, ex);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) emax = max(emax, __shfl_xor_sync(FULL, emax, o));
  const int c = emax - 8;
  if (lane == 0) *shift = c;
  __syncwarp();
  if (!xs) return;
  // bytes 2(b&1), 2(b&1)+1 of the word of the row in 64-element chunk b/2
  for (int b = lane; b < nb; b += 32) {
    const uint32_t u = ue4m3_pow2((int)e_s[b] - 127 - c);
    *reinterpret_cast<uint16_t*>(xs + (size_t)(b / 2) * 512 + row * 16 + 2 * (b & 1)) = (uint16_t)(u | (u << 8));
  }
}

// Token row t < 16 of a step of up to 16 tokens (rows t >= T get zero scale
// words).
__device__ void quant_row_nv(const DcArgs& a, int t, uint8_t* e_s) {
  const int lane = threadIdx.x & 31;
  if (t >= a.T) {
    for (int kb = lane; kb < a.H / 64; kb += 32) *reinterpret_cast<uint32_t*>(a.xs_mma + (size_t)kb * 512 + t * 16) = 0u;
    return;
  }
  quant_row_nv_to(a, t, a.xq + (size_t)t * (a.H / 2), a.xs_mma, t, a.xshift + t, e_s);
}

// Wide steps, before the routing: x in token order, MXFP4 codes to xq_tok and
// E8M0 bytes to xe_tok (NVFP4 also the row shift c_t to xshift[t]); the
// epilogue warps of every block take a share while the router parts land.
template <bool NV>
__device__ void quant_tokens_w(const DcArgs& a, int et, uint8_t* e_s) {
  const int T = a.T, H = a.H, nb = H / 32;
  if (NV) {
    for (int t = blockIdx.x * (EPI_THREADS / 32) + (et >> 5); t < T; t += a.G * (EPI_THREADS / 32))
      quant_row_nv_to(a, t, a.xq_tok + (size_t)t * (H / 2), nullptr, 0, a.xshift + t, e_s, a.xe_tok + (size_t)t * nb);
  } else {
    for (int i = blockIdx.x * EPI_THREADS + et; i < T * nb; i += a.G * EPI_THREADS)
      a.xe_tok[i] = quant32(a.x + (size_t)i * 32, a.xq_tok + (size_t)i * 16);
  }
}

// Wide steps, after the routing: item i = (sorted row p, 32-element block b)
// copies token tok[p]'s 16 code bytes to xq row p and writes its scale into
// row c (p's row in its slot) of the slot's MMA-layout scale blocks: the
// E8M0 byte (MXFP4), or the UE4M3 pair 2^(e - c_t) (NVFP4).  The slot's first
// row also zeroes the scale words of the rows the slot leaves empty (its B
// tile's other rows belong to the next slot or lie past T k).
template <bool NV>
__device__ void sort_x_w(const DcArgs& a, const DcRouting<true>& R, int i) {
  const int H = a.H, nb = H / 32;
  const int p = i / nb, b = i % nb;
  const int e = R.sorted_e[p], r = p - R.eoff[e];
  const int slot = R.soff[e] + (r >> 4), c = r & 15, t = R.tok[p];
  *reinterpret_cast<uint4*>(a.xq + (size_t)p * (H / 2) + b * 16) =
      __ldcg(reinterpret_cast<const uint4*>(a.xq_tok + (size_t)t * (H / 2) + b * 16));
  const int e8 = __ldcg(a.xe_tok + (size_t)t * nb + b);
  const int cnt = imin(16, R.eoff[e + 1] - (p - c));
  if (NV) {
    uint8_t* blk = a.xs_mma + ((size_t)slot * (H / 64) + b / 2) * 512;
    const uint32_t u = ue4m3_pow2(e8 - 127 - __ldcg(a.xshift + t));
    *reinterpret_cast<uint16_t*>(blk + c * 16 + 2 * (b & 1)) = (uint16_t)(u | (u << 8));
    if (c == 0 && (b & 1) == 0)
      for (int rr = cnt; rr < 16; ++rr) *reinterpret_cast<uint32_t*>(blk + rr * 16) = 0u;
  } else {
    uint8_t* blk = a.xs_mma + ((size_t)slot * (H / 128) + b / 4) * 512 + (b % 4);
    blk[c * 16] = (uint8_t)e8;
    if (c == 0)
      for (int rr = cnt; rr < 16; ++rr) blk[rr * 16] = 0;
  }
}

// Token t's top-k (lane j holds choice j) published with the launch number in
// the high word: [T kr] ids, then [T kr] weights.
__device__ __forceinline__ void publish_topk(const DcArgs& a, int t, const int (&sel)[MAX_TOPK],
                                             const float (&wt)[MAX_TOPK], uint32_t epoch) {
  const int lane = threadIdx.x & 31, kr = a.kr, nr = a.T * kr;
#pragma unroll
  for (int j = 0; j < MAX_TOPK; ++j)
    if (j == lane && j < kr) {
      st_relaxed_u64(a.topk64 + t * kr + j, ((unsigned long long)epoch << 32) | (uint32_t)sel[j]);
      st_relaxed_u64(a.topk64 + nr + t * kr + j, ((unsigned long long)epoch << 32) | __float_as_uint(wt[j]));
    }
}

// Every token's published top-k into R.ids / R.w (bounded wait for this
// launch's number), plus the folded shared expert (expert Er, weight 1).
template <bool W>
__device__ void gather_topk(const DcArgs& a, DcRouting<W>& R, int et, uint32_t epoch, int* failed) {
  const int T = a.T, k = a.k, kr = a.kr, nr = T * kr;
  const uint64_t t0 = globaltimer_ns();
  for (int i = et; i < nr; i += EPI_THREADS) {
    unsigned long long vi = 0, vw = 0;
    for (uint32_t it = 0;; ++it) {
      vi = ld_relaxed_u64(a.topk64 + i);
      vw = ld_relaxed_u64(a.topk64 + nr + i);
      if ((uint32_t)(vi >> 32) == epoch && (uint32_t)(vw >> 32) == epoch) break;
      if (globaltimer_ns() - t0 > a.limit_ns || it > (1u << 26)) {
        *failed = 1;
        vi = 0;
        break;
      }
      __nanosleep(64);
    }
    const int t = i / kr, j = i % kr;
    const int id = (int)(uint32_t)vi;
    R.ids[t * k + j] = id >= 0 && id < a.Er ? id : 0;  // a failed wait leaves a valid index
    R.w[t * k + j] = __uint_as_float((uint32_t)vw);
  }
  if (kr < k)  // the shared expert folded into the table: expert Er, weight 1
    for (int t = et; t < T; t += EPI_THREADS) {
      R.ids[t * k + kr] = a.Er;
      R.w[t * k + kr] = 1.0f;
    }
}

// Top-k of every token (one epilogue warp per token), then the stable sort
// of the T*k <= 128 assignments by expert (each assignment counts the ones
// that precede it) and the distinct-expert slots (runs of one expert in the
// sorted order, numbered with a ballot).  128 epilogue threads, et = 0..127.
// *failed is set (by some thread) when a logit row never arrived.
__device__ void build_routing(const DcArgs& a, DcRouting<false>& R, int et, uint32_t epoch, int* failed) {
  const int T = a.T, k = a.k, kr = a.kr, n = T * k;
  const int w = et >> 5, lane = et & 31;
  // Up to 4 tokens every block picks them itself (one token per warp).  More
  // tokens would queue on the warps: block b picks tokens b, b + G, ... (warp 0) and
  // publishes it, and every block gathers them (one more round trip instead
  // of up to four top-k passes in a row).
  const bool spread = T > EPI_THREADS / 32;
  for (int t = spread ? (w == 0 ? (int)blockIdx.x : T) : w; t < T; t += spread ? a.G : EPI_THREADS / 32) {
    float v[8];
    if (!wait_logit_row(a, t, epoch, v)) {
      if (lane == 0) *failed = 1;
      continue;
    }
    int sel[MAX_TOPK];
    float wt[MAX_TOPK];
    route_row(v, a.Er, kr, a.score, a.bias, sel, wt);
    if (spread) {
      publish_topk(a, t, sel, wt, epoch);
      continue;
    }
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
  if (spread) gather_topk(a, R, et, epoch, failed);
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

// Wide steps (T k <= 1024 assignments).  Once every block's router parts are
// in, each block takes tokens blockIdx.x + G i one at a time: its epilogue
// threads add the token's logit parts, warp 0 picks the top-k and publishes
// it with the launch number in the high word, so a reader that sees the
// number has the value; every
// block then reads all T kr entries (bounded wait), adds the folded shared
// expert, and sorts the assignments by expert, stably: warp w counts its
// contiguous quarter of the assignments per expert (__match_any_sync), one
// warp scans the counts into expert offsets, per-warp bases and first slots,
// and each warp places its quarter.  Slot s is a run of at most 16 sorted
// positions of one expert; an expert's runs are consecutive slots.
__device__ void build_routing_w(const DcArgs& a, DcRouting<true>& R, int et, uint32_t epoch, int* failed) {
  const int T = a.T, k = a.k, kr = a.kr, n = T * k, E = a.E;
  const int w = et >> 5, lane = et & 31;
  if ((int)blockIdx.x < T) {  // this block has tokens: every block's router parts must be in
    if (et == 0 && !wait_at_least(a.ctr + C_DC_RT, a.G, a.ctr + C_STATUS, a.limit_ns)) *failed = 1;
    epi_sync();
  }
  float* lg = reinterpret_cast<float*>(R.sorted_e);  // a token's logits (the sort comes later)
  for (int t = blockIdx.x; t < T && !*failed; t += a.G) {
    logits_w(a, t, et, lg);
    epi_sync();
    if (w != 0) {
      epi_sync();
      continue;
    }
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = lane + 32 * i < a.Er ? lg[lane + 32 * i] : 0.0f;
    int sel[MAX_TOPK];
    float wt[MAX_TOPK];
    route_row(v, a.Er, kr, a.score, a.bias, sel, wt);
    publish_topk(a, t, sel, wt, epoch);
    epi_sync();  // lg is rewritten for the next token
  }
  gather_topk(a, R, et, epoch, failed);
  int* wh = R.whist + w * EH;
  for (int e = lane; e < E; e += 32) wh[e] = 0;
  epi_sync();
  if (*failed) return;  // the same answer in every thread after the barrier
  const int per = (n + 3) / 4, lo = imin(n, w * per), hi = imin(n, lo + per);
  for (int i0 = lo; i0 < hi; i0 += 32) {
    const int i = i0 + lane;
    const int e = i < hi ? R.ids[i] : -1;
    const unsigned peers = __match_any_sync(FULL, e);
    if (e >= 0 && lane == __ffs(peers) - 1) wh[e] += __popc(peers);
    __syncwarp();
  }
  epi_sync();
  if (w == 0) {
    constexpr int EPL = (EH + 31) / 32;  // experts per lane
    int cnt[EPL], tot = 0, stot = 0;
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
      const int e = lane * EPL + q;
      int c = 0;
      if (e < E)
        for (int ww = 0; ww < EPI_THREADS / 32; ++ww) c += R.whist[ww * EH + e];
      cnt[q] = c;
      tot += c;
      stot += (c + 15) >> 4;
    }
    int it = tot, is = stot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x1 = __shfl_up_sync(FULL, it, o), x2 = __shfl_up_sync(FULL, is, o);
      if (lane >= o) {
        it += x1;
        is += x2;
      }
    }
    int eo = it - tot, so = is - stot;
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
      const int e = lane * EPL + q;
      if (e < E) {
        R.eoff[e] = eo;
        R.soff[e] = so;
        int b = eo;
        for (int ww = 0; ww < EPI_THREADS / 32; ++ww) {
          const int c = R.whist[ww * EH + e];
          R.whist[ww * EH + e] = b;
          b += c;
        }
      }
      eo += cnt[q];
      so += (cnt[q] + 15) >> 4;
    }
    if (lane == 31) {
      R.eoff[E] = eo;
      R.soff[E] = so;
      R.n_slots = so;
    }
  }
  epi_sync();
  for (int i0 = lo; i0 < hi; i0 += 32) {
    const int i = i0 + lane;
    const int e = i < hi ? R.ids[i] : -1;
    const unsigned peers = __match_any_sync(FULL, e);
    const int pos = e >= 0 ? wh[e] + __popc(peers & ((1u << lane) - 1u)) : 0;
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wh[e] += __popc(peers);
    __syncwarp();
    if (e >= 0) {
      R.inv[i] = pos;
      R.tok[pos] = i / k;
      R.sorted_e[pos] = e;
    }
  }
  epi_sync();
  for (int p = et; p < n; p += EPI_THREADS) {
    const int e = R.sorted_e[p], r = p - R.eoff[e];
    if ((r & 15) == 0) {
      R.slot_e[R.soff[e] + (r >> 4)] = e;
      R.slot_beg[R.soff[e] + (r >> 4)] = p;
    }
  }
  if (et == 0) R.slot_beg[R.n_slots] = n;
  epi_sync();
}

// Halves of a stage that a unit uses: gate/up and routed down units one K
// chunk (two weight tiles, one activation tile), shared down units two K
// chunks (the second may be past the end of K).
__device__ __forceinline__ int stage_halves(const DcArgs& a, const Unit& U, int st) {
  if (U.kind == U_SDN) return 2 * st + 1 < a.I / (a.sh8 ? 128 : 64) ? 2 : 1;
  return 2;
}

// Scale bytes per 128 rows and 256-element K chunk.
template <bool NV> __device__ __forceinline__ constexpr uint32_t sf_chunk() { return 512u * nblk<NV>(); }

// Bytes one stage of a unit brings in (the mbarrier transaction count).
template <bool NV>
__device__ __forceinline__ uint32_t stage_tx(const DcArgs& a, const Unit& U, int st) {
  const uint32_t h = stage_halves(a, U, st);
  switch (U.kind) {
    case U_SGU: return 2 * A_TILE + B_TILE + (a.sh8 ? 3 * 512 : 0);
    case U_SDN: return h * (A_TILE + B_TILE + (a.sh8 ? 2 * 512 : 0));
    default: return 2 * A_TILE + B_TILE + 3 * sf_chunk<NV>();  // routed gate/up and down
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
    if (a.sh8) {  // the gate and up tiles' scale blocks for this 128-element K chunk
      const size_t kb = a.H / 128;
      tc::bulk_load(sp + ST_SFA, a.w13s8_mma + ((size_t)U.tile * kb + st) * 512, 512, fb);
      tc::bulk_load(sp + ST_SFA + 512, a.w13s8_mma + ((size_t)(nbI + U.tile) * kb + st) * 512, 512, fb);
    }
  } else if (U.kind == U_RGU) {
    const int row = e * 2 * a.I + 128 * U.tile;
    const uint32_t sfc = sf_chunk<NV>();
    const size_t bpr = (size_t)a.H / 256 * (sfc / 512);  // scale blocks per 128-row tile
    const size_t rt = (size_t)e * (2 * nbI) + U.tile;    // gate row tile; the up tile is nbI further
    const uint64_t pol = tc::l2_evict_first();  // routed weights are read once per step
    tc::tma_load_2d_hint(sp + ST_A0, &m.w13r, st * 128, row, fb, pol);
    tc::tma_load_2d_hint(sp + ST_A1, &m.w13r, st * 128, row + a.I, fb, pol);
    tc::bulk_load_hint(sp + ST_SFA, a.w13s_mma + rt * bpr * 512 + (size_t)st * sfc, sfc, fb, pol);
    tc::bulk_load_hint(sp + ST_SFA + sfc, a.w13s_mma + (rt + nbI) * bpr * 512 + (size_t)st * sfc, sfc, fb, pol);
  } else if (U.kind == U_SDN) {
    const int halves = stage_halves(a, U, st);
    for (int h = 0; h < halves; ++h)
      tc::tma_load_2d(sp + (h ? ST_A1 : ST_A0), &m.w2s, (2 * st + h) * 128, 128 * U.tile, fb);
    if (a.sh8)
      tc::bulk_load(sp + ST_SFA, a.w2s8_mma + ((size_t)U.tile * (a.I / 128) + 2 * st) * 512, halves * 512, fb);
  } else {  // routed down: two 128-row tiles of H, one K chunk
    const uint64_t pol = tc::l2_evict_first();
    const int row = e * a.H + 256 * U.tile;
    tc::tma_load_2d_hint(sp + ST_A0, &m.w2r, st * 128, row, fb, pol);
    tc::tma_load_2d_hint(sp + ST_A1, &m.w2r, st * 128, row + 128, fb, pol);
    const uint32_t sfc = sf_chunk<NV>();
    const size_t bpr = (size_t)a.I / 256 * (sfc / 512);
    const size_t rt = (size_t)e * nbH + 2 * U.tile;
    tc::bulk_load_hint(sp + ST_SFA, a.w2s_mma + rt * bpr * 512 + (size_t)st * sfc, sfc, fb, pol);
    tc::bulk_load_hint(sp + ST_SFA + sfc, a.w2s_mma + (rt + 1) * bpr * 512 + (size_t)st * sfc, sfc, fb, pol);
  }
}

// TMA / bulk copies of the activation tiles (and their scales) of stage st.
// Shared units take the 16 token rows of their chunk; routed gate/up units
// every token row (steps of up to 16 tokens) or their slot's 16 sorted rows
// (wide steps).
template <bool NV, bool W>
__device__ __forceinline__ void issue_acts(const DcArgs& a, const DcMaps& m, const Unit& U, int st, int beg,
                                           uint8_t* sp, uint64_t* fb) {
  if (U.kind == U_SGU) {
    tc::tma_load_2d(sp + ST_B0, &m.x, st * 128, 16 * U.chunk, fb);
    if (a.sh8) tc::bulk_load(sp + st_sfb<NV>(), a.x8s + ((size_t)U.chunk * (a.H / 128) + st) * 512, 512, fb);
  } else if (U.kind == U_RGU) {
    tc::tma_load_2d(sp + ST_B0, &m.xq, st * 128, W ? beg : 0, fb);
    const size_t set = W ? (size_t)U.slot * (a.H / 256) * sf_chunk<NV>() : 0;  // the slot's scale blocks
    tc::bulk_load(sp + st_sfb<NV>(), a.xs_mma + set + (size_t)st * sf_chunk<NV>(), sf_chunk<NV>(), fb);
  } else if (U.kind == U_SDN) {
    const int halves = stage_halves(a, U, st);
    for (int h = 0; h < halves; ++h)
      tc::tma_load_2d(sp + (h ? ST_B1 : ST_B0), &m.hsh, (2 * st + h) * 128, 16 * U.chunk, fb);
    if (a.sh8)
      tc::bulk_load(sp + st_sfb<NV>(), a.h8s + ((size_t)U.chunk * (a.I / 128) + 2 * st) * 512, halves * 512, fb);
  } else {
    const size_t bpr = (size_t)a.I / 256 * nblk<NV>();  // scale blocks of one slot
    tc::tma_load_2d(sp + ST_B0, &m.hq, st * 128, beg, fb);
    tc::bulk_load(sp + st_sfb<NV>(), a.hs_mma + (size_t)U.slot * bpr * 512 + (size_t)st * sf_chunk<NV>(),
                  sf_chunk<NV>(), fb);
  }
}

// Row shift c of sorted h row p (NVFP4), final once every routed h tile is done.
__device__ __forceinline__ int h_row_shift(const DcArgs& a, int p);

// NVFP4: the UE4M3 scale blocks of slot s's h rows (sorted positions beg ..
// beg+cnt-1) for the down MMA, [I/64][512 B], from their E8M0 bytes and the
// row shift 2^c (c = the row's largest exponent - 8).  128 threads; thread
// et writes word et of every block (row et/4 when et % 4 == 0, else zero).
// A row's bytes (I/32, a multiple of 8) are loaded 64 at a time by eight
// 8-byte loads in flight together: one round trip, not one per block.
__device__ void convert_h_scales_nv(const DcArgs& a, int slot, int beg, int cnt, int et) {
  const int nb = a.I / 32, ng = a.I / 64, r = et >> 2;
  const bool real = (et & 3) == 0 && r < cnt;
  const uint2* hsr = reinterpret_cast<const uint2*>(a.hsc + (size_t)(beg + (real ? r : 0)) * nb);
  uint32_t* dst = reinterpret_cast<uint32_t*>(a.hs_mma) + (size_t)slot * ng * 128 + et;
  int c = 0;
  for (int g0 = 0; g0 < ng; g0 += 32) {  // blocks g0 .. g0 + 31: bytes 2 g0 .. 2 g0 + 63
    uint2 b[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) b[j] = real && 2 * g0 + 8 * j < nb ? __ldcg(hsr + g0 / 4 + j) : make_uint2(0, 0);
    if (g0 == 0 && real) c = h_row_shift(a, beg + r);  // after the first bytes' loads: both in flight
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (g0 + j < ng) {
        uint32_t word = 0;
        if (real) {
          // block g0 + j: bytes 2j and 2j + 1 of the chunk
          const uint32_t w32 = (j & 2) ? b[j / 4].y : b[j / 4].x;
          const int sh = 16 * (j & 1);
          const uint32_t u0 = ue4m3_pow2((int)((w32 >> sh) & 0xffu) - 127 - c);
          const uint32_t u1 = ue4m3_pow2((int)((w32 >> (sh + 8)) & 0xffu) - 127 - c);
          word = u0 | (u0 << 8) | (u1 << 16) | (u1 << 24);
        }
        dst[(size_t)(g0 + j) * 128] = word;
      }
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

template <bool NV, bool W, bool DYN>
__global__ void __launch_bounds__(DT, 1) k_decode_tc(const __grid_constant__ DcMaps maps, const DcArgs a) {
  constexpr uint32_t STAGE_BYTES = stage_bytes<NV>();
  constexpr uint32_t ST_SFB = st_sfb<NV>();
  constexpr int NB = nblk<NV>();
  extern __shared__ __align__(1024) uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[DSTAGES], empty[DSTAGES], acc_full[NACC], acc_empty[NACC], drain, routing_ready, comb;
  __shared__ uint64_t uq_full[DYN ? UQ : 1], uq_empty[DYN ? UQ : 1];
  __shared__ int s_uq[DYN ? UQ : 1], s_unit[2];
  __shared__ int never_s;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag, s_ok, s_last, s_fail;
  __shared__ uint32_t s_epoch;
  __shared__ DcRouting<W> R;
  static_assert(!W || sizeof(DcRouting<W>) >= 16 * 256 * sizeof(float), "the wide router stages x in R");
  static_assert(alignof(DcRouting<W>) >= 16, "float4 accesses to the staged x");
  __shared__ float red_s[EPI_THREADS / 32][MAX_DECODE_T];
  __shared__ __align__(4) uint8_t s_hsb[MAX_DECODE_T * 4];
  __shared__ int s_rows[MAX_DECODE_T];  // NVFP4: the current slot's per-row exponent shifts
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
    tc::mbar_init(&comb, 1);
    if (DYN)
      for (int q = 0; q < UQ; ++q) {
        tc::mbar_init(&uq_full[q], 1);
        tc::mbar_init(&uq_empty[q], 2);  // the MMA issuer and epilogue thread 0
      }
    never_s = 0;
    tc::mbar_fence_init();
    abort_flag = 0;
    s_fail = 0;
    // Launch number: never 0 (the tag of zero-filled words), so after 2^32
    // launches it skips from 0xFFFFFFFF to 1.
    const uint32_t ep = (uint32_t)ld_acquire(a.ctr + C_DC_EPOCH) + 1u;
    s_epoch = ep == 0u ? 1u : ep;
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, tmem_cols<NV>());
  if (threadIdx.x == 0) DC_TRACE(TR_START);
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
      // Stage gi may be issued once stage gi - d is consumed (d <= DSTAGES:
      // consumption in order, so slot gi % DSTAGES is free then).
      auto claim = [&](int d) -> bool {
        if (gi < (uint32_t)d) return true;
        const uint32_t j = gi - (uint32_t)d;
        return tc::mbar_wait(&empty[j % DSTAGES], (j / DSTAGES) & 1, a.limit_ns, &abort_flag);
      };
      int n_slots = -1;
      bool hsh_ok = false, xr_ok = false, all_h = false, x8_ok = false;
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
      if (W && a.pf_experts > 0) {
        // A wide step that touches about every expert: while the routing is
        // computed (HBM is otherwise nearly idle then), the gate/up weights
        // and scales of the first experts go to L2, so the first routed
        // units (slots in ascending expert order) start from L2.
        const int kb = a.H / 256, nbox = (2 * a.I / 128) * kb;  // 128-row x 128-byte boxes per expert
        for (int b = blockIdx.x; b < a.pf_experts * nbox; b += a.G) {
          const int e = b / nbox, r = b % nbox;
          tc::tma_prefetch_2d(&maps.w13r, (r % kb) * 128, e * 2 * a.I + 128 * (r / kb));
        }
        const size_t sbytes = (size_t)a.pf_experts * 2 * a.I * (a.H / (NV ? 16 : 32));
        for (size_t o = (size_t)blockIdx.x * 16384; o < sbytes; o += (size_t)a.G * 16384)
          tc::bulk_prefetch_l2(a.w13s_mma + o, (uint32_t)(sbytes - o < 16384 ? sbytes - o : 16384));
      }
      int u = blockIdx.x;
      for (int i = 0;; ++i) {
        if (u >= a.n_sgu && n_slots < 0) {
          if (!tc::mbar_wait(&routing_ready, 0, a.limit_ns, &abort_flag)) { fail(); break; }
          n_slots = R.n_slots;
          // x was quantised by plain stores of other blocks (wide steps: a
          // dependency of the routed gate/up units, below)
          if (!W) {
            if (!wait_at_least(a.ctr + C_DC_READY, a.G, status, a.limit_ns)) { fail(); break; }
            tc::fence_proxy_async_global();
          }
        }
        const bool done = u >= units_total(a, n_slots < 0 ? 0 : n_slots);
        if constexpr (DYN) {  // hand the unit number (or the end, -1) to the MMA and epilogue warps
          const int q = i % UQ;
          if (i >= UQ && !tc::mbar_wait(&uq_empty[q], (i / UQ - 1) & 1, a.limit_ns, &abort_flag)) { fail(); break; }
          s_uq[q] = done ? -1 : u;
          tc::mbar_arrive(&uq_full[q]);
        }
        if (done) break;
        // the next unit's number (dynamic: read while this unit's copies are issued)
        const int next = DYN ? a.G + atomicAdd(a.ctr + C_DC_QUEUE, 1) : u + a.G;
        const Unit U = unit_at(a, n_slots < 0 ? 0 : n_slots, u);
        const int ud = U.kind == U_RDN ? DSTAGES : a.depth;
        int e = 0, beg = 0;
        if (U.kind == U_RGU || U.kind == U_RDN) {
          e = R.slot_e[U.slot];
          beg = R.slot_beg[U.slot];
          DC_SLOT_FIRST(U.slot, U.kind == U_RGU ? TS_RGU_FIRST : TS_RDN_FIRST);
          DC_SLOT_LAST(U.slot, U.kind == U_RGU ? TS_RGU_LAST : TS_RDN_LAST);
        }
        // Down units read h that other blocks write (and, in wide steps,
        // routed gate/up units the sorted x rows).  While it is not there
        // yet, the unit's weight tiles already go into the ring (up to its
        // depth); their activation tiles follow once the dependency is met.
        int npre = 0;
        uint32_t pre_stage[DSTAGES];
        const bool dep_sdn = U.kind == U_SDN && !hsh_ok, dep_rdn = U.kind == U_RDN && !all_h;
        const bool dep_rgu = W && U.kind == U_RGU && !xr_ok;
        const bool dep_sgu = U.kind == U_SGU && a.sh8 && !x8_ok;
        if (dep_sdn || dep_rdn || dep_rgu || dep_sgu) {
          // every slot's h finished (relaxed load, read with the unit's own
          // dependency below): later down units need no check at all
          const int h_done = dep_rdn ? ld_relaxed(a.ctr + C_DC_HR) : 0;
          int* cnt = dep_sdn ? a.ctr + C_DC_HSH
                     : dep_rdn ? a.tickets + a.tk_slot + U.slot
                     : dep_rgu ? a.ctr + C_DC_READY
                               : a.ctr + C_DC_X8;
          const int target = dep_sdn ? nbI * a.nck : dep_rdn ? (NV ? 1 : nbI) : a.G;
          // a routed down unit's weights go into the ring before its slot's
          // counter is read, so that load overlaps the weight copies
          if (dep_rdn || ld_acquire(cnt) < target) {
            npre = imin(U.st1 - U.st0, ud);
            bool ok = true;
            for (int j = 0; j < npre; ++j) {
              if (!claim(ud)) { fail(); ok = false; break; }
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
          if (dep_sdn) {
            hsh_ok = true;
            DC_TRACE(TR_HSH_SEEN);
          } else if (dep_rgu) {
            xr_ok = true;
            DC_TRACE(TR_X_SEEN);
          } else if (dep_sgu) {
            x8_ok = true;
          } else if (h_done >= (NV ? n_slots : n_slots * nbI)) {
            __threadfence();  // with the relaxed load above: acquires every slot's h
            all_h = true;
            DC_TRACE(TR_H_SEEN);
          }
          tc::fence_proxy_async_global();
        }
        for (int j = 0; j < npre; ++j)
          issue_acts<NV, W>(a, maps, U, U.st0 + j, beg, dsm + pre_stage[j] * STAGE_BYTES, &full[pre_stage[j]]);
        bool ok = true;
        for (int st = U.st0 + npre; st < U.st1; ++st) {
          if (!claim(ud)) { fail(); ok = false; break; }
          uint8_t* sp = dsm + stage * STAGE_BYTES;
          tc::mbar_expect_tx(&full[stage], stage_tx<NV>(a, U, st));
          issue_weights<NV>(a, maps, U, st, e, sp, &full[stage]);
          issue_acts<NV, W>(a, maps, U, st, beg, sp, &full[stage]);
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          ++gi;
          if (++stage == DSTAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        u = next;
      }
      DC_TRACE(TR_PRODUCER);
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
      int n_slots = -1;
      for (int i = 0;; ++i) {
        int u = blockIdx.x + i * a.G;
        if constexpr (DYN) {
          const int q = i % UQ;
          if (!tc::mbar_wait(&uq_full[q], (i / UQ) & 1, a.limit_ns, &abort_flag)) { fail(); break; }
          u = s_uq[q];
          tc::mbar_arrive(&uq_empty[q]);
          if (u < 0) break;
        }
        if (u >= a.n_sgu && n_slots < 0) {
          if (!tc::mbar_wait(&routing_ready, 0, a.limit_ns, &abort_flag)) { fail(); break; }
          n_slots = R.n_slots;
        }
        if (!DYN && u >= units_total(a, n_slots < 0 ? 0 : n_slots)) break;
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
          if (U.kind == U_SGU && a.sh8) {
            // MXFP8: 128 K per stage, an MMA of K = 32 reads scale byte kk
            tc::sf_copy(tsf, tc::desc_sf(sa + ST_SFA));
            tc::sf_copy(tsf + 4, tc::desc_sf(sa + ST_SFA + 512));
            tc::sf_copy(tsf + 8, tc::desc_sf(sa + ST_SFB));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = tc::desc_sw128(sa + ST_B0 + 32 * kk);
              const uint32_t accum = (first && kk == 0) ? 0u : 1u;
              const uint32_t id8 = tc::idesc_mxf8(128, 16, kk, kk);
              tc::mma_mxf8(acc, tc::desc_sw128(sa + ST_A0 + 32 * kk), bd, id8, tsf, tsf + 8, accum);
              tc::mma_mxf8(acc + 16, tc::desc_sw128(sa + ST_A1 + 32 * kk), bd, id8, tsf + 4, tsf + 8, accum);
            }
          } else if (U.kind == U_SGU) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = tc::desc_sw128(sa + ST_B0 + 32 * kk);
              const uint32_t accum = (first && kk == 0) ? 0u : 1u;
              tc::mma_bf16(acc, tc::desc_sw128(sa + ST_A0 + 32 * kk), bd, id_bf, accum);
              tc::mma_bf16(acc + 16, tc::desc_sw128(sa + ST_A1 + 32 * kk), bd, id_bf, accum);
            }
          } else if (U.kind == U_RGU || U.kind == U_RDN) {
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
          } else if (U.kind == U_SDN && a.sh8) {
            const int halves = stage_halves(a, U, st);
            for (int h = 0; h < halves; ++h) {
              tc::sf_copy(tsf + 4 * h, tc::desc_sf(sa + ST_SFA + 512 * h));
              tc::sf_copy(tsf + 8 + 4 * h, tc::desc_sf(sa + ST_SFB + 512 * h));
            }
            for (int h = 0; h < halves; ++h) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t accum = (first && h == 0 && kk == 0) ? 0u : 1u;
                tc::mma_mxf8(acc, tc::desc_sw128(sa + (h ? ST_A1 : ST_A0) + 32 * kk),
                             tc::desc_sw128(sa + (h ? ST_B1 : ST_B0) + 32 * kk), tc::idesc_mxf8(128, 16, kk, kk),
                             tsf + 4 * h, tsf + 8 + 4 * h, accum);
              }
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
    if (a.sh8) {  // the MXFP8 shared expert's units wait for x8 (and start before the routing)
      quant_x8(a, et);
      tc::fence_proxy_async_global();
      epi_sync();
      if (et == 0) red_release_add(a.ctr + C_DC_X8, 1);
    }
    if constexpr (W) {
      // the routing table is not built yet: its storage stages x for the router
      router_w(a, et, reinterpret_cast<float*>(&R));
      quant_tokens_w<NV>(a, et, s_qe[et >> 5]);
    } else {
      for (int e = blockIdx.x; e < a.Er; e += a.G) router_row(a, e, et, red_s, epoch);
    }
    if (et == 0) DC_TRACE(TR_ROUTER);
    if constexpr (!W) {
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
      if (et == 0) {
        red_release_add(a.ctr + C_DC_READY, 1);
        DC_TRACE(TR_X);
      }
      build_routing(a, R, et, epoch, &s_fail);
    } else {
      build_routing_w(a, R, et, epoch, &s_fail);
    }
    if (et == 0) DC_TRACE(TR_ROUTING);
    if (s_fail) {
      if (et == 0) fail();
    } else {
      if (et == 0) tc::mbar_arrive(&routing_ready);
      if constexpr (W) {
        // x into sorted order, this block's share, then counted
        for (int i = blockIdx.x * EPI_THREADS + et; i < n * (H / 32); i += a.G * EPI_THREADS) sort_x_w<NV>(a, R, i);
        tc::fence_proxy_async_global();
        epi_sync();
        if (et == 0) {
          red_release_add(a.ctr + C_DC_READY, 1);
          DC_TRACE(TR_X);
        }
      }
      if (blockIdx.x == 0)  // the router's top-k, [T][kr]
        for (int i = et; i < n; i += EPI_THREADS)
          if (i % a.k < a.kr) {
            const int o = i / a.k * a.kr + i % a.k;
            if (a.ids_out) a.ids_out[o] = R.ids[i];
            if (a.w_out) a.w_out[o] = R.w[i];
          }
      const int n_slots = R.n_slots;

      const int dn_total = nbH * ((a.shared ? a.s_sdn * a.nck : 0) + n_slots);  // down parts over all tiles
      for (int i = 0;; ++i) {
        const int buf = i % NACC;
        const uint32_t use = (uint32_t)(i / NACC);
        if (!DYN && (int)blockIdx.x + i * a.G >= units_total(a, n_slots)) break;
        if (et == 0) {
          int uu = blockIdx.x + i * a.G;
          s_ok = true;
          if constexpr (DYN) {
            const int q = i % UQ;
            s_ok = tc::mbar_wait(&uq_full[q], (i / UQ) & 1, a.limit_ns, &abort_flag);
            uu = -1;
            if (s_ok) {
              uu = s_uq[q];
              tc::mbar_arrive(&uq_empty[q]);
            }
          }
          if (s_ok && uu >= 0) s_ok = tc::mbar_wait(&acc_full[buf], use & 1, a.limit_ns, &abort_flag);
          if (!s_ok) fail();
          s_unit[i & 1] = uu;
        }
        epi_sync();
        const int u = s_unit[i & 1];
        if (!s_ok || u < 0) break;
        const Unit U = unit_at(a, n_slots, u);
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
        float rg_sg = 1.0f, rg_su = 1.0f;  // one-part routed tiles: the gate / up factors
        if (U.kind == U_SGU) {
          // column c is token 16 chunk + c
          // (a tile of one part keeps its sums in registers for the finisher)
          float* dst = a.gu_sh + ((size_t)U.part * T + 16 * U.chunk) * 2 * I + 128 * U.tile + m;
          const int nt = imin(16, T - 16 * U.chunk);
          if (a.s_sgu > 1)
#pragma unroll
            for (int c = 0; c < 16; ++c)
              if (c < nt) {
                dst[(size_t)c * 2 * I] = v[c];
                dst[(size_t)c * 2 * I + I] = v[16 + c];
              }
          ticket = U.tile * a.nck + U.chunk;
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
            // the rows' x shifts 2^c_t, loaded together (one round trip)
            if (et < cnt) s_rows[et] = __ldcg(a.xshift + R.tok[beg + et]);
            epi_sync();
          }
          if (a.s_rgu == 1) {
            // the tile's only part: the finisher takes the sums from v
            rg_sg = sg;
            rg_su = su;
          } else if constexpr (W) {
            // wide steps: B held the slot's sorted rows, column c is position beg + c
#pragma unroll
            for (int c = 0; c < 16; ++c)
              if (c < cnt) {
                const float f = NV ? pow2f(s_rows[c]) : 1.0f;
                dst[(size_t)c * 2 * I] = v[c] * (sg * f);
                dst[(size_t)c * 2 * I + I] = v[16 + c] * (su * f);
              }
          } else {
            for (int c = 0; c < cnt; ++c) {
              const int t = R.tok[beg + c];
              const float f = NV ? pow2f(s_rows[c]) : 1.0f;
              dst[(size_t)c * 2 * I] = pick16(v, 0, t) * (sg * f);
              dst[(size_t)c * 2 * I + I] = pick16(v, 16, t) * (su * f);
            }
          }
          ticket = a.tk_rgu + U.slot * nbI + U.tile;
          target = a.s_rgu;
        } else if (U.kind == U_SDN) {
          float* dst = a.ys + ((size_t)U.part * T + 16 * U.chunk) * H + 128 * U.tile + m;
          const int nt = imin(16, T - 16 * U.chunk);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (c < nt) dst[(size_t)c * H] = v[c];
          ticket = -1;
          target = 0;
        } else {
          // B held the slot's sorted rows: column c is sorted position beg + c
          // (NVFP4: times the expert's down tensor scale and 2^c of the h row)
          // columns 0-15: the pair's first 128 rows of H, 16-31: its second
          float* dst = a.y_assign + (size_t)beg * H + 256 * U.tile + m;
          const float sd = NV ? __ldg(a.tscale + 3 * R.slot_e[U.slot] + 2) : 1.0f;
          if (NV) {  // the rows' shifts, loaded together (one round trip, not one per row)
            if (et < cnt) s_rows[et] = h_row_shift(a, beg + et);
            epi_sync();
          }
#pragma unroll
          for (int c = 0; c < MAX_DECODE_T; ++c)
            if (c < cnt) {
              const float f = NV ? sd * pow2f(s_rows[c]) : 1.0f;
              dst[(size_t)c * H] = NV ? v[c] * f : v[c];
              dst[(size_t)c * H + 128] = NV ? v[16 + c] * f : v[16 + c];
            }
          ticket = -1;
          target = 0;
        }
        if (et == 0) DC_TRACE(TR_LAST_UNIT + U.kind);
        if (et == 0 && U.kind == U_RGU) DC_SLOT_LAST(U.slot, TS_RGU_DONE);
        if (ticket < 0) {
          // a down part: counted without waiting; the combine runs after the unit list
          epi_sync();
          if (et == 0) red_release_add(a.ctr + C_DC_DN, U.kind == U_RDN ? 2 : 1);
          if (et == 0 && U.kind == U_RDN) DC_SLOT_LAST(U.slot, TS_RDN_DONE);
          continue;
        }
        // split-K arrival: the block that brings the last part finishes the
        // tile (a tile of one part needs no ticket: its own stores precede)
        if (target > 1) {
          epi_sync();
          if (et == 0) {
            s_last = atom_add_acq_rel(a.tickets + ticket, 1) == target - 1;
            if (s_last) a.tickets[ticket] = 0;  // no other arrival follows in this launch
          }
          epi_sync();
          if (!s_last) continue;
        }
        if (U.kind == U_SGU) {
          const float* src = a.gu_sh + 128 * U.tile + m;
          const size_t stride = (size_t)T * 2 * I;
          const int tb = 16 * U.chunk, te = imin(T, tb + 16);  // the chunk's tokens
          for (int t0 = tb; t0 < te; t0 += 2) {  // two tokens' loads in flight together
            float g[2], up[2];
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
              const int t = imin(t0 + tt, te - 1);
              if (a.s_sgu == 1) {
                g[tt] = pick16(v, 0, t - tb);
                up[tt] = pick16(v, 16, t - tb);
              } else {
                g[tt] = sum_parts(src + (size_t)t * 2 * I, stride, a.s_sgu);
                up[tt] = sum_parts(src + (size_t)t * 2 * I + I, stride, a.s_sgu);
              }
            }
#pragma unroll
            for (int tt = 0; tt < 2; ++tt)
              if (t0 + tt < te) {
                const float hv = silu(g[tt]) * up[tt];
                if (a.sh8) {
                  // MXFP8 per 32 along I: warp q holds one block of the row
                  const int ex = mx8_scale_exp(warp_max(fabsf(hv)));
                  reinterpret_cast<uint8_t*>(a.h_shared)[(size_t)(t0 + tt) * I + 128 * U.tile + m] =
                      (uint8_t)e4m3_rne1(hv * pow2_neg(ex));
                  if (lane == 0)
                    a.h8s[((size_t)U.chunk * nbI + U.tile) * 512 + ((t0 + tt) & 15) * 16 + q] = (uint8_t)(ex + 127);
                } else {
                  a.h_shared[(size_t)(t0 + tt) * I + 128 * U.tile + m] = f32_to_bf16_rn(hv);
                }
              }
          }
          if (a.sh8 && lane == 0)  // rows of the chunk past T: zero scales in the B tile
            for (int r = te - tb; r < 16; ++r) a.h8s[((size_t)U.chunk * nbI + U.tile) * 512 + r * 16 + q] = 0;
          tc::fence_proxy_async_global();
          epi_sync();
          if (et == 0) red_release_add(a.ctr + C_DC_HSH, 1);
        } else if (U.kind == U_RGU) {
          // h = SiLU(G) U requantised to MXFP4: warp q holds one 32-column block
          const float* src = a.gu_r + (size_t)beg * 2 * I + 128 * U.tile + m;
          const size_t stride = (size_t)n * 2 * I;
          for (int c = 0; c < cnt; ++c) {
            float g, up;
            if (a.s_rgu == 1) {  // the same products the part store would hold
              const int col = W ? c : R.tok[beg + c];
              const float f = NV ? pow2f(s_rows[c]) : 1.0f;  // loaded at the unit's start
              g = pick16(v, 0, col) * (rg_sg * f);
              up = pick16(v, 16, col) * (rg_su * f);
            } else {
              g = sum_parts(src + (size_t)c * 2 * I, stride, a.s_rgu);
              up = sum_parts(src + (size_t)c * 2 * I + I, stride, a.s_rgu);
            }
            const float h = silu(g) * up;
            const int ex = mx_scale_exp(warp_max_nonneg(fabsf(h)));
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
            if (et == 0) {
              red_release_add(a.tickets + a.tk_slot + U.slot, 1);
              red_release_add(a.ctr + C_DC_HR, 1);
              DC_SLOT_LAST(U.slot, TS_H);
              DC_SLOT_SET(U.slot, TS_INFO, ((unsigned long long)R.slot_e[U.slot] << 8) | (unsigned)cnt);
            }
          } else {
            // NVFP4: the slot's last finished tile knows every row's largest
            // exponent and writes the slot's UE4M3 scale blocks for the down MMA
            if (et == 0) {
              s_last = atom_add_acq_rel(a.tickets + a.tk_nv + U.slot, 1) == nbI - 1;
              if (s_last) a.tickets[a.tk_nv + U.slot] = 0;
            }
            epi_sync();
            if (s_last) {
              convert_h_scales_nv(a, U.slot, beg, cnt, et);
              tc::fence_proxy_async_global();
              epi_sync();
              if (et == 0) {
                red_release_add(a.tickets + a.tk_slot + U.slot, 1);
                red_release_add(a.ctr + C_DC_HR, 1);
                DC_SLOT_LAST(U.slot, TS_H);
                DC_SLOT_SET(U.slot, TS_INFO, ((unsigned long long)R.slot_e[U.slot] << 8) | (unsigned)cnt);
              }
            }
          }
        }
      }
      if (et == 0) DC_TRACE(TR_UNITS);
      // out = BF16(ys + sum_j w_j y_j), summed in a fixed order, once every
      // down part is stored.  Items (128 columns of H x CT tokens) are spread
      // over all blocks.  The rows an item reads (per token its k y rows and
      // the shared expert's down parts, 512 B each) come into the idle stage
      // ring by bulk copies, all in flight at once, and are summed from
      // shared memory, so an item costs one load round trip and the code,
      // which runs once per launch, stays compact.
      const int nsp = a.shared ? a.s_sdn : 0, rpt = k + nsp;  // rows per token
      // wide steps: 32 tokens per item (one round of items at 128 tokens)
      // where their rows fit the ring, else 16; narrow steps 4
      const int CT = W ? (32 * rpt * 512 <= DSTAGES * (int)STAGE_BYTES ? 32 : 16) : 4;
      const int n_items = nbH * ((T + CT - 1) / CT);
      if ((int)blockIdx.x < n_items) {
        if (et == 0) {
          s_ok = wait_at_least(a.ctr + C_DC_DN, dn_total, status, a.limit_ns);
          if (!s_ok) fail();
        }
        epi_sync();
      }
      if (et == 0) DC_TRACE(TR_DOWN_SEEN);
      float* cbuf = reinterpret_cast<float*>(dsm);  // [CT][rpt][128]: the ring's consumers are done
      uint32_t it = 0;
      for (int item = blockIdx.x; item < n_items && s_ok; item += a.G, ++it) {
        const int cg = item % nbH, t0 = CT * (item / nbH), nt = imin(CT, T - t0), nrows = nt * rpt;
        if (et == 0) tc::mbar_expect_tx(&comb, (uint32_t)nrows * 512u);
        epi_sync();  // the expected bytes precede every copy; the last item's reads are done
        for (int r = et; r < nrows; r += EPI_THREADS) {
          const int tt = r / rpt, j = r % rpt, t = t0 + tt;
          const float* src = j < k ? a.y_assign + (size_t)R.inv[t * k + j] * H + 128 * cg
                                   : a.ys + ((size_t)(j - k) * T + t) * H + 128 * cg;
          tc::bulk_load(cbuf + (size_t)r * 128, src, 512, &comb);
        }
        if (!tc::mbar_wait(&comb, it & 1, a.limit_ns, &abort_flag)) {
          fail();
          tc::mbar_wait(&comb, it & 1, a.limit_ns, &never_s);  // the copies land before the block exits
          break;
        }
        for (int tt = 0; tt < nt; ++tt) {
          const int t = t0 + tt;
          const float* row = cbuf + (size_t)tt * rpt * 128 + m;
          float yv[MAX_TOPK], wv[MAX_TOPK], pv[DC_SDN_MAX];  // a token's loads issued together
#pragma unroll
          for (int j = 0; j < MAX_TOPK; ++j) {
            yv[j] = j < k ? row[j * 128] : 0.0f;
            wv[j] = j < k ? R.w[t * k + j] : 0.0f;
          }
#pragma unroll
          for (int p = 0; p < DC_SDN_MAX; ++p) pv[p] = p < nsp ? row[(k + p) * 128] : 0.0f;
          float acc = 0.0f;
#pragma unroll
          for (int p = 0; p < DC_SDN_MAX; ++p)
            if (p < nsp) acc += pv[p];
#pragma unroll
          for (int j = 0; j < MAX_TOPK; ++j)
            if (j < k) acc = fmaf(wv[j], yv[j], acc);
          a.out[(size_t)t * H + 128 * cg + m] = f32_to_bf16_rn(acc);
        }
      }
    }
  }

  if (threadIdx.x == 64) DC_TRACE(TR_END);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, tmem_cols<NV>());
  }
  // The last block out resets the launch's counters for the next call and
  // clears the NVFP4 row exponents (atomicMax words: a word tagged with an
  // older launch number than the next launch's would otherwise win it).
  if (threadIdx.x == 0) s_last = atom_add_acq_rel(a.ctr + C_DC_EXIT, 1) == a.G - 1;
  __syncthreads();
  if (s_last) {
    if (a.nv)
      for (int i = threadIdx.x; i < a.T * a.k; i += blockDim.x) a.rowmax[i] = 0ull;
    for (int i = threadIdx.x; i < a.nslot_max; i += blockDim.x) a.tickets[a.tk_slot + i] = 0;
    if (threadIdx.x == 0) {
      a.ctr[C_DC_READY] = 0;
      a.ctr[C_DC_HSH] = 0;
      a.ctr[C_DC_HR] = 0;
      a.ctr[C_DC_EXIT] = 0;
      a.ctr[C_DC_DN] = 0;
      a.ctr[C_DC_RT] = 0;
      a.ctr[C_DC_X8] = 0;
      a.ctr[C_DC_QUEUE] = 0;
      a.ctr[C_DC_EPOCH] = (int)s_epoch;
    }
    // (the launch's end makes these stores visible to the next launch)
  }
}

}  // namespace

bool fused_decode_tc_supported(const Shape& sh, const ExpertsDev& ex) {
  return ex.w13s_mma && ex.w2s_mma && sh.T >= 1 && sh.T <= MAX_WIDE_T && sh.H % 256 == 0 && sh.I % 256 == 0 &&
         (!ex.nv || sh.H <= 8192);  // the NVFP4 quantiser keeps a row's 32-block exponents in shared memory
}

cudaError_t launch_fused_decode_tc(const Shape& sh, const ExpertsDev& ex, const SharedDev& shd, const float* wr,
                                   const float* bias, const uint16_t* x, uint16_t* out, int* ids_out, float* w_out,
                                   void* ws, uint64_t wait_limit_ns, cudaStream_t s, int fold, int score,
                                   const Shared8Dev* sh8) {
  if (sh.T == 0) return cudaSuccess;
  if (!fused_decode_tc_supported(sh, ex)) return cudaErrorInvalidValue;
  if (sh8 && (!sh8->w13s_mma || !sh8->w2s_mma || shd.w13 || fold)) return cudaErrorInvalidValue;
  const int T = sh.T, H = sh.H, I = sh.I, E = sh.E, k = sh.k, n = T * k;
  const WsLayout L = ws_layout(T, H, I, E, k);
  uint8_t* base = static_cast<uint8_t*>(ws);
  const bool nv = ex.nv != 0;
  // One block per SM: the stage ring leaves no room for a second block,
  // whose TMA stream would share the SM's copy engine.
  const size_t smem = (size_t)DSTAGES * (nv ? stage_bytes<true>() : stage_bytes<false>()) + 1024;
  static_assert(DSTAGES * stage_bytes<false>() + 1024 > 114 * 1024, "the ring must keep one block per SM");
  const bool wide = T > MAX_DECODE_T;
  // one block per SM: every block holds a 200 KB stage ring and a TMEM allocation
  const int G = imin(sm_count(), DC_MAX_GRID);
  // dynamic hand-out where the routed gate/up units take more than one round
  const bool dyn = !wide && imin(n, E) * (I / 128) >= G;
  auto kern = nv ? (wide ? k_decode_tc<true, true, false> : dyn ? k_decode_tc<true, false, true> : k_decode_tc<true, false, false>)
                 : (wide ? k_decode_tc<false, true, false>
                         : dyn ? k_decode_tc<false, false, true> : k_decode_tc<false, false, false>);
  cudaError_t err = cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, DT, smem)) != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const bool shared = shd.w13 != nullptr || sh8 != nullptr;
  DcSplits sp = dc_splits(T, H, I, E, k, G);
  if (sh8) {  // MXFP8 stages hold 128 K elements: no more parts than stages
    sp.sgu = imin(sp.sgu, H / 128);
    sp.sdn = imin(sp.sdn, (I / 128 + 1) / 2);
  }

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
  a.nck = dc_nck(T);
  a.n_sgu = shared ? (I / 128) * sp.sgu * a.nck : 0;
  a.n_sdn = shared ? (H / 128) * sp.sdn * a.nck : 0;
  a.nslot_max = dc_nslot_max(T, k, E);
  a.tk_rgu = (I / 128) * a.nck;
  a.tk_nv = a.tk_rgu + a.nslot_max * (I / 128) + H / 128;
  a.tk_slot = a.tk_nv + a.nslot_max;
  a.shared = shared ? 1 : 0;
  a.nv = ex.nv;
  a.sh8 = sh8 ? 1 : 0;
  if (sh8) {
    a.w13s8_mma = sh8->w13s_mma;
    a.w2s8_mma = sh8->w2s_mma;
    a.x8 = base + L.dc_x8;
    a.x8s = base + L.dc_x8s;
    a.h8s = base + L.dc_h8s;
  }
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
  a.xq = wide ? base + L.dc_xqs : base + L.xq;
  a.topk64 = reinterpret_cast<unsigned long long*>(base + L.dc_topk64);
  a.rpart = reinterpret_cast<float*>(base + L.dc_rpart);
  {  // wide steps with about as many assignments as experts: ~80 MB of the first experts' W13 to L2
    const double per = (double)2 * I * (H / 2) * (1.0 + (nv ? 1.0 / 8 : 1.0 / 16));
    a.pf_experts = wide && n >= E ? imin(E - fold, (int)(80e6 / per)) : 0;
  }
  a.xq_tok = base + L.xq;  // [T, H/2]
  a.xe_tok = base + L.xs;  // [T, H/32]
  a.xs_mma = base + L.dc_xs;
  a.xshift = reinterpret_cast<int*>(base + L.dc_xshift);
  a.hsc = base + L.dc_hsc;
  a.depth = imin(n, E) >= 16 ? 4 : 2;
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
  if ((err = make_map(&m.xq, a.xq, wide ? n : T, H / 2, 16)) != cudaSuccess) return err;
  if ((err = make_map(&m.hq, a.hq, n, I / 2, 16)) != cudaSuccess) return err;
  if (sh8) {  // E4M3 rows: one byte per element
    if ((err = make_map(&m.w13s, sh8->w13, (uint64_t)2 * I, (uint64_t)H)) != cudaSuccess) return err;
    if ((err = make_map(&m.w2s, sh8->w2, H, (uint64_t)I)) != cudaSuccess) return err;
    if ((err = make_map(&m.x, a.x8, T, (uint64_t)H, 16)) != cudaSuccess) return err;
    if ((err = make_map(&m.hsh, a.h_shared, T, (uint64_t)I, 16)) != cudaSuccess) return err;
  } else if (shared) {
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

extern "C" MOE_API moe_status_t moe_debug_decode_trace(uint64_t* dst, size_t bytes) {
#if MOEFP4_TRACE
  void* p = nullptr;
  void* q = nullptr;
  if (cudaGetSymbolAddress(&p, moefp4::g_dc_trace) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaGetSymbolAddress(&q, moefp4::g_dc_slot_trace) != cudaSuccess) return MOE_ERR_CUDA;
  const size_t nb = sizeof(moefp4::g_dc_trace), ns = sizeof(moefp4::g_dc_slot_trace);
  cudaError_t e;
  if (!dst) {
    e = cudaMemset(p, 0, nb);
    if (e == cudaSuccess) e = cudaMemset(q, 0, ns);
  } else {
    e = cudaMemcpy(dst, p, bytes < nb ? bytes : nb, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && bytes > nb)
      e = cudaMemcpy(reinterpret_cast<uint8_t*>(dst) + nb, q, bytes - nb < ns ? bytes - nb : ns,
                     cudaMemcpyDeviceToHost);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
#else
  (void)dst;
  (void)bytes;
  return MOE_ERR_UNSUPPORTED;
#endif
}
