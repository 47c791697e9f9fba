// Workspace layout and limits of libmoefp4, shared by host and device code.
#pragma once

#include <stddef.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__
#else
#define MOE_HD
#endif

namespace moefp4 {

constexpr int MAX_TOPK = 8;
constexpr int MAX_E = 256;
constexpr int MAX_DECODE_T = 16;   // fused single-launch decode range (both engines)
constexpr int MAX_WIDE_T = 128;    // single-launch range of the tensor-core engine (17..128: wide steps)
constexpr int PERM_CHUNK = 1024;   // assignments ranked per block in the permutation
constexpr int TC_MIN_ASSIGN = 256; // routed experts on tensor cores from this many assignments
constexpr int TC_MIN_T_SHARED = 128; // shared expert on tensor cores from this many tokens
constexpr int SPLIT_SMS = 152;        // SMs the split-K counts are balanced for

// Tensor-core decode (T <= MAX_WIDE_T): one block per SM, at most this many.
constexpr int DC_MAX_GRID = 256;
constexpr int DC_MAX_SPLIT = 16;

MOE_HD inline int imin(int a, int b) { return a < b ? a : b; }
MOE_HD inline int imax(int a, int b) { return a > b ? a : b; }

// Split-K factor: as many parts as keep `tiles` output tiles within one work
// unit per block of a `grid`-block launch, at most one part per K stage.
MOE_HD inline int dc_split(int tiles, int stages, int grid) {
  int s = grid / (tiles > 0 ? tiles : 1);
  s = imin(imin(s, stages), DC_MAX_SPLIT);
  return s < 1 ? 1 : s;
}

// The tensor-core decode's B operand holds 16 token rows.  Steps of up to 16
// tokens have one such chunk; wider steps (17..MAX_WIDE_T tokens) run the
// shared expert per 16-token chunk and the routed experts per slot, a run of
// at most 16 sorted assignments of one expert.
MOE_HD inline int dc_nck(int T) { return T <= MAX_DECODE_T ? 1 : (T + 15) / 16; }
// Expert slots a step can have: one per distinct expert, plus (wide steps)
// one more per 16 assignments of an expert.
MOE_HD inline int dc_nslot_max(int T, int k, int E) {
  const int n = T * k;
  return T <= MAX_DECODE_T ? imin(n, E) : imin(n, E) + (n + 15) / 16;
}
// Arrival tickets: shared gate/up tiles per chunk, routed gate/up tiles per
// slot, (unused) H tiles, NVFP4 per-slot scale tickets, then per-slot
// counters of finished routed h (the down units' dependency).
MOE_HD inline int dc_ticket_count(int T, int H, int I, int E, int k) {
  const int ns = dc_nslot_max(T, k, E);
  return (I / 128) * dc_nck(T) + ns * (I / 128) + H / 128 + 2 * ns;
}

// Split factors of the tensor-core decode: shared gate/up (K = H in 64-element
// BF16 stages), routed gate/up (K = H in 256-element FP4 stages) and shared
// down (K = I in stages of two 64-element chunks; four parts make a part the
// size of one routed down unit).
struct DcSplits {
  int sgu, rgu, sdn;
};
MOE_HD inline DcSplits dc_splits(int T, int H, int I, int E, int k, int grid) {
  const int nslot = imin(T * k, E);
  const int nck = dc_nck(T);
  DcSplits d;
  d.sgu = dc_split(I / 128 * nck, H / 64, grid);
  d.rgu = dc_split((nslot > 0 ? nslot : 1) * (I / 128), H / 256 > 0 ? H / 256 : 1, grid);
  d.sdn = imin(4, (I / 64 + 1) / 2);
  if (nck > 1) d.sdn = imin(d.sdn, dc_split(H / 128 * nck, (I / 64 + 1) / 2, grid));
  return d;
}

// Split-K parts of the batched router (T > 512): enough 128 x 128 tiles for
// two blocks per SM of a 152-SM GPU, at most 8.
// Split-K count of the router.  T <= 16: one pass per expert row, no split.
// 16 < T <= 512 (64 x 64 tiles): the largest power of two that keeps K parts
// a multiple of 32 elements, at least 64 long, and the grid within 608
// blocks.  Larger T (128 x 128 tiles, two 256-thread blocks per SM): S in
// 1..8 minimising the busiest SM's share, ceil(tiles S / SMs) / S (the
// smallest S on ties).
MOE_HD inline int router_splits(int T, int E, int H) {
  if (T <= 16) return 1;
  if (T <= 512) {
    const int tiles = ((T + 63) / 64) * ((E + 63) / 64);
    int s = 1;
    while (H % (2 * s * 32) == 0 && H / (2 * s) >= 64 && tiles * 2 * s <= 608) s *= 2;
    return s;
  }
  const int tiles = ((T + 127) / 128) * ((E + 127) / 128);
  int best = 1;
  for (int s = 2; s <= 8; ++s)
    if ((int64_t)((tiles * s + SPLIT_SMS - 1) / SPLIT_SMS) * best <
        (int64_t)((tiles * best + SPLIT_SMS - 1) / SPLIT_SMS) * s)
      best = s;
  return best;
}

// Split-K count of a dense tensor-core GEMM of the shared expert with `tiles`
// output tiles and `nks` K stages: enough parts to give every SM a unit when
// the tiles alone do not (1 from SPLIT_SMS / 2 tiles up), at most 16 and
// at most the stages.
MOE_HD inline int shared_ksplit(int tiles, int nks) {
  if (2 * tiles >= SPLIT_SMS) return 1;
  int s = SPLIT_SMS / tiles;
  if (s > 16) s = 16;
  if (s > nks) s = nks;
  return s < 1 ? 1 : s;
}
// The BF16 shared expert runs on tensor cores from TC_MIN_T_SHARED tokens when
// its 128 x 256 tiles and 64-element K stages divide the shape.
MOE_HD inline bool shared_tc_path(int T, int H, int I) {
  return T >= TC_MIN_T_SHARED && H % 256 == 0 && I % 128 == 0;
}
// Output tiles of the shared expert's gate/up (first) and down GEMMs on
// tensor cores: 128 tokens x 256 weight rows.
MOE_HD inline int shared_tiles_gu(int T, int I) { return (T + 127) / 128 * (2 * I / 256); }
MOE_HD inline int shared_tiles_dn(int T, int H) { return (T + 127) / 128 * (H / 256); }

// Rows of the per-expert padded order (each expert's rows rounded up to 128).
MOE_HD inline int tc_padded_rows(int n, int E) { return ((n + E * 127) + 127) / 128 * 128; }
// The same with windows of `win` rows (128, or 64 for the weights-as-A GEMMs).
MOE_HD inline int tc_padded_rows_win(int n, int E, int win) {
  return ((n + E * (win - 1)) + win - 1) / win * win;
}
// Routed tensor-core GEMM orientation: tokens as the MMA's A operand
// (128-token tiles), or weights as A with up to 64 tokens as B, chosen when
// the average expert has at most WA_MAX_AVG_ROWS assignments.
enum { TC_GEMM_AUTO = 0, TC_GEMM_TOKENS_AS_A = 1, TC_GEMM_WEIGHTS_AS_A = 2 };
constexpr int WA_MAX_AVG_ROWS = 32;
MOE_HD inline bool tc_routed_enabled(int n) { return n >= TC_MIN_ASSIGN; }

// Device status word values (mirror moe_status_t).
constexpr int MOE_DEV_OK = 0;
constexpr int MOE_DEV_INVALID = 1;  // a caller-given index out of range (checked builds)
constexpr int MOE_DEV_TIMEOUT = 4;

// Counters of the fused decode launch (ints at the start of the workspace).
enum Counter : int {
  C_STATUS = 0,    // device status word
  C_QUEUE = 1,     // next work unit to hand out
  C_ROUTER = 2,    // router rows finished
  C_QUANT = 3,     // token rows quantised
  C_GU = 4,        // gate/up units finished (shared + routed)
  C_EXIT = 5,      // blocks finished (the last one resets the counters)
  C_TEST = 6,      // never written by the library: a wait on it always times out
  C_HPATH = 7,     // low byte: layout the last expert FFN left h in (0 sorted, 1 / 2 windows of 128 / 64)
  C_DC_READY = 8,  // tensor-core decode: blocks done with their quantisation slice
  C_DC_HSH = 9,    // tensor-core decode: shared-expert h tiles finished
  C_DC_HR = 10,    // tensor-core decode: routed h tiles finished
  C_DC_EXIT = 11,  // tensor-core decode: blocks finished
  C_DC_EPOCH = 12, // tensor-core decode: launches completed on this workspace (tags the logits)
  C_DC_DN = 13,    // tensor-core decode: down-projection parts stored
  C_DC_RT = 14,    // tensor-core decode, wide steps: blocks done with their router parts
  C_DC_X8 = 15,    // tensor-core decode, MXFP8 shared expert: blocks done quantising x to MXFP8
  C_DC_QUEUE = 16, // tensor-core decode: units handed out after each block's first
  N_COUNTERS = 32
};

MOE_HD inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Byte offsets of every workspace region for one layer shape.
struct WsLayout {
  size_t counters;     // int [N_COUNTERS]
  size_t dc_tickets;   // int: split-K arrival tickets of the tensor-core decode
  size_t dc_logit64;   // uint64 [T, E]: tensor-core decode logits tagged with the launch number
  size_t dc_rowmax;    // uint64 [T*k]: NVFP4 h row exponents tagged with the launch number
  size_t dc_topk64;    // uint64 [2][T*k]: wide steps' router top-k (ids, weights) tagged with the launch number
  size_t zero_end;     // end of the part that must start zero-filled
  size_t logits;       // float [T, E]
  size_t rt_part;      // float [splits, T, E]: split-K parts of the batched router
  size_t rt_wsplit;    // bf16 [3][E][H]: the tensor-core router's three terms of the weights (T > 512)
  size_t ids;          // int [T, k]       (when the caller passes no output)
  size_t wts;          // float [T, k]
  size_t ids_r;        // int [T, k]: the router's top-k when the shared expert is folded into the table
  size_t wts_r;        // float [T, k]
  size_t xq;           // uint8 [T, H/2]
  size_t xs;           // uint8 [T, H/32]
  size_t counts;       // int [E]
  size_t offsets;      // int [E+1]
  size_t perm;         // int [T*k]
  size_t inv_perm;     // int [T*k]
  size_t rank;         // int [T*k]        permutation scratch
  size_t chunk_cnt;    // int [nchunks, E]
  size_t chunk_base;   // int [nchunks, E]
  size_t hq;           // uint8 [T*k, I/2]
  size_t hs;           // uint8 [T*k, I/32]
  size_t h_shared;     // bf16 [T, I]
  size_t y_assign;     // float [T*k, H]   (layer_forward only)
  size_t y_shared;     // float [T, H]     (layer_forward only)
  size_t sh_part;      // float split-K parts of the shared expert's GEMMs
  size_t s8_xq, s8_xs, s8_xs_mma, s8_hq, s8_hs_mma, s8_w13s, s8_w2s;  // MXFP8 shared expert
  // tensor-core path (present when the routed experts run on tensor cores)
  size_t tc_poff;      // int [E+1]
  size_t tc_mtiles;    // 16-byte tile descriptors [padded rows / 128]
  size_t tc_num_mt;    // int
  size_t tc_xq;        // uint8 [padded rows, H/2]
  size_t tc_xs;        // scale blocks [padded rows/128][H/128][512 B]
  size_t tc_hq;        // uint8 [padded rows, I/2]
  size_t tc_hs;        // scale blocks [padded rows/128][I/128][512 B]
  size_t tc_w13s;      // weight scale blocks [E][2I/128][H/128][512 B]
  size_t tc_w2s;       // weight scale blocks [E][H/128][I/128][512 B]
  // tensor-core decode (T <= MAX_WIDE_T)
  size_t dc_xs;        // x scales, MMA layout [H/128][512 B] (E8M0) or [H/64][512 B] (UE4M3), 16 token
                       // rows; wide steps: one such set per slot
  size_t dc_xshift;    // int [16] (wide steps: [T*k]): NVFP4 per-row power of two of the x scales
  size_t dc_xqs;       // wide steps: uint8 [T*k, H/2] x codes in sorted-assignment order
  size_t dc_rpart;     // wide steps: float [H/256][T][E] router partial sums (256-element K parts)
  size_t dc_x8;        // MXFP8 shared expert: uint8 [T, H] E4M3 codes of x (h's codes go to h_shared)
  size_t dc_x8s;       // their scales, MMA layout [16-token chunks][H/128][512 B]
  size_t dc_h8s;       // h's scales, MMA layout [16-token chunks][I/128][512 B]
  size_t dc_hs;        // routed h scales, MMA layout [slots][I/128][512 B] (E8M0) or [slots][I/64][512 B] (UE4M3)
  size_t dc_hsc;       // NVFP4: E8M0 bytes of h [T*k][I/32] before the per-row UE4M3 conversion
  size_t dc_gu_sh;     // float [splits][T][2I]  shared gate/up partial sums
  size_t dc_gu_r;      // float [splits][T*k][2I] routed gate/up partial sums
  size_t dc_ys;        // float [splits][T][H]   shared down partial sums
  size_t total;
};

// E, k: experts in the table and assignments per token (with a shared expert
// folded into the table: the router's E + 1 and top_k + 1).  The router's
// regions fit a router over E or E - 1 experts, so the layout depends on the
// table shape alone.
MOE_HD inline WsLayout ws_layout(int T, int H, int I, int E, int k) {
  const int Er = E > 1 ? E - 1 : E;
  WsLayout L{};
  const size_t n = (size_t)T * k;
  const size_t nchunks = (n + PERM_CHUNK - 1) / PERM_CHUNK;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + (bytes ? bytes : 1));
    return at;
  };
  const bool dc = T <= MAX_WIDE_T;
  const bool wide = T > MAX_DECODE_T;
  const int nslot = dc_nslot_max(T, k, E);
  const DcSplits sp = dc_splits(T, H, I, E, k, DC_MAX_GRID);
  // The regions the tensor-core decode needs zeroed (or tagged) across calls
  // sit at the same offsets, sized for the whole single-launch range, in the
  // layout of every T: no call of any size writes anything else there.
  L.counters = take(sizeof(int) * N_COUNTERS);
  L.dc_tickets = take(sizeof(int) * (size_t)dc_ticket_count(MAX_WIDE_T, H, I, E, k));
  L.dc_logit64 = take(sizeof(uint64_t) * (size_t)MAX_WIDE_T * E);
  L.dc_rowmax = take(sizeof(uint64_t) * (size_t)MAX_WIDE_T * MAX_TOPK);
  L.dc_topk64 = take(sizeof(uint64_t) * 2 * (size_t)MAX_WIDE_T * MAX_TOPK);
  L.zero_end = o;
  L.logits = take(sizeof(float) * (size_t)T * E);
  const size_t rparts = (size_t)imax(router_splits(T, E, H) * E, router_splits(T, Er, H) * Er);
  L.rt_part = take(rparts > (size_t)E || (T > 16 && T <= 512) ? sizeof(float) * rparts * (size_t)T : 0);
  L.rt_wsplit = take(T > 512 ? (size_t)6 * E * H : 0);
  L.ids = take(sizeof(int) * n);
  L.wts = take(sizeof(float) * n);
  L.ids_r = take(sizeof(int) * n);
  L.wts_r = take(sizeof(float) * n);
  L.xq = take((size_t)T * H / 2);
  L.xs = take((size_t)T * H / 32);
  L.counts = take(sizeof(int) * E);
  L.offsets = take(sizeof(int) * (E + 1));
  L.perm = take(sizeof(int) * n);
  L.inv_perm = take(sizeof(int) * n);
  L.rank = take(sizeof(int) * n);
  L.chunk_cnt = take(sizeof(int) * nchunks * E);
  L.chunk_base = take(sizeof(int) * nchunks * E);
  L.hq = take(n * I / 2);
  L.hs = take(n * I / 32);
  L.h_shared = take((size_t)2 * T * I);
  L.y_assign = take(sizeof(float) * n * H);
  L.y_shared = take(sizeof(float) * (size_t)T * H);
  {  // split-K partial sums of the shared expert's tensor-core GEMMs
    const bool shtc = shared_tc_path(T, H, I);
    const size_t s1 = shtc ? shared_ksplit(shared_tiles_gu(T, I), H / 64) : 1;
    const size_t s2 = shtc ? shared_ksplit(shared_tiles_dn(T, H), I / 64) : 1;
    const size_t a = s1 > 1 ? s1 * T * 2 * (size_t)I : 0, b = s2 > 1 ? s2 * T * (size_t)H : 0;
    L.sh_part = take(sizeof(float) * (a > b ? a : b));
  }

  const bool tc = tc_routed_enabled((int)n);
  const size_t R = tc ? (size_t)tc_padded_rows((int)n, E) : 0;
  // 64-row windows (weights-as-A GEMMs): no more rows, up to twice the tiles
  // and scale blocks per row
  const size_t R64 = tc ? (size_t)tc_padded_rows_win((int)n, E, 64) : 0;
  const size_t tiles = R / 128 > R64 / 64 ? R / 128 : R64 / 64;
  L.tc_poff = take(tc ? sizeof(int) * (E + 1) : 0);
  L.tc_mtiles = take(16 * tiles);
  L.tc_num_mt = take(tc ? sizeof(int) : 0);
  L.tc_xq = take(R * H / 2);
  L.tc_xs = take(tiles * (H / 128) * 512);
  L.tc_hq = take(R * I / 2);
  L.tc_hs = take(tiles * (I / 128) * 512);
  L.tc_w13s = take(tc ? (size_t)E * 2 * I * H / 32 : 0);
  L.tc_w2s = take(tc ? (size_t)E * H * I / 32 : 0);
  L.dc_xs = take(dc ? (size_t)(wide ? nslot : 1) * (H / 64) * 512 : 0);
  L.dc_xshift = take(dc ? sizeof(int) * (wide ? n : (size_t)MAX_DECODE_T) : 0);
  L.dc_xqs = take(wide ? n * H / 2 : 0);
  L.dc_rpart = take(wide ? sizeof(float) * (size_t)(H / 256 > 0 ? H / 256 : 1) * T * E : 0);
  L.dc_x8 = take(dc ? (size_t)T * H : 0);
  L.dc_x8s = take(dc ? (size_t)dc_nck(T) * (H / 128) * 512 : 0);
  L.dc_h8s = take(dc ? (size_t)dc_nck(T) * (I / 128) * 512 : 0);
  L.dc_hs = take(dc ? (size_t)nslot * (I / 64) * 512 : 0);
  L.dc_hsc = take(dc ? n * (I / 32) : 0);
  L.dc_gu_sh = take(dc ? sizeof(float) * sp.sgu * T * 2 * (size_t)I : 0);
  L.dc_gu_r = take(dc ? sizeof(float) * sp.rgu * n * 2 * (size_t)I : 0);
  L.dc_ys = take(dc ? sizeof(float) * sp.sdn * T * (size_t)H : 0);
  L.total = o;
  {  // MXFP8 shared expert (T rounded up to 128 rows).  Inside a layer call it
     // runs between the routing and the routed experts, so it keeps clear of
     // every region above except the tensor-core decode's scratch (from dc_xs
     // on), which only the single-launch decode uses and which holds nothing
     // across calls.
    size_t o8 = L.dc_xs;
    auto take8 = [&](size_t bytes) {
      size_t at = o8;
      o8 = align256(o8 + (bytes ? bytes : 1));
      return at;
    };
    const size_t tp = ((size_t)T + 127) / 128 * 128;
    L.s8_xq = take8(tp * H);
    L.s8_xs = take8(tp * H / 32);
    L.s8_xs_mma = take8(tp * H / 32);
    L.s8_hq = take8(tp * I);
    L.s8_hs_mma = take8(tp * I / 32);
    L.s8_w13s = take8((size_t)2 * I * H / 32);
    L.s8_w2s = take8((size_t)H * I / 32);
    if (o8 > L.total) L.total = o8;
  }
  return L;
}

}  // namespace moefp4
