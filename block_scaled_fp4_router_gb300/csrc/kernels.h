// Host-side launchers of libmoefp4's kernels (C++ linkage, internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "layout.h"

namespace moefp4 {

// Instrumentation (defined in api.cu): every kernel launch of the library is
// counted (moe_debug_launch_count), and the routed tensor-core GEMMs of the
// batched path are bracketed by the events set with moe_set_timing_events.
void count_launch();
enum TimingMark { MARK_ROUTED_GEMM_BEGIN = 0, MARK_ROUTED_GEMM_END = 1 };
void record_mark(TimingMark m, cudaStream_t s);

struct ExpertsDev {
  int nv;  // 0 = MXFP4, 1 = NVFP4
  const uint8_t* w13;
  const uint8_t* w13s;
  const uint8_t* w2;
  const uint8_t* w2s;
  const float* tscale;  // NVFP4 [E, 3]
  const uint8_t* w13s_mma;  // prepared tensor-core scale layout, or null
  const uint8_t* w2s_mma;
};

struct SharedDev {
  const uint16_t* w13;  // BF16 [2I, H] or null
  const uint16_t* w2;   // BF16 [H, I]
};

struct Shape {
  int T, H, I, E, k;
};

// Canonical scale bytes [E][R][K/32] -> tensor-core layout [E][R/128][K/128][512 B].
cudaError_t launch_relayout_weight_sf(const uint8_t* s, int E, int R, int K, uint8_t* out, cudaStream_t st);
// A4
cudaError_t launch_quant_mxfp4(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                               cudaStream_t s);
// A4 for the MXFP8 shared expert: E4M3 codes [rows][K], E8M0 scales [rows][K/32].
cudaError_t launch_quant_mxfp8(const uint16_t* x, int rows, int K, uint8_t* codes, uint8_t* scales,
                               cudaStream_t s);
// A1.  part: [router_splits][T][E].  With wsplit ([3][E][H] BF16 scratch) and
// a shape router_tc_supported accepts, the products run on tensor cores
// (three BF16 terms of the weights, 64-element K chunks summed in FP32).
cudaError_t launch_router_logits(const uint16_t* x, const float* wr, const float* bias, float* logits,
                                 int T, int H, int E, float* part, cudaStream_t s, uint16_t* wsplit = nullptr,
                                 int* status = nullptr, uint64_t limit_ns = 0);
bool router_tc_supported(int T, int H, int E);
int router_tc_splits(int T, int H, int E);
cudaError_t launch_router_tc(const uint16_t* x, const float* wr, const float* bias, float* out, int T, int H,
                             int E, int S, uint16_t* wsplit, int* status, uint64_t limit_ns, cudaStream_t s);
// A2.  score: SCORE_SOFTMAX (logits hold the bias) or SCORE_SIGMOID (raw
// logits; sel_bias, may be null, corrects the choice only).
// ids_ext / w_ext (optional): [T][k + 1], the last column the shared expert
// folded into the table (id E, weight 1).
cudaError_t launch_topk(const float* logits, int T, int E, int k, int score, const float* sel_bias, int* ids,
                        float* w, cudaStream_t s, int* ids_ext = nullptr, float* w_ext = nullptr);
// A3
// status: where a checked build records an out-of-range id (may be null)
cudaError_t launch_permute(const int* ids, int T, int k, int E, int* counts, int* offsets, int* perm,
                           int* inv_perm, int* rank, int* chunk_cnt, int* chunk_base, cudaStream_t s,
                           int* status = nullptr);
// A5 - A7 on CUDA cores (any T; the decode-sized path)
cudaError_t launch_routed_simt(const Shape& sh, const ExpertsDev& ex, const uint8_t* xq, const uint8_t* xs,
                               const int* offsets, const int* perm, uint8_t* hq, uint8_t* hs, float* y_assign,
                               cudaStream_t s, int* status = nullptr);
// A8 on CUDA cores
cudaError_t launch_shared_simt(const Shape& sh, const SharedDev& shd, const uint16_t* x, uint16_t* h_shared,
                               float* y_shared, cudaStream_t s);

// Workspace regions of the tensor-core path.
struct TcWorkspace {
  int* poff;
  void* mtiles;
  int* num_mt;
  uint8_t* xq_perm;
  uint8_t* xs_mma;
  uint8_t* hq_perm;
  uint8_t* hs_mma;
  uint8_t* w13s_mma;
  uint8_t* w2s_mma;
};
// The combine fused into the routed down GEMM (A9 in A7's epilogue): acc FP32
// [T][H] += topk_w[a] * y of every assignment a (already holding the shared
// expert's output, or zero).
struct CombineArgs {
  const float* topk_w;  // [T * k], flat assignment t * k + j
  float* acc;
  int slice_rows;       // acc laid out by 256-column slices [H/256][T][256] (slice_rows = T), or 0: [T][H]
};
// A5 - A7 on tensor cores (MXFP4 weights)
// wa: weights as the MMA's A operand and 64-row token windows as B (small
// per-expert batches); otherwise 128-token tiles as A, where comb (optional)
// replaces the y_assign store by the fused combine.
cudaError_t launch_expert_ffn_tc(const Shape& sh, const ExpertsDev& ex, const TcWorkspace& w, const uint8_t* xq,
                                 const uint8_t* xs, const int* offsets, const int* perm, float* y_assign,
                                 int* status, uint64_t limit_ns, bool wa, cudaStream_t s,
                                 const CombineArgs* comb = nullptr);
// out BF16 [T][H] = acc FP32, laid out [T][H] or (slice_rows = T) [H/256][T][256].
cudaError_t launch_acc_to_bf16(const float* acc, int T, int H, int slice_rows, uint16_t* out, cudaStream_t s);
// Whether n assignments over E experts take the weights-as-A GEMMs under an
// orientation mode (TC_GEMM_*).
bool tc_weights_as_a(int n, int E, int mode);
// A8 on tensor cores
// parts: split-K scratch, float [max(s1 * T * 2I, s2 * T * H)] (see shared_ksplit)
// slice_rows = T: y_shared written by 256-column slices [H/256][T][256]
cudaError_t launch_shared_tc(const Shape& sh, const SharedDev& shd, const uint16_t* x, uint16_t* h_shared,
                             float* y_shared, float* parts, int* status, uint64_t limit_ns, cudaStream_t s,
                             int slice_rows = 0);
// Copies the requantised h to sorted-assignment order (either layout).
cudaError_t launch_copy_h(const Shape& sh, const int* hpath, const uint8_t* hq_sorted, const uint8_t* hs_sorted,
                          const TcWorkspace& w, uint8_t* hq_out, uint8_t* hs_out, cudaStream_t s);
// The MXFP8 shared expert (E4M3 weights with E8M0 scales per 32) and its
// scratch: xq [T_pad][H], xs [T_pad][H/32], the MMA-layout scales of x, h,
// W13 and W2, and hq [T_pad][I] (T_pad = T rounded up to 128).
struct Shared8Dev {
  const uint8_t* w13;
  const uint8_t* w13s;
  const uint8_t* w2;
  const uint8_t* w2s;
  const uint8_t* w13s_mma;  // prepared scale layout, or null (re-laid per call)
  const uint8_t* w2s_mma;
};
struct Shared8Ws {
  uint8_t* xq;
  uint8_t* xs;
  uint8_t* xs_mma;
  uint8_t* hq;
  uint8_t* hs_mma;
  uint8_t* w13s_mma;
  uint8_t* w2s_mma;
};
cudaError_t launch_shared_mxfp8_tc(const Shape& sh, const Shared8Dev& sh8, const uint16_t* x, const Shared8Ws& w,
                                   float* y_shared, int* status, uint64_t limit_ns, cudaStream_t s,
                                   int slice_rows = 0);
// A9
cudaError_t launch_combine(const Shape& sh, const float* y_assign, const int* inv_perm, const float* w,
                           const float* y_shared, uint16_t* out, cudaStream_t s, int* status = nullptr);
// A10 on CUDA cores: needs H and I multiples of 64 (rows streamed in
// 64-element pairs by 32-byte loads).
inline bool fused_decode_supported(const Shape& sh) {
  return sh.T >= 1 && sh.T <= MAX_DECODE_T && sh.H % 64 == 0 && sh.I % 64 == 0;
}
cudaError_t launch_fused_decode(const Shape& sh, const ExpertsDev& ex, const SharedDev& shd,
                                const float* wr, const float* bias, const uint16_t* x, uint16_t* out,
                                int* ids_out, float* w_out, void* ws, uint64_t wait_limit_ns,
                                cudaStream_t s, int score = 0);
// A10 on tensor cores (MXFP4 weights with prepared scales, H and I multiples of 256).
bool fused_decode_tc_supported(const Shape& sh, const ExpertsDev& ex);
// sh: the table shape (E experts, k assignments per token).  fold = 1: the
// shared expert is table entry E - 1, the router has E - 1 rows and picks
// k - 1 experts; ids_out / w_out are [T][k - fold].
cudaError_t launch_fused_decode_tc(const Shape& sh, const ExpertsDev& ex, const SharedDev& shd, const float* wr,
                                   const float* bias, const uint16_t* x, uint16_t* out, int* ids_out, float* w_out,
                                   void* ws, uint64_t wait_limit_ns, cudaStream_t s, int fold = 0, int score = 0,
                                   const Shared8Dev* sh8 = nullptr);
// bytes (a multiple of 16) from src to dst, both 16-byte aligned, device or
// GPU-addressable pinned host memory, by SM loads and stores.
cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t s);
// NVFP4 -> MXFP4 conversion of the routed experts (load time).
cudaError_t launch_nvfp4_to_mxfp4(const Shape& sh, const ExpertsDev& ex, uint8_t* w13_out, uint8_t* w13s_out,
                                  uint8_t* w2_out, uint8_t* w2s_out, cudaStream_t s);
// MXFP8 (E4M3 codes [n], E8M0 scales [n/32]) -> BF16 [n], n a multiple of 32.
cudaError_t launch_mxfp8_to_bf16(const uint8_t* codes, const uint8_t* scales, size_t n, uint16_t* out,
                                 cudaStream_t s);
// A bounded wait on a counter nothing ever advances (exercises the timeout path).
cudaError_t launch_wait_probe(void* ws, uint64_t wait_limit_ns, cudaStream_t s);

}  // namespace moefp4
