// The C ABI of libmoefp4 (declared in include/moefp4.h): argument validation
// on the host, workspace carving, and the launch sequences of the unfused and
// fused layer paths.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>

#include "moefp4.h"
#include "kernels.h"
#include "layout.h"
#include "routing.cuh"

using namespace moefp4;

namespace {

// An NVTX range over one entry point (named after it in profiler timelines;
// without an attached tool the push and pop do nothing).
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
};
#define MOE_RANGE() const Range moe_range_(__func__)

std::atomic<uint64_t> g_wait_limit_ns{500ull * 1000 * 1000};
std::atomic<int> g_routed_gemm{TC_GEMM_AUTO};
std::atomic<uint64_t> g_launches{0};
std::atomic<cudaEvent_t> g_marks[2] = {{nullptr}, {nullptr}};

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status_t check_desc(const moe_layer_desc_t* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->H <= 0 || d->I <= 0 || d->E <= 0) return MOE_ERR_INVALID_ARG;
  if (d->H % 32 || d->I % 32) return MOE_ERR_INVALID_ARG;  // whole MXFP4 blocks along H and I
  if (d->top_k < 1 || d->top_k > MAX_TOPK || d->E < d->top_k || d->E > MAX_E) return MOE_ERR_INVALID_ARG;
  if ((int64_t)d->T * d->top_k > (int64_t)1 << 30) return MOE_ERR_INVALID_ARG;
  if ((int64_t)d->H > (1 << 20) || (int64_t)d->I > (1 << 20)) return MOE_ERR_INVALID_ARG;
  if (d->renormalize != 1 || d->act_quant != 1) return MOE_ERR_UNSUPPORTED;
  if (d->shared_in_table != 0 && d->shared_in_table != 1) return MOE_ERR_INVALID_ARG;
  if (d->shared_in_table && (d->top_k + 1 > MAX_TOPK || d->E + 1 > MAX_E)) return MOE_ERR_UNSUPPORTED;
  if (d->score_func != SCORE_SOFTMAX && d->score_func != SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

// The router bias goes into the logits (softmax scoring) or only into the
// top-k choice (sigmoid scoring).
inline const float* logit_bias(const moe_layer_desc_t* d, const float* bias) {
  return d->score_func == SCORE_SOFTMAX ? bias : nullptr;
}
inline const float* select_bias(const moe_layer_desc_t* d, const float* bias) {
  return d->score_func == SCORE_SIGMOID ? bias : nullptr;
}

// The shape of the expert table and of the per-token assignments: with the
// shared expert folded into the table, E + 1 experts and top_k + 1
// assignments (the last one expert E with weight 1).
moe_layer_desc_t table_desc(const moe_layer_desc_t* d) {
  moe_layer_desc_t t = *d;
  t.E += d->shared_in_table;
  t.top_k += d->shared_in_table;
  t.shared_in_table = 0;
  return t;
}

WsLayout layout_of(const moe_layer_desc_t* d) {
  const moe_layer_desc_t t = table_desc(d);
  return ws_layout(t.T, t.H, t.I, t.E, t.top_k);
}

moe_status_t check_ws(const moe_layer_desc_t* d, void* ws, size_t ws_bytes) {
  if (!ws || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < layout_of(d).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status_t check_experts(const moe_layer_desc_t* d, const moe_experts_t* ex, ExpertsDev* out) {
  if (!ex) return MOE_ERR_INVALID_ARG;
  if (ex->fmt != MOE_W_MXFP4 && ex->fmt != MOE_W_NVFP4) return MOE_ERR_INVALID_ARG;
  const bool nv = ex->fmt == MOE_W_NVFP4;
  if (!ex->w13 || !ex->w13_scale || !ex->w2 || !ex->w2_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(ex->w13, 16) || !aligned(ex->w2, 16)) return MOE_ERR_INVALID_ARG;
  if (nv) {
    if (!ex->tensor_scale || !aligned(ex->w13_scale, 2) || !aligned(ex->w2_scale, 2)) return MOE_ERR_INVALID_ARG;
  } else if (ex->tensor_scale) {
    return MOE_ERR_INVALID_ARG;
  }
  if ((ex->w13_scale_mma && !aligned(ex->w13_scale_mma, 16)) || (ex->w2_scale_mma && !aligned(ex->w2_scale_mma, 16)))
    return MOE_ERR_INVALID_ARG;
  const bool prepared = ex->w13_scale_mma && ex->w2_scale_mma;
  *out = ExpertsDev{nv ? 1 : 0, ex->w13, ex->w13_scale, ex->w2, ex->w2_scale, ex->tensor_scale,
                    prepared ? ex->w13_scale_mma : nullptr, prepared ? ex->w2_scale_mma : nullptr};
  return MOE_OK;
}

moe_status_t check_shared(const moe_shared_bf16_t* sh, SharedDev* out) {
  *out = SharedDev{nullptr, nullptr};
  if (!sh || (!sh->w13 && !sh->w2)) return MOE_OK;
  if (!sh->w13 || !sh->w2 || !aligned(sh->w13, 16) || !aligned(sh->w2, 16)) return MOE_ERR_INVALID_ARG;
  *out = SharedDev{static_cast<const uint16_t*>(sh->w13), static_cast<const uint16_t*>(sh->w2)};
  return MOE_OK;
}

moe_status_t check_shared8(const moe_layer_desc_t* d, const moe_shared_mxfp8_t* sh, Shared8Dev* out) {
  if (d->shared_in_table) return MOE_ERR_INVALID_ARG;  // one shared expert, not two
  if (d->H % 256 || d->I % 256) return MOE_ERR_UNSUPPORTED;
  if (!sh || !sh->w13 || !sh->w13_scale || !sh->w2 || !sh->w2_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(sh->w13, 16) || !aligned(sh->w2, 16) || !aligned(sh->w13_scale, 4) || !aligned(sh->w2_scale, 4))
    return MOE_ERR_INVALID_ARG;
  if ((sh->w13_scale_mma && !aligned(sh->w13_scale_mma, 16)) || (sh->w2_scale_mma && !aligned(sh->w2_scale_mma, 16)))
    return MOE_ERR_INVALID_ARG;
  const bool prepared = sh->w13_scale_mma && sh->w2_scale_mma;
  *out = Shared8Dev{sh->w13, sh->w13_scale, sh->w2, sh->w2_scale, prepared ? sh->w13_scale_mma : nullptr,
                    prepared ? sh->w2_scale_mma : nullptr};
  return MOE_OK;
}

inline moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                   \
  do {                                  \
    const moe_status_t st_ = (expr);    \
    if (st_ != MOE_OK) return st_;      \
  } while (0)

#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

Shape shape_of(const moe_layer_desc_t* d) { return Shape{d->T, d->H, d->I, d->E, d->top_k}; }

// A5 - A8: the routed experts on tensor cores when the batch is large enough
// and the weights are MXFP4 (kind::mxf4 takes E8M0 scales), otherwise on CUDA
// cores; the shared expert likewise from TC_MIN_T_SHARED tokens.
//
// With fuse_w (the flat routing weights [T * k]) and the routed experts on
// 128-token tensor-core tiles, the combine runs inside the routed down GEMM:
// the shared expert first writes ys into acc (FP32 [T][H]; zero-filled
// without a shared expert), the down GEMM adds every weighted expert output
// into it, and *fused reports that acc then holds the layer output in FP32
// (y_assign is not written).
moe_status_t run_expert_ffn(const moe_layer_desc_t* d, const ExpertsDev& ex, const SharedDev& shd,
                            const uint16_t* x, const uint8_t* xq, const uint8_t* xs, const int* offsets,
                            const int* perm, float* y_assign, float* y_shared, void* ws, cudaStream_t s,
                            const float* fuse_w = nullptr, float* acc = nullptr, bool* fused = nullptr,
                            const Shared8Dev* sh8 = nullptr, int* slice_rows = nullptr) {
  const WsLayout L = ws_layout(d->T, d->H, d->I, d->E, d->top_k);
  const Shape sh = shape_of(d);
  const uint64_t limit = g_wait_limit_ns.load();
  int* status = at<int>(ws, L.counters) + C_STATUS;
  const bool tc = !ex.nv && tc_routed_enabled(d->T * d->top_k) && d->H % 256 == 0 && d->I % 256 == 0 &&
                  aligned(ex.w13s, 4) &&
                  aligned(ex.w2s, 4);
  const bool wa = tc && tc_weights_as_a(d->T * d->top_k, d->E, g_routed_gemm.load());
  const bool fuse = fuse_w && acc && tc && !wa;
  if (fused) *fused = fuse;
  // record which layout h is left in (read by moe_debug_requantized_h)
  MOE_CUDA(cudaMemsetAsync(at<int>(ws, L.counters) + C_HPATH, tc ? (wa ? 2 : 1) : 0, sizeof(int), s));
  const bool has_shared = shd.w13 || sh8;
  // The fused combine keeps the accumulator by 256-column slices (each pass
  // of the down GEMM then works on one contiguous T x 1 KB block) when its
  // first writer, the shared expert, is a tensor-core GEMM or absent.
  const int slice = fuse && (!has_shared || sh8 || shared_tc_path(d->T, d->H, d->I)) ? d->T : 0;
  if (slice_rows) *slice_rows = slice;
  auto shared_expert = [&](float* ys, int sl) -> moe_status_t {
    if (sh8) {  // MXFP8 on kind::mxf8f6f4 tensor cores
      const Shared8Ws w8{at<uint8_t>(ws, L.s8_xq), at<uint8_t>(ws, L.s8_xs),     at<uint8_t>(ws, L.s8_xs_mma),
                         at<uint8_t>(ws, L.s8_hq), at<uint8_t>(ws, L.s8_hs_mma), at<uint8_t>(ws, L.s8_w13s),
                         at<uint8_t>(ws, L.s8_w2s)};
      return cuda_status(launch_shared_mxfp8_tc(sh, *sh8, x, w8, ys, status, limit, s, sl));
    }
    uint16_t* h = at<uint16_t>(ws, L.h_shared);
    if (shared_tc_path(d->T, d->H, d->I))
      return cuda_status(launch_shared_tc(sh, shd, x, h, ys, at<float>(ws, L.sh_part), status, limit, s, sl));
    return cuda_status(launch_shared_simt(sh, shd, x, h, ys, s));
  };
  if (fuse) {  // the accumulator starts as ys (or zero)
    if (has_shared)
      MOE_TRY(shared_expert(acc, slice));
    else
      MOE_CUDA(cudaMemsetAsync(acc, 0, sizeof(float) * (size_t)d->T * d->H, s));
  }
  if (tc) {
    TcWorkspace w{at<int>(ws, L.tc_poff), at<uint8_t>(ws, L.tc_mtiles), at<int>(ws, L.tc_num_mt),
                  at<uint8_t>(ws, L.tc_xq), at<uint8_t>(ws, L.tc_xs), at<uint8_t>(ws, L.tc_hq),
                  at<uint8_t>(ws, L.tc_hs), at<uint8_t>(ws, L.tc_w13s), at<uint8_t>(ws, L.tc_w2s)};
    const CombineArgs comb{fuse_w, acc, slice};
    MOE_CUDA(launch_expert_ffn_tc(sh, ex, w, xq, xs, offsets, perm, y_assign, status, limit, wa, s,
                                  fuse ? &comb : nullptr));
  } else {
    MOE_CUDA(launch_routed_simt(sh, ex, xq, xs, offsets, perm, at<uint8_t>(ws, L.hq), at<uint8_t>(ws, L.hs),
                                y_assign, s, status));
  }
  if (has_shared && !fuse) MOE_TRY(shared_expert(y_shared, 0));
  return MOE_OK;
}

// The whole layer through the per-step kernels (any T).  With the shared
// expert folded into the table, top-k also writes [T][k + 1] copies whose
// last column is expert E with weight 1, and the rest runs on the table
// shape with no BF16 shared expert.
moe_status_t run_forward(const moe_layer_desc_t* desc, const ExpertsDev& ex, const SharedDev& shd,
                         const float* w_router, const float* bias, const uint16_t* xb, uint16_t* out,
                         int32_t* topk_ids, float* topk_w, void* ws, cudaStream_t s,
                         const Shared8Dev* sh8 = nullptr) {
  const moe_layer_desc_t dt = table_desc(desc);
  const int fold = desc->shared_in_table;
  const WsLayout L = ws_layout(dt.T, dt.H, dt.I, dt.E, dt.top_k);
  const Shape sh = shape_of(&dt);
  int* ids_r = topk_ids ? topk_ids : at<int>(ws, fold ? L.ids_r : L.ids);
  float* w_r = topk_w ? topk_w : at<float>(ws, fold ? L.wts_r : L.wts);
  int* ids = fold ? at<int>(ws, L.ids) : ids_r;  // [T][table k]
  float* w = fold ? at<float>(ws, L.wts) : w_r;
  MOE_CUDA(launch_router_logits(xb, w_router, logit_bias(desc, bias), at<float>(ws, L.logits), desc->T, desc->H,
                                desc->E, at<float>(ws, L.rt_part), s, at<uint16_t>(ws, L.rt_wsplit),
                                at<int>(ws, L.counters) + C_STATUS, g_wait_limit_ns.load()));
  MOE_CUDA(launch_topk(at<float>(ws, L.logits), desc->T, desc->E, desc->top_k, desc->score_func,
                       select_bias(desc, bias), ids_r, w_r, s, fold ? ids : nullptr, fold ? w : nullptr));
  MOE_CUDA(launch_quant_mxfp4(xb, sh.T, sh.H, at<uint8_t>(ws, L.xq), at<uint8_t>(ws, L.xs), s));
  MOE_CUDA(launch_permute(ids, sh.T, sh.k, sh.E, at<int>(ws, L.counts), at<int>(ws, L.offsets),
                          at<int>(ws, L.perm), at<int>(ws, L.inv_perm), at<int>(ws, L.rank),
                          at<int>(ws, L.chunk_cnt), at<int>(ws, L.chunk_base), s));
  float* ysh = (shd.w13 || sh8) ? at<float>(ws, L.y_shared) : nullptr;
  bool fused = false;
  int slice = 0;
  MOE_TRY(run_expert_ffn(&dt, ex, shd, xb, at<uint8_t>(ws, L.xq), at<uint8_t>(ws, L.xs), at<int>(ws, L.offsets),
                         at<int>(ws, L.perm), at<float>(ws, L.y_assign), ysh, ws, s, w, at<float>(ws, L.y_shared),
                         &fused, sh8, &slice));
  if (fused)  // the combine ran in the down GEMM: the FP32 output is rounded to BF16
    return cuda_status(launch_acc_to_bf16(at<float>(ws, L.y_shared), sh.T, sh.H, slice, out, s));
  return cuda_status(launch_combine(sh, at<float>(ws, L.y_assign), at<int>(ws, L.inv_perm), w, ysh, out, s,
                                    at<int>(ws, L.counters) + C_STATUS));
}

}  // namespace

namespace moefp4 {

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void record_mark(TimingMark m, cudaStream_t s) {
  cudaEvent_t ev = g_marks[m].load();
  if (!ev) return;
  // inside a stream capture the record must become an event node of the graph
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}

}  // namespace moefp4

extern "C" {

void moe_debug_launch_count(uint64_t* n) {
  if (n) *n = g_launches.load();
}

void moe_set_timing_events(void* routed_gemm_begin, void* routed_gemm_end) {
  g_marks[MARK_ROUTED_GEMM_BEGIN].store(static_cast<cudaEvent_t>(routed_gemm_begin));
  g_marks[MARK_ROUTED_GEMM_END].store(static_cast<cudaEvent_t>(routed_gemm_end));
}

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_workspace_size(const moe_layer_desc_t* desc, size_t* bytes) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = layout_of(desc).total;
  return MOE_OK;
}

moe_status_t moe_get_status(void* ws, moe_status_t* st) {
  MOE_RANGE();
  if (!ws || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  if (!st) return MOE_ERR_INVALID_ARG;
  int v = 0;
  int* word = reinterpret_cast<int*>(ws) + C_STATUS;
  MOE_CUDA(cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost));
  if (v != 0) MOE_CUDA(cudaMemset(word, 0, sizeof(int)));
  *st = static_cast<moe_status_t>(v);
  return MOE_OK;
}

moe_status_t moe_prepare_weights(const moe_layer_desc_t* desc, const moe_experts_t* experts, uint8_t* w13_scale_mma,
                                 uint8_t* w2_scale_mma, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  const moe_layer_desc_t t = table_desc(desc);  // every expert of the table, a folded shared one included
  ExpertsDev ex;
  MOE_TRY(check_experts(&t, experts, &ex));
  if (!w13_scale_mma || !w2_scale_mma || !aligned(w13_scale_mma, 16) || !aligned(w2_scale_mma, 16) ||
      !aligned(ex.w13s, 4) || !aligned(ex.w2s, 4))
    return MOE_ERR_INVALID_ARG;
  // the tensor-core scale blocks are 128 rows x 128 (MXFP4) or 64 (NVFP4) K elements
  if (t.H % 128 || t.I % 128) return MOE_ERR_UNSUPPORTED;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Both formats keep 4 scale bytes per row per block column (128 elements of
  // MXFP4, 64 of NVFP4): the NVFP4 re-layout is the MXFP4 one over 2K.
  const int kf = ex.nv ? 2 : 1;
  MOE_CUDA(launch_relayout_weight_sf(ex.w13s, t.E, 2 * t.I, kf * t.H, w13_scale_mma, s));
  return cuda_status(launch_relayout_weight_sf(ex.w2s, t.E, t.H, kf * t.I, w2_scale_mma, s));
}

moe_status_t moe_convert_nvfp4_to_mxfp4(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                        uint8_t* w13_out, uint8_t* w13_scale_out, uint8_t* w2_out,
                                        uint8_t* w2_scale_out, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  const moe_layer_desc_t t = table_desc(desc);
  ExpertsDev ex;
  MOE_TRY(check_experts(&t, experts, &ex));
  if (!ex.nv) return MOE_ERR_INVALID_ARG;
  if (!w13_out || !w13_scale_out || !w2_out || !w2_scale_out || !aligned(w13_out, 16) || !aligned(w2_out, 16))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_nvfp4_to_mxfp4(shape_of(&t), ex, w13_out, w13_scale_out, w2_out, w2_scale_out,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_debug_requantized_h(const moe_layer_desc_t* desc, const void* ws, size_t ws_bytes, uint8_t* hq,
                                     uint8_t* hs, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  if (desc->shared_in_table) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ws(desc, const_cast<void*>(ws), ws_bytes));
  if (desc->T == 0) return MOE_OK;
  if (!hq || !hs || !aligned(hq, 16)) return MOE_ERR_INVALID_ARG;
  void* w = const_cast<void*>(ws);
  const WsLayout L = ws_layout(desc->T, desc->H, desc->I, desc->E, desc->top_k);
  TcWorkspace tw{at<int>(w, L.tc_poff), at<uint8_t>(w, L.tc_mtiles), at<int>(w, L.tc_num_mt), at<uint8_t>(w, L.tc_xq),
                 at<uint8_t>(w, L.tc_xs), at<uint8_t>(w, L.tc_hq), at<uint8_t>(w, L.tc_hs), at<uint8_t>(w, L.tc_w13s),
                 at<uint8_t>(w, L.tc_w2s)};
  return cuda_status(launch_copy_h(shape_of(desc), at<int>(w, L.counters) + C_HPATH, at<uint8_t>(w, L.hq),
                                   at<uint8_t>(w, L.hs), tw, hq, hs, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_copy_rows(void* dst, const void* src, size_t bytes, moe_stream_t stream) {
  MOE_RANGE();
  if (bytes == 0) return MOE_OK;
  if (!dst || !src || bytes % 16 || !aligned(dst, 16) || !aligned(src, 16)) return MOE_ERR_INVALID_ARG;
  // only memory the GPU addresses: device, managed, or pinned host memory
  // mapped into the GPU's address space (its device address is used)
  void* p[2] = {dst, const_cast<void*>(src)};
  for (void*& q : p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_INVALID_ARG;
    }
    if (at.type == cudaMemoryTypeHost) {
      if (!at.devicePointer) return MOE_ERR_INVALID_ARG;
      q = at.devicePointer;
    } else if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) {
      return MOE_ERR_INVALID_ARG;
    }
  }
  if (!aligned(p[0], 16) || !aligned(p[1], 16)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_copy16(p[0], p[1], bytes, reinterpret_cast<cudaStream_t>(stream)));
}

void moe_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns ? ns : 1); }

moe_status_t moe_set_routed_gemm(int32_t mode) {
  MOE_RANGE();
  if (mode < TC_GEMM_AUTO || mode > TC_GEMM_WEIGHTS_AS_A) return MOE_ERR_INVALID_ARG;
  g_routed_gemm.store(mode);
  return MOE_OK;
}

moe_status_t moe_debug_wait_probe(void* ws, size_t ws_bytes, uint64_t limit_ns, moe_stream_t stream) {
  MOE_RANGE();
  if (!ws || !aligned(ws, 256) || ws_bytes < sizeof(int) * N_COUNTERS) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_wait_probe(ws, limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_quant_act_mxfp4(int32_t rows, int32_t K, const void* x, uint8_t* codes, uint8_t* scales,
                                 moe_stream_t stream) {
  MOE_RANGE();
  if (rows < 0 || K <= 0 || K % 32) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 4)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quant_mxfp4(static_cast<const uint16_t*>(x), rows, K, codes, scales,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_quant_act_mxfp8(int32_t rows, int32_t K, const void* x, uint8_t* codes, uint8_t* scales,
                                 moe_stream_t stream) {
  MOE_RANGE();
  if (rows < 0 || K <= 0 || K % 32) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 8)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quant_mxfp8(static_cast<const uint16_t*>(x), rows, K, codes, scales,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_dequant_mxfp8_to_bf16(int32_t rows, int32_t K, const uint8_t* codes, const uint8_t* scales,
                                       void* out, moe_stream_t stream) {
  MOE_RANGE();
  if (rows < 0 || K <= 0 || K % 32) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!codes || !scales || !out || !aligned(codes, 8) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_mxfp8_to_bf16(codes, scales, (size_t)rows * K, static_cast<uint16_t*>(out),
                                          reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_router_topk(const moe_layer_desc_t* desc, const void* x, const float* w_router,
                             const float* bias, int32_t* topk_ids, float* topk_w, float* logits,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  if (desc->shared_in_table) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ws(desc, ws, ws_bytes));
  if (desc->T == 0) return MOE_OK;
  if (!x || !w_router || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16)) return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const WsLayout L = ws_layout(desc->T, desc->H, desc->I, desc->E, desc->top_k);
  float* lg = logits ? logits : at<float>(ws, L.logits);
  MOE_CUDA(launch_router_logits(static_cast<const uint16_t*>(x), w_router, logit_bias(desc, bias), lg, desc->T,
                                desc->H, desc->E, at<float>(ws, L.rt_part), s, at<uint16_t>(ws, L.rt_wsplit),
                                at<int>(ws, L.counters) + C_STATUS, g_wait_limit_ns.load()));
  return cuda_status(launch_topk(lg, desc->T, desc->E, desc->top_k, desc->score_func, select_bias(desc, bias),
                                 topk_ids, topk_w, s));
}

moe_status_t moe_permute(const moe_layer_desc_t* desc, const int32_t* topk_ids, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* ws, size_t ws_bytes,
                         moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  if (desc->shared_in_table) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ws(desc, ws, ws_bytes));
  if (!counts || !offsets || (desc->T > 0 && (!topk_ids || !perm || !inv_perm))) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(desc->T, desc->H, desc->I, desc->E, desc->top_k);
  return cuda_status(launch_permute(topk_ids, desc->T, desc->top_k, desc->E, counts, offsets, perm, inv_perm,
                                    at<int>(ws, L.rank), at<int>(ws, L.chunk_cnt), at<int>(ws, L.chunk_base),
                                    reinterpret_cast<cudaStream_t>(stream), at<int>(ws, L.counters) + C_STATUS));
}

moe_status_t moe_expert_ffn_fp4(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                const moe_shared_bf16_t* shared, const void* x, const uint8_t* xq,
                                const uint8_t* xs, const int32_t* offsets, const int32_t* perm,
                                float* y_assign, float* y_shared, void* ws, size_t ws_bytes,
                                moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  if (desc->shared_in_table) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ws(desc, ws, ws_bytes));
  ExpertsDev ex;
  SharedDev shd;
  MOE_TRY(check_experts(desc, experts, &ex));
  MOE_TRY(check_shared(shared, &shd));
  if (desc->T == 0) return MOE_OK;
  if (!xq || !xs || !offsets || !perm || !y_assign) return MOE_ERR_INVALID_ARG;
  if (!aligned(xq, 16) || !aligned(y_assign, 16)) return MOE_ERR_INVALID_ARG;
  if (shd.w13 && (!x || !y_shared || !aligned(x, 16) || !aligned(y_shared, 16))) return MOE_ERR_INVALID_ARG;
  if (!shd.w13 && y_shared) return MOE_ERR_INVALID_ARG;
  return run_expert_ffn(desc, ex, shd, static_cast<const uint16_t*>(x), xq, xs, offsets, perm, y_assign, y_shared,
                        ws, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_shared_expert_mxfp8(const moe_layer_desc_t* desc, const moe_shared_mxfp8_t* shared,
                                     const void* x, float* y_shared, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  if (desc->shared_in_table) return MOE_ERR_UNSUPPORTED;
  if (desc->H % 256 || desc->I % 256) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ws(desc, ws, ws_bytes));
  if (!shared || !shared->w13 || !shared->w13_scale || !shared->w2 || !shared->w2_scale) return MOE_ERR_INVALID_ARG;
  if (!aligned(shared->w13, 16) || !aligned(shared->w2, 16) || !aligned(shared->w13_scale, 4) ||
      !aligned(shared->w2_scale, 4))
    return MOE_ERR_INVALID_ARG;
  if (desc->T == 0) return MOE_OK;
  if (!x || !y_shared || !aligned(x, 16) || !aligned(y_shared, 16)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout_of(desc);
  Shared8Dev sh8;
  MOE_TRY(check_shared8(desc, shared, &sh8));
  const Shared8Ws w{at<uint8_t>(ws, L.s8_xq),  at<uint8_t>(ws, L.s8_xs),   at<uint8_t>(ws, L.s8_xs_mma),
                    at<uint8_t>(ws, L.s8_hq),  at<uint8_t>(ws, L.s8_hs_mma), at<uint8_t>(ws, L.s8_w13s),
                    at<uint8_t>(ws, L.s8_w2s)};
  return cuda_status(launch_shared_mxfp8_tc(shape_of(desc), sh8, static_cast<const uint16_t*>(x), w, y_shared,
                                            at<int>(ws, L.counters) + C_STATUS, g_wait_limit_ns.load(),
                                            reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_prepare_shared_mxfp8(const moe_layer_desc_t* desc, const moe_shared_mxfp8_t* shared,
                                      uint8_t* w13_scale_mma, uint8_t* w2_scale_mma, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  Shared8Dev sh8;
  MOE_TRY(check_shared8(desc, shared, &sh8));
  if (!w13_scale_mma || !w2_scale_mma || !aligned(w13_scale_mma, 16) || !aligned(w2_scale_mma, 16))
    return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MOE_CUDA(launch_relayout_weight_sf(sh8.w13s, 1, 2 * desc->I, desc->H, w13_scale_mma, s));
  return cuda_status(launch_relayout_weight_sf(sh8.w2s, 1, desc->H, desc->I, w2_scale_mma, s));
}

moe_status_t moe_debug_shared_mxfp8_h(const moe_layer_desc_t* desc, const void* ws, size_t ws_bytes, uint8_t* hq,
                                      uint8_t* hs, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  MOE_TRY(check_ws(desc, const_cast<void*>(ws), ws_bytes));
  if (desc->T == 0) return MOE_OK;
  if (!hq || !hs) return MOE_ERR_INVALID_ARG;
  const WsLayout L = layout_of(desc);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t* base = static_cast<const uint8_t*>(ws);
  const size_t tp = ((size_t)desc->T + 127) / 128 * 128;
  MOE_CUDA(cudaMemcpyAsync(hq, base + L.s8_hq, (size_t)desc->T * desc->I, cudaMemcpyDeviceToDevice, s));
  return cuda_status(cudaMemcpyAsync(hs, base + L.s8_hs_mma, tp * desc->I / 32, cudaMemcpyDeviceToDevice, s));
}

moe_status_t moe_layer_forward_shared_mxfp8(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                            const moe_shared_mxfp8_t* shared, const float* w_router,
                                            const float* bias, const void* x, void* out, int32_t* topk_ids,
                                            float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  MOE_TRY(check_ws(desc, ws, ws_bytes));
  ExpertsDev ex;
  Shared8Dev sh8;
  MOE_TRY(check_experts(desc, experts, &ex));
  MOE_TRY(check_shared8(desc, shared, &sh8));
  if (desc->T == 0) return MOE_OK;
  if (!x || !out || !w_router || !aligned(x, 16) || !aligned(out, 16) || !aligned(w_router, 16))
    return MOE_ERR_INVALID_ARG;
  return run_forward(desc, ex, SharedDev{nullptr, nullptr}, w_router, bias, static_cast<const uint16_t*>(x),
                     static_cast<uint16_t*>(out), topk_ids, topk_w, ws, reinterpret_cast<cudaStream_t>(stream), &sh8);
}

moe_status_t moe_layer_decode_shared_mxfp8(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                           const moe_shared_mxfp8_t* shared, const float* w_router,
                                           const float* bias, const void* x, void* out, int32_t* topk_ids,
                                           float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  if (desc->T > MAX_WIDE_T) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ws(desc, ws, ws_bytes));
  ExpertsDev ex;
  Shared8Dev sh8;
  MOE_TRY(check_experts(desc, experts, &ex));
  MOE_TRY(check_shared8(desc, shared, &sh8));
  if (desc->T == 0) return MOE_OK;
  if (!x || !out || !w_router || !aligned(x, 16) || !aligned(out, 16) || !aligned(w_router, 16))
    return MOE_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  uint16_t* ob = static_cast<uint16_t*>(out);
  // One launch needs the routed experts' and the shared expert's prepared
  // scales; otherwise the batched path with the same arithmetic.
  if (fused_decode_tc_supported(shape_of(desc), ex) && sh8.w13s_mma && sh8.w2s_mma)
    return cuda_status(launch_fused_decode_tc(shape_of(desc), ex, SharedDev{nullptr, nullptr}, w_router, bias, xb,
                                              ob, topk_ids, topk_w, ws, g_wait_limit_ns.load(), s, 0,
                                              desc->score_func, &sh8));
  return run_forward(desc, ex, SharedDev{nullptr, nullptr}, w_router, bias, xb, ob, topk_ids, topk_w, ws, s, &sh8);
}

moe_status_t moe_combine(const moe_layer_desc_t* desc, const float* y_assign, const int32_t* inv_perm,
                         const float* topk_w, const float* y_shared, void* out, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  if (desc->shared_in_table) return MOE_ERR_UNSUPPORTED;
  if (desc->T == 0) return MOE_OK;
  if (!y_assign || !inv_perm || !topk_w || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(y_assign, 16) || !aligned(out, 16) || (y_shared && !aligned(y_shared, 16)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(shape_of(desc), y_assign, inv_perm, topk_w, y_shared,
                                    static_cast<uint16_t*>(out), reinterpret_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_forward(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                               const moe_shared_bf16_t* shared, const float* w_router, const float* bias,
                               const void* x, void* out, int32_t* topk_ids, float* topk_w, void* ws,
                               size_t ws_bytes, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  MOE_TRY(check_ws(desc, ws, ws_bytes));
  const moe_layer_desc_t dt = table_desc(desc);
  ExpertsDev ex;
  SharedDev shd;
  MOE_TRY(check_experts(&dt, experts, &ex));
  MOE_TRY(check_shared(shared, &shd));
  if (desc->shared_in_table && shd.w13) return MOE_ERR_INVALID_ARG;  // one shared expert, not two
  if (desc->T == 0) return MOE_OK;
  if (!x || !out || !w_router || !aligned(x, 16) || !aligned(out, 16) || !aligned(w_router, 16))
    return MOE_ERR_INVALID_ARG;
  return run_forward(desc, ex, shd, w_router, bias, static_cast<const uint16_t*>(x), static_cast<uint16_t*>(out),
                     topk_ids, topk_w, ws, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_layer_decode(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                              const moe_shared_bf16_t* shared, const float* w_router, const float* bias,
                              const void* x, void* out, int32_t* topk_ids, float* topk_w, void* ws,
                              size_t ws_bytes, moe_stream_t stream) {
  MOE_RANGE();
  MOE_TRY(check_desc(desc));
  if (desc->T > MAX_WIDE_T) return MOE_ERR_UNSUPPORTED;
  MOE_TRY(check_ws(desc, ws, ws_bytes));
  const moe_layer_desc_t dt = table_desc(desc);
  ExpertsDev ex;
  SharedDev shd;
  MOE_TRY(check_experts(&dt, experts, &ex));
  MOE_TRY(check_shared(shared, &shd));
  if (desc->shared_in_table && shd.w13) return MOE_ERR_INVALID_ARG;
  if (desc->T == 0) return MOE_OK;
  if (!x || !out || !w_router || !aligned(x, 16) || !aligned(out, 16) || !aligned(w_router, 16))
    return MOE_ERR_INVALID_ARG;
  const Shape sh = shape_of(&dt);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  uint16_t* ob = static_cast<uint16_t*>(out);
  // Prepared scales (moe_prepare_weights) select the tensor-core launch (1-128
  // tokens); without them, steps of more than 16 tokens and a folded shared
  // expert take the batched path.
  if (fused_decode_tc_supported(sh, ex))
    return cuda_status(launch_fused_decode_tc(sh, ex, shd, w_router, bias, xb, ob, topk_ids, topk_w, ws,
                                              g_wait_limit_ns.load(), s, desc->shared_in_table, desc->score_func));
  // The CUDA-core single launch streams weight rows in 64-element pairs (32-byte
  // code loads, 2- or 4-byte scale loads): shapes with H or I not a multiple of
  // 64 take the per-step kernels, which work in 32-element blocks.
  if (desc->shared_in_table || !fused_decode_supported(sh))
    return run_forward(desc, ex, shd, w_router, bias, xb, ob, topk_ids, topk_w, ws, s);
  return cuda_status(launch_fused_decode(sh, ex, shd, w_router, bias, xb, ob, topk_ids, topk_w, ws,
                                         g_wait_limit_ns.load(), s, desc->score_func));
}

}  // extern "C"
