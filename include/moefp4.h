/*
 * moefp4.h -- C ABI of libmoefp4, a block-scaled FP4 sparse MoE FFN layer for
 * NVIDIA GB300 (sm_103a).
 *
 * The layer (AMD technical article "MiniMax-M3.1 on AMD Instinct GPUs: Day-0
 * support and optimization", section "MiniMax-M3.1 at a glance"): a
 * high-precision router over E routed experts with top-k selection, an
 * always-on shared expert, routed SwiGLU experts whose gate/up and down
 * projections are block-scaled FP4, and a weighted combine.  Routed-expert
 * weights are OCP MXFP4 (E2M1 codes + one E8M0 scale per 32) or NVFP4 (E2M1 +
 * one E4M3 scale per 16 + an FP32 tensor scale); routed-expert activations are
 * quantised to OCP MXFP4 at run time (model card
 * "amd/MiniMax-M3.1-Flash-Quark-MXFP4", section "Model Overview").
 *
 * Conventions for every entry point:
 *   - Pointers named *_h or documented "host" are host memory; every other
 *     pointer is device memory owned by the caller (moe_copy_rows also takes
 *     pinned host memory).  The library never keeps a pointer beyond the call.
 *   - Work is enqueued on the caller's stream; no entry point synchronises the
 *     host or allocates device memory, except moe_get_status (which copies one
 *     word device-to-host and therefore waits for that copy).
 *   - Scratch memory comes from a caller-provided workspace (ws, ws_bytes) of
 *     at least moe_workspace_size() bytes, 256-byte aligned, zero-filled once
 *     before its first use (the library leaves it ready for the next call).
 *     Calls that share one workspace must not overlap on the device.
 *   - Device pointers to weights, activations and outputs must be 16-byte
 *     aligned (MOE_ERR_INVALID_ARG otherwise).
 *   - Arguments are validated on the host before anything is enqueued; an
 *     invalid call returns an error and enqueues nothing.
 *   - Device-side failures (a dependency wait that exceeded its bound) are
 *     recorded in a status word inside the workspace; read it with
 *     moe_get_status() after the stream has been synchronised.
 *
 * Layouts (row-major, C order, little-endian):
 *   x         BF16 [T, H]
 *   codes     E2M1, two per byte, the low nibble holds the even element
 *   w13       [E, 2I, H/2] codes; rows [0, I) are gate, rows [I, 2I) are up
 *   w13_scale MXFP4: E8M0 [E, 2I, H/32];  NVFP4: E4M3 [E, 2I, H/16]
 *   w2        [E, H, I/2] codes
 *   w2_scale  MXFP4: E8M0 [E, H, I/32];   NVFP4: E4M3 [E, H, I/16]
 *   tensor_scale  NVFP4 only: FP32 [E, 3] = (gate, up, down) per expert
 *   shared w13    BF16 [2I, H] (gate rows then up rows); shared w2 BF16 [H, I]
 *   w_router  FP32 [E, H]; router bias FP32 [E] (optional)
 *
 * Arithmetic of every entry point (and of the layer as a whole):
 *   logits = x . Wr^T + bias                       (FP32 accumulation)
 *   p = softmax(logits); ids = top-k by logit (ties: lower expert index),
 *   weights = p[ids] / sum p[ids]
 *   xq = MXFP4(x): per 32 along H, X = 2^(floor(log2 amax) - 2) clamped to
 *        [2^-127, 2^127], codes = E2M1 nearest-even of v / X, clamped to 6,
 *        a zero result is code 0
 *   routed expert e on xq:  G, U = deq(xq) . deq(Wgate/up[e])^T  (FP32)
 *        h = SiLU(G) * U; hq = MXFP4(h) per 32 along I;  y = deq(hq) . deq(W2[e])^T
 *   shared expert on x:     G, U = x . Ws_gate/up^T (FP32); h = BF16(SiLU(G) * U);
 *        ys = h . Ws2^T
 *        (folded into the table, shared_in_table = 1: ys = the routed-expert
 *        arithmetic above with table entry E)
 *   out = BF16(ys + sum_j weights_j * y_j)
 */
#ifndef MOEFP4_H
#define MOEFP4_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* An opaque CUDA stream (the runtime's cudaStream_t); NULL = legacy stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* bad pointer, shape, alignment or format    */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but outside this entry point's range */
  MOE_ERR_CUDA = 3,         /* a CUDA runtime call failed                 */
  MOE_ERR_TIMEOUT = 4,      /* a device-side wait exceeded its bound      */
  MOE_ERR_WORKSPACE = 5     /* workspace missing, too small or misaligned */
} moe_status_t;

typedef enum { MOE_W_MXFP4 = 1, MOE_W_NVFP4 = 2 } moe_wfmt_t;

/* Shape of one MoE layer call.
 * T tokens (>= 0), hidden size H, intermediate size I, E routed experts,
 * top_k experts per token.  Requirements: H and I multiples of 32 (whole
 * MXFP4 activation blocks; NVFP4 weights then hold whole 16-element blocks
 * too), 1 <= top_k <= 8, top_k <= E <= 256.  The tensor-core paths run where
 * their tiles divide the shape (H and I multiples of 256 for the routed
 * experts and the fused decode; moe_prepare_weights needs multiples of 128);
 * every other shape runs on CUDA cores with the same arithmetic.  renormalize must be 1
 * (weights renormalised over the selected experts) and act_quant must be 1
 * (routed-expert activations quantised to MXFP4); other values return
 * MOE_ERR_UNSUPPORTED.
 *
 * shared_in_table = 1 folds the shared expert into the routed-expert table
 * (model card "amd/MiniMax-M3.1-Flash-Quark-MXFP4", section "Experimental
 * MXFP4 shared experts"; AMD article, section "Performance, mono decode on vs
 * off"): the expert arrays then hold E + 1 experts in the same FP4 format,
 * and expert E is the shared expert, applied to every token with weight 1 on
 * the same MXFP4 activations as a routed expert.  The router still has E
 * rows and picks top_k of them (topk outputs stay [T, top_k]); the BF16
 * shared expert must then be absent.  Needs top_k + 1 <= 8 and E + 1 <= 256.
 * moe_layer_decode, moe_layer_decode_noalloc, moe_layer_forward,
 * moe_workspace_size, moe_prepare_weights and moe_convert_nvfp4_to_mxfp4 take
 * it (the last two act on all E + 1 experts); the per-step entry points
 * return MOE_ERR_UNSUPPORTED (call them with the table shape, E + 1 experts
 * and top_k + 1 assignments, instead).  0 = no folded shared expert.
 *
 * score_func picks the router's score function (the pages only call the
 * router high precision: AMD article, section "MiniMax-M3.1 at a glance"):
 *   0 = softmax: the bias, when given, is added to the logits; the top_k
 *       largest logits are selected, weighted by their softmax probabilities
 *       renormalised over the selection;
 *   1 = sigmoid with a bias-corrected choice: scores s = sigmoid(x . Wr^T);
 *       the top_k largest s + bias are selected (the bias only corrects the
 *       choice), weighted by s_selected / sum s_selected.
 * Ties go to the lower expert index in both.  Other values return
 * MOE_ERR_INVALID_ARG. */
typedef struct {
  int32_t T, H, I, E, top_k;
  int32_t renormalize;
  int32_t act_quant;
  int32_t shared_in_table;
  int32_t score_func;
} moe_layer_desc_t;

/* Routed-expert weights (device pointers, layouts above).  The two *_mma
 * fields are optional copies of the scale bytes in the tensor-core layout
 * written by moe_prepare_weights (NULL = not prepared). */
typedef struct {
  moe_wfmt_t fmt;
  const uint8_t* w13;
  const uint8_t* w13_scale;
  const uint8_t* w2;
  const uint8_t* w2_scale;
  const float* tensor_scale;   /* NVFP4: [E, 3]; MXFP4: must be NULL */
  const uint8_t* w13_scale_mma;
  const uint8_t* w2_scale_mma;
} moe_experts_t;

/* The BF16 shared expert; both NULL = the layer has no shared expert. */
typedef struct {
  const void* w13;  /* BF16 [2I, H] */
  const void* w2;   /* BF16 [H, I]  */
} moe_shared_bf16_t;

/* An MXFP8 shared expert (OCP MX: E4M3 elements, one E8M0 scale per 32
 * along K), the format the pages' fused decode runs the shared expert in.
 * The two *_mma fields are optional copies of the scales in the tensor-core
 * layout written by moe_prepare_shared_mxfp8 (NULL = re-laid on every call). */
typedef struct {
  const uint8_t* w13;        /* E4M3 [2I, H] (gate rows then up rows), 16-byte aligned */
  const uint8_t* w13_scale;  /* E8M0 [2I, H/32], 4-byte aligned */
  const uint8_t* w2;         /* E4M3 [H, I], 16-byte aligned */
  const uint8_t* w2_scale;   /* E8M0 [H, I/32], 4-byte aligned */
  const uint8_t* w13_scale_mma;
  const uint8_t* w2_scale_mma;
} moe_shared_mxfp8_t;

/* Human-readable name of a status code (static storage). */
MOE_API const char* moe_status_string(moe_status_t st);

/* Bytes of workspace any entry point below needs for this layer shape
 * (the maximum over all of them).  desc must be valid. */
MOE_API moe_status_t moe_workspace_size(const moe_layer_desc_t* desc, size_t* bytes);

/* Load-time re-layout of expert scales for the tensor-core paths (the pages
 * convert expert weights at load time: AMD article, section "Enabling the
 * MXFP4 checkpoint with the AMD Quark"; vLLM PR #64273, section "Purpose").
 * Writes the scale bytes of W13 and W2 again, in blocks of 128 rows x 128 K
 * elements (MXFP4, E8M0 per 32) or 128 rows x 64 K elements (NVFP4, E4M3 per
 * 16): 512 bytes each, word (i, j) at byte 16 i + 4 j holding the 4 scales of
 * row 32 j + i, block order [E][rows/128][K blocks]; the same byte counts as
 * the canonical scales:
 *   w13_scale_mma  out, E * 2I * H/32 (MXFP4) or E * 2I * H/16 (NVFP4) bytes
 *   w2_scale_mma   out, E * H * I/32 (MXFP4) or E * H * I/16 (NVFP4) bytes
 * (16-byte aligned; the canonical scales 4-byte aligned).  H and I must be
 * multiples of 128 (else MOE_ERR_UNSUPPORTED).  Point
 * experts->w13_scale_mma / w2_scale_mma at them afterwards: moe_layer_decode
 * then runs its contractions on tensor cores (when H and I are multiples of
 * 256), and the MXFP4 batched path skips its per-call re-layout. */
MOE_API moe_status_t moe_prepare_weights(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                         uint8_t* w13_scale_mma, uint8_t* w2_scale_mma, moe_stream_t stream);

/* Load-time conversion of NVFP4 routed experts to OCP MXFP4 (the pages convert
 * NVFP4 checkpoints to MXFP4 before serving: AMD article, section "Enabling
 * the MXFP4 checkpoint with the AMD Quark"; vLLM PR #64273, section
 * "Purpose").  Per 32-element block the exact values code x E4M3 scale x FP32
 * tensor scale (gate, up and down scales of experts->tensor_scale [E, 3]) are
 * requantised with the MXFP4 rule of moe_quant_act_mxfp4; every decision is
 * taken in exact arithmetic.  experts must be NVFP4 (else
 * MOE_ERR_INVALID_ARG).  Outputs, caller-allocated (codes 16-byte aligned):
 *   w13_out [E, 2I, H/2], w13_scale_out [E, 2I, H/32],
 *   w2_out  [E, H, I/2],  w2_scale_out  [E, H, I/32]. */
MOE_API moe_status_t moe_convert_nvfp4_to_mxfp4(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                                uint8_t* w13_out, uint8_t* w13_scale_out, uint8_t* w2_out,
                                                uint8_t* w2_scale_out, moe_stream_t stream);

/* Reads (and clears) the device status word of a workspace into *st.  Call
 * after synchronising the stream the workspace was used on.  This is the one
 * entry point that waits: it copies 4 bytes device-to-host. */
MOE_API moe_status_t moe_get_status(void* ws, moe_status_t* st);

/* A1 + A2: router logits, scores, top-k, renormalisation (desc->score_func).
 * The router is "high precision" and "stacked" (AMD article, sections
 * "MiniMax-M3.1 at a glance" and "What we Optimized"): FP32 weights, FP32
 * accumulation.
 *   x         BF16 [T, H]
 *   w_router  FP32 [E, H];  bias FP32 [E] or NULL
 *   topk_ids  int32 [T, top_k] out, descending logit, ties to lower index
 *   topk_w    FP32 [T, top_k] out, the renormalised weights
 *   logits    FP32 [T, E] out, or NULL: x . Wr^T + bias (softmax scoring) or
 *             the raw x . Wr^T (sigmoid scoring)
 * ws: workspace for desc. */
MOE_API moe_status_t moe_router_topk(const moe_layer_desc_t* desc, const void* x, const float* w_router,
                             const float* bias, int32_t* topk_ids, float* topk_w, float* logits,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* A4: dynamic OCP MXFP4 quantisation of BF16 rows (model card, section
 * "Model Overview": routed-expert activations "OCP MXFP4, Dynamic").
 *   x      BF16 [rows, K], K a multiple of 32, row pitch K elements
 *   codes  uint8 [rows, K/2] out;  scales  uint8 E8M0 [rows, K/32] out
 * Non-finite inputs give unspecified codes. */
MOE_API moe_status_t moe_quant_act_mxfp4(int32_t rows, int32_t K, const void* x, uint8_t* codes,
                                 uint8_t* scales, moe_stream_t stream);

/* Dynamic OCP MXFP8 quantisation of BF16 rows: E4M3 elements with one E8M0
 * scale per 32, X = 2^(floor(log2 amax) - 8), elements nearest-even E4M3
 * saturated to +-448, a zero result +0 (the format of the pages' MXFP8
 * shared expert: AMD article, section "What we Optimized").
 *   x      BF16 [rows, K], K a multiple of 32
 *   codes  uint8 E4M3 [rows, K] out (8-byte aligned);  scales  uint8 E8M0 [rows, K/32] out
 * Non-finite inputs give unspecified codes. */
MOE_API moe_status_t moe_quant_act_mxfp8(int32_t rows, int32_t K, const void* x, uint8_t* codes,
                                         uint8_t* scales, moe_stream_t stream);

/* Lossless MXFP8 -> BF16 dequantising copy (vLLM PR #64273, section
 * "Purpose": an E4M3 value times a power-of-two scale is exact in BF16, so an
 * MXFP8 checkpoint tensor dequantises to BF16 without rounding):
 *   out[r, c] = BF16(E4M3(codes[r, c]) * 2^(scales[r, c / 32] - 127))
 * with one rounding, to nearest even, which changes nothing where the value
 * lies in BF16's normal range (BF16 keeps 8 significant bits, E4M3 has at
 * most 4); below it BF16 subnormals round, at or above 2^128 the result is
 * +-inf, and a NaN code or the E8M0 NaN byte 0xFF gives NaN.
 *   codes   uint8 E4M3 [rows, K] (8-byte aligned), K a multiple of 32
 *   scales  uint8 E8M0 [rows, K/32]
 *   out     BF16 [rows, K] (16-byte aligned)
 * Meant for load time (for example an MXFP8 shared expert kept as BF16). */
MOE_API moe_status_t moe_dequant_mxfp8_to_bf16(int32_t rows, int32_t K, const uint8_t* codes,
                                               const uint8_t* scales, void* out, moe_stream_t stream);

/* A3: stable counting sort of the T*top_k (token, slot) assignments by
 * expert: the token-to-expert permutation and per-expert histogram by which
 * a fused MoE groups its work, each expert running on the tokens routed to
 * it (AMD article, section "What we Optimized": the MXFP4 fused MoE; section
 * "MiniMax-M3.1 at a glance": 4 of 128 routed experts active per token).
 * Bit-exact and deterministic.
 *   topk_ids  int32 [T, top_k]  (every id in [0, E))
 *   counts    int32 [E] out;  offsets int32 [E+1] out (exclusive prefix sum)
 *   perm      int32 [T*top_k] out: sorted position -> t*top_k + j, ordered by
 *             expert, then token, then slot
 *   inv_perm  int32 [T*top_k] out: t*top_k + j -> sorted position
 * ws: workspace for desc.  Out-of-range ids give unspecified results. */
MOE_API moe_status_t moe_permute(const moe_layer_desc_t* desc, const int32_t* topk_ids, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv_perm, void* ws,
                         size_t ws_bytes, moe_stream_t stream);

/* A5 - A8: routed expert FFNs on the permuted MXFP4 activations plus the BF16
 * shared expert (AMD article, section "What we Optimized": the MXFP4 fused MoE
 * with the shared expert).
 *   x         BF16 [T, H]   (shared expert input; may be NULL if no shared)
 *   xq, xs    MXFP4 of x in token order: uint8 [T, H/2], E8M0 [T, H/32]
 *   offsets   int32 [E+1], perm int32 [T*top_k]  (from moe_permute)
 *   y_assign  FP32 [T*top_k, H] out, row p = expert output of sorted
 *             assignment p (unweighted)
 *   y_shared  FP32 [T, H] out (NULL iff the layer has no shared expert)
 * ws: workspace for desc. */
MOE_API moe_status_t moe_expert_ffn_fp4(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                const moe_shared_bf16_t* shared, const void* x,
                                const uint8_t* xq, const uint8_t* xs, const int32_t* offsets,
                                const int32_t* perm, float* y_assign, float* y_shared, void* ws,
                                size_t ws_bytes, moe_stream_t stream);

/* A8 with an MXFP8 shared expert (AMD article, section "What we Optimized":
 * the fused decode runs the shared expert in MXFP8), on tcgen05
 * kind::mxf8f6f4 tensor cores:
 *   xq = MXFP8(x) per 32 along H (moe_quant_act_mxfp8's rule);
 *   G, U = deq(xq) . deq(W13 gate / up)^T (FP32); h = SiLU(G) * U;
 *   hq = MXFP8(h) per 32 along I;  y_shared = deq(hq) . deq(W2)^T (FP32 [T, H]).
 * Needs H and I multiples of 256 (else MOE_ERR_UNSUPPORTED) and the
 * workspace of desc (its per-call scratch, which the next call of any entry
 * point may reuse); desc->shared_in_table must be 0.  The combine takes
 * y_shared as for the BF16 shared expert. */
MOE_API moe_status_t moe_shared_expert_mxfp8(const moe_layer_desc_t* desc, const moe_shared_mxfp8_t* shared,
                                             const void* x, float* y_shared, void* ws, size_t ws_bytes,
                                             moe_stream_t stream);

/* Load-time re-layout of an MXFP8 shared expert's scales for the tensor
 * cores (the same 512-byte blocks as moe_prepare_weights over 128 rows x 128
 * K elements):
 *   w13_scale_mma  out, 2I * H/32 bytes;  w2_scale_mma  out, H * I/32 bytes
 * (16-byte aligned).  H and I multiples of 256 (else MOE_ERR_UNSUPPORTED).
 * Point shared->w13_scale_mma / w2_scale_mma at them afterwards. */
MOE_API moe_status_t moe_prepare_shared_mxfp8(const moe_layer_desc_t* desc, const moe_shared_mxfp8_t* shared,
                                              uint8_t* w13_scale_mma, uint8_t* w2_scale_mma, moe_stream_t stream);

/* A9: weighted combine (vLLM PR #64273 commit list: "MoE finalize").
 *   out[t] = BF16(y_shared[t] + sum_j topk_w[t, j] * y_assign[inv_perm[t*k + j]])
 *   y_shared may be NULL (treated as 0).  out BF16 [T, H]. */
MOE_API moe_status_t moe_combine(const moe_layer_desc_t* desc, const float* y_assign,
                         const int32_t* inv_perm, const float* topk_w, const float* y_shared,
                         void* out, moe_stream_t stream);

/* A10: the whole layer in one launch for decode steps of 1 to 16 tokens
 * (AMD article, section "What we Optimized": one fused launch per MoE layer
 * for pure decode steps of at most 16 tokens), and for wider steps of 17 to
 * 128 tokens (the article's section "What's next": wider mono steps).
 * T > 128 returns MOE_ERR_UNSUPPORTED (use moe_layer_forward).
 *   x          BF16 [T, H];  out BF16 [T, H]
 *   topk_ids   int32 [T, top_k] out or NULL;  topk_w FP32 [T, top_k] out or NULL
 * The launch is persistent (one block per SM); its dependency waits are
 * bounded and report MOE_ERR_TIMEOUT through moe_get_status.  One launch
 * needs the routed experts' prepared scales (moe_prepare_weights) and H, I
 * multiples of 256 for 17-128 tokens; up to 16 tokens, H and I multiples of
 * 64 also run in one launch on CUDA cores.  Other cases run as the per-step
 * sequence of moe_layer_forward (same arithmetic, several launches).  The
 * output is bit-reproducible run to run on the one-launch paths. */
MOE_API moe_status_t moe_layer_decode(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                              const moe_shared_bf16_t* shared, const float* w_router,
                              const float* bias, const void* x, void* out, int32_t* topk_ids,
                              float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_layer_decode with the shared expert in MXFP8 (AMD article, section
 * "What we Optimized": the fused decode runs the shared expert in MXFP8),
 * 1 to 128 tokens.  The shared expert's arithmetic is moe_shared_expert_mxfp8's
 * (x and h quantised to MXFP8 per 32, E4M3 x E4M3 on kind::mxf8f6f4 tensor
 * cores).  One launch when the routed experts' scales and shared->w13_scale_mma
 * / w2_scale_mma are prepared (moe_prepare_weights, moe_prepare_shared_mxfp8),
 * else the batched path of moe_layer_forward_shared_mxfp8.  H and I multiples
 * of 256 (else MOE_ERR_UNSUPPORTED); desc->shared_in_table must be 0; T > 128
 * returns MOE_ERR_UNSUPPORTED.  Arguments and errors as moe_layer_decode. */
MOE_API moe_status_t moe_layer_decode_shared_mxfp8(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                                   const moe_shared_mxfp8_t* shared, const float* w_router,
                                                   const float* bias, const void* x, void* out, int32_t* topk_ids,
                                                   float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Trace builds only (libmoefp4_trace.so, compiled with MOEFP4_TRACE=1): the
 * per-block %globaltimer stamps (ns) of the last single-launch decode,
 * uint64 [256 blocks][16 events], events in the order start, router done,
 * routing built, x quantised, x seen, shared h seen, routed h seen, producer
 * done, units done, down parts seen, end, last SGU / RGU / SDN / RDN unit;
 * then uint64 [320 expert slots][8]: first (stored as ~t) and last hand-out
 * of the slot's routed gate/up units, last gate/up unit done, h ready, first
 * (~t) and last hand-out of its down units, last down unit stored, and
 * expert << 8 | rows (0: slot not reached).  Copies min(bytes, 53248) bytes
 * to host memory dst; dst NULL clears both.  Other builds return
 * MOE_ERR_UNSUPPORTED. */
MOE_API moe_status_t moe_debug_decode_trace(uint64_t* dst, size_t bytes);

/* The whole layer for any T, as the sequence router -> quantise -> permute ->
 * expert FFNs -> combine: the standard path the pages run outside the fused
 * decode range, i.e. prefill and decode steps of more than 16 tokens (AMD
 * article, section "What we Optimized": the stacked router GEMM, then the
 * MXFP4 fused MoE with the shared expert; the single fused launch is kept for
 * pure decode steps of at most 16 tokens).  Arguments, layouts and results
 * as for moe_layer_decode; every T >= 0 is accepted. */
MOE_API moe_status_t moe_layer_forward(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                               const moe_shared_bf16_t* shared, const float* w_router,
                               const float* bias, const void* x, void* out, int32_t* topk_ids,
                               float* topk_w, void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_layer_forward with the shared expert in MXFP8 (AMD article, section
 * "What we Optimized": the shared expert runs in MXFP8), on kind::mxf8f6f4
 * tensor cores with the arithmetic of moe_shared_expert_mxfp8 (the token and
 * h quantised to MXFP8 per 32), weight 1 in the combine.  Needs H and I
 * multiples of 256 and desc->shared_in_table = 0 (else MOE_ERR_UNSUPPORTED /
 * MOE_ERR_INVALID_ARG); every other argument as for moe_layer_forward. */
MOE_API moe_status_t moe_layer_forward_shared_mxfp8(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                                    const moe_shared_mxfp8_t* shared, const float* w_router,
                                                    const float* bias, const void* x, void* out,
                                                    int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
                                                    moe_stream_t stream);

/* Size of the scratch array built into the library for
 * moe_layer_decode_noalloc (8 MiB, held on every GPU that loads the library
 * until the process exits). */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/* moe_layer_decode without a caller workspace.  The paper has no counterpart
 * to this entry point; it exists for callers that cannot hand the library
 * device memory: a plain C host program that links only this library and the
 * CUDA runtime and keeps no device allocator of its own, or a plugin inside a
 * host framework whose memory pool does not allow outside device
 * allocations.  It allocates nothing: its scratch is a fixed array inside the
 * library (MOE_NOALLOC_SCRATCH_BYTES).  Inputs, outputs and results are
 * exactly those of moe_layer_decode.
 *   - Shapes whose moe_workspace_size exceeds MOE_NOALLOC_SCRATCH_BYTES - 256
 *     (the array's last 256 bytes keep a sticky status word), and T > 16,
 *     return MOE_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on a device looks up that device's scratch address (with
 *     the device current); make that first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps what the
 *     previous call left; each call clears the part that must start at zero
 *     (one extra small kernel on the stream).  Calls whose launches may overlap on
 *     the GPU (different streams, no ordering between them) race on it.
 *   - A device-side wait that runs out records MOE_ERR_TIMEOUT (the call's
 *     output is then unfinished).  Each call first moves a failure left by the
 *     previous call into the sticky word, where it stays until
 *     moe_noalloc_get_status reads it; call that after synchronising the
 *     stream. */
MOE_API moe_status_t moe_layer_decode_noalloc(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                              const moe_shared_bf16_t* shared, const float* w_router,
                                              const float* bias, const void* x, void* out, int32_t* topk_ids,
                                              float* topk_w, moe_stream_t stream);

/* Reads (and clears) the device status word of the built-in scratch array of
 * moe_layer_decode_noalloc on the current device into *st: MOE_OK, or
 * MOE_ERR_TIMEOUT when a call since the last read had a device-side wait run
 * out (its output is then unfinished); both the last call's word and the
 * sticky word are read and cleared.  Call after synchronising the streams
 * of those calls; like moe_get_status it waits for a 4-byte device-to-host
 * copy.  The paper has no counterpart to this entry point either. */
MOE_API moe_status_t moe_noalloc_get_status(moe_status_t* st);

/* Upper bound, in nanoseconds, of every device-side dependency wait of later
 * launches in this process (default 500 ms).  A wait that runs out records
 * MOE_ERR_TIMEOUT in the workspace status word and the launch returns without
 * finishing its work; the workspace must then be zero-filled again. */
MOE_API void moe_set_wait_limit_ns(uint64_t ns);

/* Orientation of the routed-expert tensor-core GEMMs of later
 * moe_expert_ffn_fp4 / moe_layer_forward calls in this process (MXFP4
 * experts, from 256 assignments): 0 = automatic (the default: weights as A
 * when the average expert has at most 32 assignments), 1 = 128-token tiles as
 * the MMA's A operand, 2 = 128 weight rows as A and up to 64 of an expert's
 * tokens as B.  Results agree within rounding; the choice only moves time.
 * Other values return MOE_ERR_INVALID_ARG and change nothing. */
MOE_API moe_status_t moe_set_routed_gemm(int32_t mode);

/* Copies bytes (a multiple of 16, both pointers 16-byte aligned) from src
 * to dst on the stream, moved by the GPU's SMs rather than a copy engine.
 * Each pointer is device memory or pinned host memory that the GPU can
 * address (cudaHostAlloc / cudaHostRegister; on a Grace-Blackwell node the
 * CPU-GPU link carries the loads and stores); the whole range must lie in one
 * allocation.  Meant for a decode step's token rows and outputs, a few KB
 * each way, captured in a CUDA graph with moe_layer_decode, where a kernel
 * costs less than a copy-engine transfer.  Other memory kinds return
 * MOE_ERR_INVALID_ARG. */
MOE_API moe_status_t moe_copy_rows(void* dst, const void* src, size_t bytes, moe_stream_t stream);

/* Test hook: copies the MXFP4-requantised intermediate h of the last
 * moe_expert_ffn_fp4 / moe_layer_forward call made with this workspace (A6)
 * into caller buffers in sorted-assignment order: codes [T*top_k, I/2] and
 * E8M0 scales [T*top_k, I/32].  Enqueued on the stream; needs nothing but the
 * workspace of that call. */
MOE_API moe_status_t moe_debug_requantized_h(const moe_layer_desc_t* desc, const void* ws, size_t ws_bytes,
                                             uint8_t* hq, uint8_t* hs, moe_stream_t stream);

/* Test hook: copies the MXFP8 shared expert's requantised h of the last call
 * that ran it with this workspace (moe_shared_expert_mxfp8 or
 * moe_layer_forward_shared_mxfp8): E4M3 codes [T, I] into hq and the E8M0
 * scales, in their tensor-core layout, [ceil(T/128)][I/128][512] bytes into
 * hs (word (i, j) of a block at byte 16 i + 4 j holds the four scales of row
 * 32 j + i for 128 consecutive columns).  Enqueued on the stream. */
MOE_API moe_status_t moe_debug_shared_mxfp8_h(const moe_layer_desc_t* desc, const void* ws, size_t ws_bytes,
                                              uint8_t* hq, uint8_t* hs, moe_stream_t stream);

/* Test hook for the failure path: launches one bounded wait on a workspace
 * counter that nothing ever advances, with the given limit.  Afterwards
 * moe_get_status reports MOE_ERR_TIMEOUT; the GPU context stays usable. */
MOE_API moe_status_t moe_debug_wait_probe(void* ws, size_t ws_bytes, uint64_t limit_ns, moe_stream_t stream);

/* The same probe on the built-in scratch array of moe_layer_decode_noalloc
 * (current device): afterwards moe_noalloc_get_status reports
 * MOE_ERR_TIMEOUT, also across moe_layer_decode_noalloc calls made in between. */
MOE_API moe_status_t moe_debug_wait_probe_noalloc(uint64_t limit_ns, moe_stream_t stream);

/* Instrumentation: the number of kernels this library has enqueued in this
 * process so far (launches captured into a CUDA graph count once, at
 * capture).  No counterpart on the pages. */
MOE_API void moe_debug_launch_count(uint64_t* n);

/* Instrumentation: two CUDA events (cudaEvent_t, created by the caller; NULL
 * = off) that later moe_expert_ffn_fp4 / moe_layer_forward calls whose routed
 * experts run on tensor cores record on their stream right before the routed
 * gate/up GEMM and right after the routed down GEMM, so the caller can time
 * the two block-scaled FP4 contractions alone (the prefill FP4 tensor-core
 * rate).  Inside a stream capture they become external event nodes of the
 * graph.  Process-wide, like moe_set_routed_gemm.  No counterpart on the
 * pages. */
MOE_API void moe_set_timing_events(void* routed_gemm_begin, void* routed_gemm_end);

#ifdef __cplusplus
}
#endif

#endif /* MOEFP4_H */
