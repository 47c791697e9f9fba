// A10: the whole MoE layer in one persistent launch for decode steps of 1-16
// tokens (AMD technical article "MiniMax-M3.1 on AMD Instinct GPUs", section
// "What we Optimized": "mono decode" runs each MoE layer as one fused launch
// for pure decode steps of at most 16 tokens).
//
// Design.  The layer is cut into work units handed out in a fixed order
// through a global counter:
//   router rows (1 expert row each)          -> logits
//   quantise x to MXFP4                      -> xq, xs
//   shared-expert gate/up (8 columns each)   -> h_shared (BF16)
//   routed gate/up (expert slot, 32 columns) -> hq, hs (SwiGLU + MXFP4 epilogue)
//   down + combine (32 rows of H each)       -> out (BF16)
// A unit only waits for units earlier in the order (routed gate/up waits for
// the router and the quantiser, down waits for every gate/up unit), and a
// block only waits on a unit it has already been handed, so the earliest
// unfinished unit always makes progress: the launch needs no co-residency
// guarantee.  Blocks that finish the routing-independent work early keep
// streaming the shared expert while the router completes, which hides the
// router's latency.  Every wait is bounded (MOE_DEV_TIMEOUT in the status
// word) and the last block to leave resets the counters for the next call.
//
// Each block computes the routing of all T tokens itself once the router rows
// are done (a few hundred logits), so no extra hand-off is needed; the output
// of the combine is summed in a fixed order and is bit-reproducible.
#include "expert_units.cuh"
#include "kernels.h"
#include "routing.cuh"

namespace moefp4 {
namespace {

constexpr int FT = 512;         // threads per block
constexpr int FW = FT / 32;     // warps per block
constexpr int MAXN = MAX_DECODE_T * MAX_TOPK;  // assignments

struct FusedArgs {
  Shape sh;
  ExpertsDev ex;
  SharedDev shd;
  const float* wr;
  const float* bias;
  const uint16_t* x;
  uint16_t* out;
  int* ids_out;
  float* w_out;
  int* ctr;
  float* logits;
  uint8_t* xq;
  uint8_t* xs;
  uint8_t* hq;
  uint8_t* hs;
  uint16_t* h_shared;
  uint64_t wait_limit_ns;
  int score;  // SCORE_SOFTMAX (the bias is part of the logit) or SCORE_SIGMOID
  // unit ranges
  int u_quant, u_sgu, u_rgu, u_down, u_end;
  // dynamic shared memory offsets
  int off_x, off_xq, off_xsc, off_gu, off_hq, off_hsc, off_hsh, off_y;
};

// Per-block routing tables (static shared memory).
struct Routing {
  int ids[MAXN];        // flat assignment a = t*k + j -> expert
  float w[MAXN];        // renormalised weight
  int sorted[MAXN];     // sorted position -> a
  int inv[MAXN];        // a -> sorted position
  int tok[MAXN];        // sorted position -> token
  int slot_e[MAXN];     // slot -> expert (distinct experts, ascending)
  int slot_beg[MAXN + 1];
  int cnt[MAX_E];
  int eoff[MAX_E];
  int eslot[MAX_E];
  int n_slots;
};

__device__ __forceinline__ void publish(int* ctr_slot) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd(ctr_slot, 1);
}

// Thread 0 waits, the block learns the outcome.
__device__ __forceinline__ bool block_wait(const FusedArgs& a, int which, int target, int* flag_s) {
  if (threadIdx.x == 0) *flag_s = wait_at_least(a.ctr + which, target, a.ctr + C_STATUS, a.wait_limit_ns);
  __syncthreads();
  const bool ok = *flag_s;
  __syncthreads();
  return ok;
}

// Top-k of every token (warp t), then the stable counting sort of the T*k
// assignments by expert and the list of distinct experts.
__device__ void build_routing(const FusedArgs& a, Routing& R) {
  const int T = a.sh.T, E = a.sh.E, k = a.sh.k, n = T * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += FT) R.cnt[e] = 0;
  if (warp < T) {
    float v[8];
    load_logit_row(a.logits + (size_t)warp * E, E, v, true);
    int sel[MAX_TOPK];
    float w[MAX_TOPK];
    route_row(v, E, k, a.score, a.bias, sel, w);
    if (lane < k) {
#pragma unroll
      for (int j = 0; j < MAX_TOPK; ++j)
        if (j == lane) {
          R.ids[warp * k + j] = sel[j];
          R.w[warp * k + j] = w[j];
        }
    }
  }
  __syncthreads();
  int e = -1, rank = 0;
  if (threadIdx.x < n) {
    e = R.ids[threadIdx.x];
    for (int b = 0; b < threadIdx.x; ++b) rank += R.ids[b] == e;
    atomicAdd(&R.cnt[e], 1);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scans over experts of counts and presence
    int run_c = 0, run_p = 0;
    for (int base = 0; base < E; base += 32) {
      const int ex = base + lane;
      const int c = ex < E ? R.cnt[ex] : 0;
      int ic = c, ip = c > 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yc = __shfl_up_sync(FULL, ic, o), yp = __shfl_up_sync(FULL, ip, o);
        if (lane >= o) { ic += yc; ip += yp; }
      }
      if (ex < E) {
        R.eoff[ex] = run_c + ic - c;
        R.eslot[ex] = run_p + ip - (c > 0);
      }
      run_c += __shfl_sync(FULL, ic, 31);
      run_p += __shfl_sync(FULL, ip, 31);
    }
    if (lane == 0) {
      R.n_slots = run_p;
      R.slot_beg[run_p] = n;
    }
  }
  __syncthreads();
  if (threadIdx.x < n) {
    const int p = R.eoff[e] + rank;
    R.sorted[p] = threadIdx.x;
    R.inv[threadIdx.x] = p;
    R.tok[p] = threadIdx.x / k;
  }
  for (int ex = threadIdx.x; ex < E; ex += FT) {
    if (R.cnt[ex] > 0) {
      R.slot_e[R.eslot[ex]] = ex;
      R.slot_beg[R.eslot[ex]] = R.eoff[ex];
    }
  }
  __syncthreads();
}

// Router row e for all tokens: the block's threads stride over H eight
// elements at a time, then a fixed-order reduction over lanes and warps.
template <int MAXT>
__device__ void unit_router(const FusedArgs& a, int e, float* red_s) {
  const int T = a.sh.T, H = a.sh.H;
  float acc[MAXT];
#pragma unroll
  for (int t = 0; t < MAXT; ++t) acc[t] = 0.0f;
  const float* wrow = a.wr + (size_t)e * H;
  for (int k = threadIdx.x * 8; k < H; k += FT * 8) {
    const uint4 wa = ldg_stream(wrow + k), wb = ldg_stream(wrow + k + 4);
#pragma unroll
    for (int t = 0; t < MAXT; ++t) {
      if (t < T) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * H + k));
        float s = acc[t];
        s = fmaf(bf16_lo(q.x), __uint_as_float(wa.x), s);
        s = fmaf(bf16_hi(q.x), __uint_as_float(wa.y), s);
        s = fmaf(bf16_lo(q.y), __uint_as_float(wa.z), s);
        s = fmaf(bf16_hi(q.y), __uint_as_float(wa.w), s);
        s = fmaf(bf16_lo(q.z), __uint_as_float(wb.x), s);
        s = fmaf(bf16_hi(q.z), __uint_as_float(wb.y), s);
        s = fmaf(bf16_lo(q.w), __uint_as_float(wb.z), s);
        s = fmaf(bf16_hi(q.w), __uint_as_float(wb.w), s);
        acc[t] = s;
      }
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < MAXT; ++t) {
    const float v = warp_sum(acc[t]);
    if (lane == 0) red_s[warp * MAXT + t] = v;
  }
  __syncthreads();
  if (threadIdx.x < T) {
    float s = 0.0f;
    for (int w = 0; w < FW; ++w) s += red_s[w * MAXT + threadIdx.x];
    if (a.bias && a.score == SCORE_SOFTMAX) s += a.bias[e];
    a.logits[(size_t)threadIdx.x * a.sh.E + e] = s;
  }
}

// MXFP4 quantisation of all T token rows (same arithmetic as the A4 kernel).
__device__ void unit_quant(const FusedArgs& a) {
  const size_t ngroups = (size_t)a.sh.T * a.sh.H / 8;
  const size_t iters = (ngroups + FT - 1) / FT;
  for (size_t i = 0; i < iters; ++i) {
    const size_t g = i * FT + threadIdx.x;
    quant8_group(a.x, g, g < ngroups, a.xq, a.xs);
  }
}

// Shared-expert gate rows 8u..8u+7 and up rows I+8u.. (one per warp), then
// h = BF16(SiLU(G) U) for the 8 columns.
template <int MAXT>
__device__ void unit_shared_gate_up(const FusedArgs& a, int u, const uint16_t* x_s, float* gu_s) {
  const int T = a.sh.T, H = a.sh.H, I = a.sh.I;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = warp < 8 ? 8 * u + warp : I + 8 * u + (warp - 8);
  stream_bf16_rows<MAXT, 1, 4>(
      1, H, [&](int) { return a.shd.w13 + (size_t)row * H; }, x_s, H, T,
      [&](int, const float(&acc)[MAXT]) {
#pragma unroll
        for (int t = 0; t < MAXT; ++t)
          if (lane == 0) gu_s[warp * MAXT + t] = acc[t];
      });
  __syncthreads();
  if (threadIdx.x < T * 8) {
    const int t = threadIdx.x >> 3, j = threadIdx.x & 7;
    const float h = silu(gu_s[j * MAXT + t]) * gu_s[(8 + j) * MAXT + t];
    a.h_shared[(size_t)t * I + 8 * u + j] = f32_to_bf16_rn(h);
  }
}

// Routed gate/up of distinct-expert slot s, columns 32b..32b+31 (warp w takes
// rows w, w+16 of the gate block and the same of the up block), then SwiGLU +
// MXFP4 requantisation into hq/hs (rows in sorted-assignment order).
template <int MAXT, bool NV>
__device__ void unit_routed_gate_up(const FusedArgs& a, const Routing& R, int s, int b,
                                    const uint8_t* xq_s, const float* xsc_s, float* gu_s) {
  const int H = a.sh.H, I = a.sh.I;
  const int e = R.slot_e[s], beg = R.slot_beg[s], nt = R.slot_beg[s + 1] - beg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t rb = (size_t)H / 2, sb = NV ? H / 16 : H / 32;
  const uint8_t* w13 = a.ex.w13 + (size_t)e * 2 * I * rb;
  const uint8_t* s13 = a.ex.w13s + (size_t)e * 2 * I * sb;
  const float tg = NV ? a.ex.tscale[e * 3 + 0] : 1.0f, tu = NV ? a.ex.tscale[e * 3 + 1] : 1.0f;
  auto local_row = [&](int i) { return warp + FW * i; };  // 0..63: gate 0..31, up 32..63
  auto global_row = [&](int r) { return r < 32 ? 32 * b + r : I + 32 * b + (r - 32); };
  stream_fp4_rows<MAXT, NV, 2, 2>(
      64 / FW, H,
      [&](int i) {
        const int g = global_row(local_row(i));
        return Fp4Src{w13 + g * rb, s13 + g * sb};
      },
      [&](int) { return Fp4Tok{&R.tok[beg], 0, nt}; }, xq_s, H / 2, xsc_s, H / 32,
      [&](int i, const Fp4Tok&, const float(&acc)[MAXT]) {
        const int r = local_row(i);
        const float ts = r < 32 ? tg : tu;
        if (lane == 0) {
#pragma unroll
          for (int t = 0; t < MAXT; ++t) gu_s[r * MAXT + t] = acc[t] * ts;
        }
      });
  __syncthreads();
  for (int t = warp; t < nt; t += FW) {
    const size_t p = (size_t)beg + t;
    swiglu_quant_block(gu_s[lane * MAXT + t], gu_s[(32 + lane) * MAXT + t], a.hq + p * (I / 2) + b * 16,
                       a.hs + p * (I / 32) + b);
  }
}

// Rows 32g..32g+31 of H (warp w takes rows w and w+16): the shared-expert
// down rows and every touched expert's down rows, then
// out = BF16(ys + sum_j w_j y_j) in a fixed order.
template <int MAXT, bool NV>
__device__ void unit_down(const FusedArgs& a, const Routing& R, int g, const uint8_t* hq_s,
                          const float* hsc_s, const uint16_t* hsh_s, float* y_s) {
  const int T = a.sh.T, H = a.sh.H, I = a.sh.I, k = a.sh.k, n = T * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t rb = (size_t)I / 2, sb = NV ? I / 16 : I / 32;
  if (a.shd.w13) {
    stream_bf16_rows<MAXT, 1, 3>(
        32 / FW, I, [&](int i) { return a.shd.w2 + (size_t)(32 * g + warp + FW * i) * I; }, hsh_s, I, T,
        [&](int i, const float(&acc)[MAXT]) {
          if (lane == 0) {
#pragma unroll
            for (int t = 0; t < MAXT; ++t)
              if (t < T) y_s[(n + t) * 32 + warp + FW * i] = acc[t];
          }
        });
  }
  constexpr int RPW = 32 / FW;  // rows per warp
  stream_fp4_rows<MAXT, NV, 4, 1>(
      RPW * R.n_slots, I,
      [&](int i) {
        const int s = i / RPW, row = 32 * g + warp + FW * (i % RPW);
        const int e = R.slot_e[s];
        return Fp4Src{a.ex.w2 + (size_t)e * H * rb + row * rb, a.ex.w2s + (size_t)e * H * sb + row * sb};
      },
      [&](int i) {
        const int s = i / RPW;
        return Fp4Tok{nullptr, R.slot_beg[s], R.slot_beg[s + 1] - R.slot_beg[s]};
      },
      hq_s, I / 2, hsc_s, I / 32,
      [&](int i, const Fp4Tok& rr, const float(&acc)[MAXT]) {
        const int s = i / RPW, r = warp + FW * (i % RPW);
        const float td = NV ? a.ex.tscale[R.slot_e[s] * 3 + 2] : 1.0f;
        if (lane == 0) {
#pragma unroll
          for (int t = 0; t < MAXT; ++t)
            if (t < rr.nt) y_s[(rr.tbase + t) * 32 + r] = acc[t] * td;
        }
      });
  __syncthreads();
  if (threadIdx.x < T * 32) {
    const int t = threadIdx.x >> 5, r = threadIdx.x & 31;
    float acc = a.shd.w13 ? y_s[(n + t) * 32 + r] : 0.0f;
    for (int j = 0; j < k; ++j) acc = fmaf(R.w[t * k + j], y_s[R.inv[t * k + j] * 32 + r], acc);
    a.out[(size_t)t * H + 32 * g + r] = f32_to_bf16_rn(acc);
  }
}

// Thread 0: bulk-prefetch into L2 the weight bytes unit u will stream, so
// that its loads hit L2 while this block still computes the current unit.
// Routed units are prefetched only once this block knows the routing.
__device__ void prefetch_unit(const FusedArgs& a, const Routing& R, bool routed_known, int u) {
  const int H = a.sh.H, I = a.sh.I, nb = I / 32;
  const bool nv = a.ex.nv != 0;
  if (u < a.u_quant) {
    prefetch_l2_bulk(a.wr + (size_t)u * H, 4u * H);
  } else if (u < a.u_sgu) {
  } else if (u < a.u_rgu) {
    const int c = u - a.u_sgu;
    prefetch_l2_bulk(a.shd.w13 + (size_t)8 * c * H, 16u * H);
    prefetch_l2_bulk(a.shd.w13 + (size_t)(I + 8 * c) * H, 16u * H);
  } else if (!routed_known) {
  } else if (u < a.u_down) {
    const int s = (u - a.u_rgu) / nb, b = (u - a.u_rgu) % nb;
    if (s >= R.n_slots) return;
    const int e = R.slot_e[s];
    const size_t rb = (size_t)H / 2, sb = nv ? H / 16 : H / 32;
    const uint8_t* w13 = a.ex.w13 + (size_t)e * 2 * I * rb;
    const uint8_t* s13 = a.ex.w13s + (size_t)e * 2 * I * sb;
    prefetch_l2_bulk(w13 + (size_t)32 * b * rb, (uint32_t)(32 * rb));
    prefetch_l2_bulk(w13 + (size_t)(I + 32 * b) * rb, (uint32_t)(32 * rb));
    prefetch_l2_bulk(s13 + (size_t)32 * b * sb, (uint32_t)(32 * sb));
    prefetch_l2_bulk(s13 + (size_t)(I + 32 * b) * sb, (uint32_t)(32 * sb));
  } else if (u < a.u_end) {
    const int g = u - a.u_down;
    const size_t rb = (size_t)I / 2, sb = nv ? I / 16 : I / 32;
    if (a.shd.w2) prefetch_l2_bulk(a.shd.w2 + (size_t)32 * g * I, 64u * I);
    for (int s = 0; s < R.n_slots; ++s) {
      const int e = R.slot_e[s];
      prefetch_l2_bulk(a.ex.w2 + (size_t)e * H * rb + (size_t)32 * g * rb, (uint32_t)(32 * rb));
      prefetch_l2_bulk(a.ex.w2s + (size_t)e * H * sb + (size_t)32 * g * sb, (uint32_t)(32 * sb));
    }
  }
}

template <int MAXT, bool NV>
__global__ void __launch_bounds__(FT, 1) k_fused_decode(FusedArgs a) {
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ Routing R;
  __shared__ float red_s[FW * MAXT];
  __shared__ int s_unit, s_next, s_flag;
  const int T = a.sh.T, H = a.sh.H, I = a.sh.I, E = a.sh.E, n = T * a.sh.k;
  const int nb = I / 32;
  const int total_gu = (a.u_rgu - a.u_sgu) + (a.u_down - a.u_rgu);
  uint16_t* x_s = reinterpret_cast<uint16_t*>(dsm + a.off_x);
  uint8_t* xq_s = dsm + a.off_xq;
  float* xsc_s = reinterpret_cast<float*>(dsm + a.off_xsc);
  float* gu_s = reinterpret_cast<float*>(dsm + a.off_gu);
  uint8_t* hq_s = dsm + a.off_hq;
  float* hsc_s = reinterpret_cast<float*>(dsm + a.off_hsc);
  uint16_t* hsh_s = reinterpret_cast<uint16_t*>(dsm + a.off_hsh);
  float* y_s = reinterpret_cast<float*>(dsm + a.off_y);
  int have_routing = 0, have_x = 0, have_xq = 0, have_down = 0;  // 1 = ready, -1 = failed

  if (threadIdx.x == 0) s_unit = atomicAdd(a.ctr + C_QUEUE, 1);
  __syncthreads();
  int u = s_unit;
  while (u < a.u_end) {
    __syncthreads();
    if (threadIdx.x == 0) {
      const int nx = atomicAdd(a.ctr + C_QUEUE, 1);
      s_next = nx;
      prefetch_unit(a, R, have_routing > 0, nx);
    }
    if (u < a.u_quant) {
      unit_router<MAXT>(a, u, red_s);
      publish(a.ctr + C_ROUTER);
    } else if (u < a.u_sgu) {
      unit_quant(a);
      publish(a.ctr + C_QUANT);
    } else if (u < a.u_rgu) {
      if (!have_x) {
        const int cnt = T * H / 8;
        for (int i = threadIdx.x; i < cnt; i += FT)
          reinterpret_cast<uint4*>(x_s)[i] = __ldg(reinterpret_cast<const uint4*>(a.x) + i);
        __syncthreads();
        have_x = 1;
      }
      unit_shared_gate_up<MAXT>(a, u - a.u_sgu, x_s, gu_s);
      publish(a.ctr + C_GU);
    } else {
      if (!have_routing) {
        have_routing = block_wait(a, C_ROUTER, E, &s_flag) ? 1 : -1;
        if (have_routing > 0) build_routing(a, R);
      }
      if (u < a.u_down) {
        const int s = (u - a.u_rgu) / nb, b = (u - a.u_rgu) % nb;
        if (have_routing > 0 && s < R.n_slots) {
          if (!have_xq) {
            have_xq = block_wait(a, C_QUANT, 1, &s_flag) ? 1 : -1;
            if (have_xq > 0) {
              for (int i = threadIdx.x; i < T * H / 32; i += FT) {
                reinterpret_cast<uint4*>(xq_s)[i] = __ldcg(reinterpret_cast<const uint4*>(a.xq) + i);
                xsc_s[i] = e8m0_to_f32(__ldcg(a.xs + i));
              }
              __syncthreads();
            }
          }
          if (have_xq > 0) unit_routed_gate_up<MAXT, NV>(a, R, s, b, xq_s, xsc_s, gu_s);
        }
        publish(a.ctr + C_GU);
      } else if (have_routing > 0) {
        if (!have_down) {
          have_down = block_wait(a, C_GU, total_gu, &s_flag) ? 1 : -1;
          if (have_down > 0) {
            for (int i = threadIdx.x; i < n * I / 32; i += FT) {
              reinterpret_cast<uint4*>(hq_s)[i] = __ldcg(reinterpret_cast<const uint4*>(a.hq) + i);
              hsc_s[i] = e8m0_to_f32(__ldcg(a.hs + i));
            }
            if (a.shd.w13)
              for (int i = threadIdx.x; i < T * I / 8; i += FT)
                reinterpret_cast<uint4*>(hsh_s)[i] = __ldcg(reinterpret_cast<const uint4*>(a.h_shared) + i);
            __syncthreads();
          }
        }
        if (have_down > 0) {
          const int g = u - a.u_down;
          unit_down<MAXT, NV>(a, R, g, hq_s, hsc_s, hsh_s, y_s);
          if (g == 0 && threadIdx.x < n) {
            if (a.ids_out) a.ids_out[threadIdx.x] = R.ids[threadIdx.x];
            if (a.w_out) a.w_out[threadIdx.x] = R.w[threadIdx.x];
          }
        }
      }
    }
    __syncthreads();
    u = s_next;
  }
  // The last block out resets the counters for the next call on this workspace.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.ctr + C_EXIT, 1) == (int)gridDim.x - 1) {
      for (int c = C_QUEUE; c <= C_EXIT; ++c) a.ctr[c] = 0;
      __threadfence();
    }
  }
}

__global__ void k_wait_probe(int* ctr, uint64_t limit_ns) {
  if (threadIdx.x == 0) wait_at_least(ctr + C_TEST, 1, ctr + C_STATUS, limit_ns);
}

struct SmemPlan {
  int off_x, off_xq, off_xsc, off_gu, off_hq, off_hsc, off_hsh, off_y, bytes;
};

SmemPlan plan_smem(const Shape& sh, bool shared) {
  auto al = [](int v) { return (v + 15) & ~15; };
  SmemPlan p{};
  const int T = sh.T, H = sh.H, I = sh.I, n = sh.T * sh.k;
  p.off_x = 0;
  p.off_xq = al(p.off_x + (shared ? T * H * 2 : 0));
  p.off_xsc = al(p.off_xq + T * H / 2);
  p.off_gu = al(p.off_xsc + 4 * T * H / 32);
  const int end_gu = p.off_gu + 4 * 64 * MAX_DECODE_T;
  p.off_hq = 0;
  p.off_hsc = al(p.off_hq + n * I / 2);
  p.off_hsh = al(p.off_hsc + 4 * n * I / 32);
  p.off_y = al(p.off_hsh + (shared ? T * I * 2 : 0));
  const int end_down = p.off_y + 4 * (n + T) * 32;
  p.bytes = al(end_gu > end_down ? end_gu : end_down);
  return p;
}

template <int MAXT>
const void* fused_kernel_t(bool nv) {
  return nv ? (const void*)k_fused_decode<MAXT, true> : (const void*)k_fused_decode<MAXT, false>;
}

const void* fused_kernel(int maxt, bool nv) {
  switch (maxt) {
    case 1: return fused_kernel_t<1>(nv);
    case 2: return fused_kernel_t<2>(nv);
    case 4: return fused_kernel_t<4>(nv);
    case 8: return fused_kernel_t<8>(nv);
    default: return fused_kernel_t<16>(nv);
  }
}

}  // namespace

cudaError_t launch_fused_decode(const Shape& sh, const ExpertsDev& ex, const SharedDev& shd,
                                const float* wr, const float* bias, const uint16_t* x, uint16_t* out,
                                int* ids_out, float* w_out, void* ws, uint64_t wait_limit_ns,
                                cudaStream_t s, int score) {
  if (sh.T == 0) return cudaSuccess;
  if (!fused_decode_supported(sh)) return cudaErrorInvalidValue;
  const WsLayout L = ws_layout(sh.T, sh.H, sh.I, sh.E, sh.k);
  uint8_t* base = static_cast<uint8_t*>(ws);
  const bool shared = shd.w13 != nullptr;
  const SmemPlan sp = plan_smem(sh, shared);
  FusedArgs a{};
  a.sh = sh;
  a.ex = ex;
  a.shd = shd;
  a.wr = wr;
  a.bias = bias;
  a.x = x;
  a.out = out;
  a.ids_out = ids_out;
  a.w_out = w_out;
  a.ctr = reinterpret_cast<int*>(base + L.counters);
  a.logits = reinterpret_cast<float*>(base + L.logits);
  a.xq = base + L.xq;
  a.xs = base + L.xs;
  a.hq = base + L.hq;
  a.hs = base + L.hs;
  a.h_shared = reinterpret_cast<uint16_t*>(base + L.h_shared);
  a.wait_limit_ns = wait_limit_ns;
  a.score = score;
  a.u_quant = sh.E;
  a.u_sgu = a.u_quant + 1;
  a.u_rgu = a.u_sgu + (shared ? sh.I / 8 : 0);
  a.u_down = a.u_rgu + sh.T * sh.k * (sh.I / 32);
  a.u_end = a.u_down + sh.H / 32;
  a.off_x = sp.off_x;
  a.off_xq = sp.off_xq;
  a.off_xsc = sp.off_xsc;
  a.off_gu = sp.off_gu;
  a.off_hq = sp.off_hq;
  a.off_hsc = sp.off_hsc;
  a.off_hsh = sp.off_hsh;
  a.off_y = sp.off_y;

  const int maxt = sh.T <= 1 ? 1 : sh.T <= 2 ? 2 : sh.T <= 4 ? 4 : sh.T <= 8 ? 8 : 16;
  const void* fn = fused_kernel(maxt, ex.nv != 0);
  cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, sp.bytes);
  if (err != cudaSuccess) return err;
  int dev = 0, sms = 0, per_sm = 0;
  if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
  if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
  if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, FT, sp.bytes)) != cudaSuccess)
    return err;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int grid = sms * per_sm;
  if (grid > a.u_end) grid = a.u_end;
  void* args[] = {&a};
  return count_launch(), cudaLaunchKernel(fn, dim3(grid), dim3(FT), args, sp.bytes, s);
}

cudaError_t launch_wait_probe(void* ws, uint64_t wait_limit_ns, cudaStream_t s) {
  int* ctr = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + ws_layout(0, 128, 128, 1, 1).counters);
  count_launch(), k_wait_probe<<<1, 32, 0, s>>>(ctr, wait_limit_ns);
  return cudaGetLastError();
}

}  // namespace moefp4
