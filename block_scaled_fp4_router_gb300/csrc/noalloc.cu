// moe_layer_decode_noalloc: the single-launch decode with its scratch memory
// built into the library instead of passed in by the caller.
//
// Some callers cannot hand the library a workspace: a plain C host program
// that links only this library and the CUDA runtime and has no device-memory
// manager of its own, or a plugin running inside a host framework whose
// memory pool does not let outside code allocate device memory.  For them this
// entry point uses a fixed scratch array that lives in the library itself; it
// allocates nothing per call.
//
// The scratch is a file-scope device array of MOE_NOALLOC_SCRATCH_BYTES
// (8 MiB).  Every GPU that loads the library holds it until the process
// exits.  In host code the array's name is only a stand-in, not a device
// address, so the real address is looked up once per device with
// cudaGetSymbolAddress (on the first call made on that device, with that
// device current) and then handed to the kernel.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "layout.h"
#include "moefp4.h"

namespace {

constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// The last 256 bytes of the array hold the sticky status word: the first
// failure recorded by any call since moe_noalloc_get_status last read it.
constexpr size_t kStickyOffset = kScratchBytes - 256;

// Start of a call: a failure left in the launch's status word (the array's
// first int) moves to the sticky word, then the status word and the rest of
// the part of the layout that must start at zero (n16 16-byte chunks, the
// counters, tickets and tagged words) are cleared.  A launch whose status
// word already says MOE_ERR_TIMEOUT would stop at its first wait, so the
// word itself cannot keep the record.
__global__ void k_noalloc_begin(uint4* __restrict__ scratch, size_t n16, int* __restrict__ sticky) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i == 0) {
    int* w = reinterpret_cast<int*>(scratch);
    const int v = w[0];
    if (v != 0) *sticky = v;
    scratch[0] = make_uint4(0, 0, 0, 0);
  } else if (i < n16) {
    scratch[i] = make_uint4(0, 0, 0, 0);
  }
}

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of the scratch array (set-up on the
// first call per device).
moe_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_layer_decode_noalloc(const moe_layer_desc_t* desc, const moe_experts_t* experts,
                                                 const moe_shared_bf16_t* shared, const float* w_router,
                                                 const float* bias, const void* x, void* out, int32_t* topk_ids,
                                                 float* topk_w, moe_stream_t stream) {
  size_t need = 0;
  const moe_status_t st = moe_workspace_size(desc, &need);
  if (st != MOE_OK) return st;
  if (desc->T > moefp4::MAX_DECODE_T) return MOE_ERR_UNSUPPORTED;
  if (need > kStickyOffset) return MOE_ERR_UNSUPPORTED;  // shape too large for the built-in scratch
  if (desc->T == 0) return MOE_OK;
  void* ws = nullptr;
  const moe_status_t sst = scratch_for_current_device(&ws);
  if (sst != MOE_OK) return sst;
  // The scratch keeps whatever the previous call left in it; the launch needs
  // its counters, status word and split-K tickets at zero.  A timeout the
  // previous call recorded moves to the sticky word first, where it stays
  // until moe_noalloc_get_status reads it.
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int fold = desc->shared_in_table;  // the table shape: E + fold experts, top_k + fold per token
  const size_t zero_bytes =
      moefp4::ws_layout(desc->T, desc->H, desc->I, desc->E + fold, desc->top_k + fold).zero_end;
  static_assert(moefp4::C_STATUS == 0, "the status word is the scratch's first int");
  const size_t n16 = zero_bytes / 16;  // zero_end is a multiple of 256
  uint8_t* base = static_cast<uint8_t*>(ws);
  moefp4::count_launch(), k_noalloc_begin<<<(unsigned)((n16 + 255) / 256), 256, 0, s>>>(reinterpret_cast<uint4*>(base), n16,
                                                                 reinterpret_cast<int*>(base + kStickyOffset));
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  return moe_layer_decode(desc, experts, shared, w_router, bias, x, out, topk_ids, topk_w, ws, kStickyOffset,
                          stream);
}

extern "C" moe_status_t moe_noalloc_get_status(moe_status_t* st) {
  if (!st) return MOE_ERR_INVALID_ARG;
  void* ws = nullptr;
  const moe_status_t sst = scratch_for_current_device(&ws);
  if (sst != MOE_OK) return sst;
  // the last call's own word first (not yet moved), then the sticky one
  int v[2] = {0, 0};
  int* word = static_cast<int*>(ws);
  int* sticky = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + kStickyOffset);
  if (cudaMemcpy(&v[0], word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&v[1], sticky, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v[0] != 0 && cudaMemset(word, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  if (v[1] != 0 && cudaMemset(sticky, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  *st = static_cast<moe_status_t>(v[0] != 0 ? v[0] : v[1]);
  return MOE_OK;
}

extern "C" moe_status_t moe_debug_wait_probe_noalloc(uint64_t limit_ns, moe_stream_t stream) {
  void* ws = nullptr;
  const moe_status_t sst = scratch_for_current_device(&ws);
  if (sst != MOE_OK) return sst;
  return moe_debug_wait_probe(ws, kStickyOffset, limit_ns, stream);
}
