// moe_copy_rows: token rows between pinned host memory and the GPU, moved by
// the SMs (16-byte loads and stores over the CPU-GPU link) instead of a copy
// engine.  On a Grace-Blackwell node the host memory that cudaHostAlloc /
// cudaHostRegister pin is directly addressable by the GPU, so a decode step's
// few KB of tokens and outputs cost one short kernel each way, which a CUDA
// graph replays with the layer.
#include "kernels.h"

namespace moefp4 {
namespace {

// Each thread copies CP16 16-byte chunks per round, one per grid-wide stride,
// the round's loads issued before its stores.
constexpr int CP16 = 4;
__global__ void __launch_bounds__(256) k_copy16(uint4* __restrict__ dst, const uint4* __restrict__ src, size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (size_t base = i0; base < n; base += CP16 * stride) {
    uint4 v[CP16];
#pragma unroll
    for (int j = 0; j < CP16; ++j) {
      const size_t i = base + j * stride;
      if (i < n) v[j] = src[i];
    }
#pragma unroll
    for (int j = 0; j < CP16; ++j) {
      const size_t i = base + j * stride;
      if (i < n) dst[i] = v[j];
    }
  }
}

}  // namespace

cudaError_t launch_copy16(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  const size_t n = bytes / 16;
  if (n == 0) return cudaSuccess;
  const size_t blocks = (n + 256 * CP16 - 1) / (256 * CP16);
  count_launch(), k_copy16<<<(unsigned)(blocks < 65535 ? blocks : 65535), 256, 0, s>>>(static_cast<uint4*>(dst),
                                                                       static_cast<const uint4*>(src), n);
  return cudaGetLastError();
}

}  // namespace moefp4
