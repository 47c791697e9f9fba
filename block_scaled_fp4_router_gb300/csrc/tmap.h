// TMA tensor maps of the tensor-core kernels (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moefp4 {

// 2D byte tensor [rows][row_bytes] read in boxes of box_rows rows x 128 bytes
// with the 128-byte swizzle; rows past the end of the tensor read as zeros.
cudaError_t make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_rows = 128);

// Streaming multiprocessors of the current device.
int sm_count();

}  // namespace moefp4
