// Tensor-map (TMA descriptor) encoding shared by the tcgen05 kernels.
#pragma once

#include <cuda.h>

namespace s2 {

// 2-D bf16 map over [rows, cols] (cols contiguous, row pitch ld elements,
// ld * 2 a multiple of 16 bytes, base 16-byte aligned) with a box of
// box_rows x 64 columns and 128-byte swizzle; rows past the end read 0.
// False when the driver entry point is missing or the encoding is refused.
bool tma_map_bf16_2d(CUtensorMap* m, const void* base, long long rows, int cols, int ld, int box_rows);

}  // namespace s2
