// tmap.h -- TMA tensor maps for fp32 row-major tensors (the weight-gradient outputs).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// 2-D fp32 row-major [rows, cols] tensor, boxes of [box_rows, 32] (128-byte rows) with
// 128-byte swizzle: the layout the TMA stores of the weight-gradient epilogue read from
// shared memory.  base 16-byte aligned, cols a multiple of 4.
cudaError_t make_tmap_f32_rows128(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);

}  // namespace moe
