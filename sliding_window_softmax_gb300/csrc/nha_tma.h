// Host side of the tensor-memory-accelerator (TMA) copies: tiled tensor maps
// over the [BH][T][D] bf16 row arrays, in the 128-byte swizzled tile format
// that the tensor-core operand tiles use (64-column blocks, 16-byte chunk c of
// row r at chunk c ^ (r & 7)).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace nha {

// Encodes a 3-D map over bf16 [BH][T][D] (innermost D) with box {64, box_rows, 1}
// and 128-byte swizzle.  Rows past T read as zeros and are not written by a
// store.  base must be 16-byte aligned.  Returns cudaErrorInvalidValue if the
// driver rejects the map, cudaErrorNotSupported if its entry point is missing.
cudaError_t tmap_rows_bf16(CUtensorMap* map, const void* base, int D, int T, int BH, int box_rows);

// Map over fp32 [BH][rows][width] with box {32, 128, 1} and 128-byte swizzle:
// a 128-row tile arrives as ceil(width / 32) boxes of 16 KB (columns past
// width read as zero).  width * 4 must be a multiple of 16.
cudaError_t tmap_rows_f32(CUtensorMap* map, const float* base, int width, int rows, int BH);

// Map over the RoPE (cos, sin) table viewed as fp32 [T][2 * H2] with box
// {32, 128} (128-byte swizzle): a 128-position tile arrives as 2 * H2 / 32
// boxes of 16 KB, box b holding the (cos, sin) pairs [16 b, 16 b + 16).
cudaError_t tmap_tab(CUtensorMap* map, const float2* tab, int H2, int T);

}  // namespace nha
