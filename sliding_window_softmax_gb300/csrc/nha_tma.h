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

}  // namespace nha
