// TMA tensor-map helper shared by the tensor-core translation units.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace kdtv {

// 2-D bf16 tensor map: a rows x cols view with a row stride of
// row_stride_elems elements (0 = cols), boxes of box_rows x box_cols, 128-byte
// swizzle (or 64-byte with swizzle_bytes = 64, for 32-column boxes).
CUresult encode_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_cols, uint32_t box_rows, uint64_t row_stride_elems = 0,
                   int swizzle_bytes = 128);

}  // namespace kdtv
