// Host-side builders of TMA tensor maps (defined in gemm_tc.cu).
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "gemm.h"

namespace ipttt {
namespace tc {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// cuTensorMapEncodeTiled from the driver (null if unavailable).
EncodeTiledFn get_encode_fn();
// 2-D map of a row-major matrix (rows x cols, row stride ld elements; bf16, or fp32 if `fp32`):
// boxes of box_cols x box_rows, their rows box_cols * element size bytes wide (32, 64 or 128)
// and swizzled with the matching pattern.
bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, bool fp32, int box_cols,
              int box_rows);
// 3-D map of tile-major hi planes read as an MN-major operand: a box is 64 K rows of
// box_cols / 16 plane blocks, landing in the 32-byte-swizzle operand layout.
bool make_plane_map(CUtensorMap* map, const Planes& w, int box_cols);

}  // namespace tc
}  // namespace ipttt
