// fa_tmap.h - TMA tensor maps over [B, H, rows, d] tensors (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_launch.h"

namespace fa {

// Encode a 4-D tiled tensor map over a bf16 [B, H, rows, d] view with the
// head dimension contiguous and element strides v (dimension 0 = d, 1 = rows,
// 2 = H, 3 = B; box = {box_w, box_rows, 1, 1}; coordinates (col, row, h, b)).
// The swizzle mode is chosen from the box's inner extent in bytes (32, 64 or
// 128).  Out-of-range rows read as zero.  base may point inside the tensor (a
// window of rows).  Strides of dimensions with extent > 1 must be multiples of
// 8 elements.  Returns cudaSuccess or an error.
cudaError_t make_tmap_bf16_4d(CUtensorMap* map, const void* base, int d, int rows, int H, int B, View v,
                              int box_w, int box_rows);

// The same view as a 3-D map over (col, row, b*H + h) when batch and head
// merge (a batch step is H head steps: every contiguous tensor), else the
// 4-D map; *rank3 says which, and the caller passes coordinates to match.
cudaError_t make_tmap_bf16_view(CUtensorMap* map, bool* rank3, const void* base, int d, int rows, int H, int B,
                                View v, int box_w, int box_rows);

// 3-D map over a contiguous [BH, S, d] fp32 array (box inner extent 64 or 128
// bytes, matching swizzle), used to reduce-add tiles into it.
cudaError_t make_tmap_f32_3d(CUtensorMap* map, const void* base, int d, int S, int BH, int box_w, int box_rows);

}  // namespace fa
