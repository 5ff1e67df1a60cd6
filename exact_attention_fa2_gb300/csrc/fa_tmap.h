// fa_tmap.h - TMA tensor maps over [B*H, S, d] bf16 tensors (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Encode a 3-D tiled tensor map over a contiguous [BH, S, d] bf16 array:
// dimension 0 = d (innermost), 1 = S, 2 = BH; box = {box_w, box_rows, 1}.
// The swizzle mode is chosen from the box's inner extent in bytes (32, 64 or
// 128).  Out-of-range rows read as zero.  Returns cudaSuccess or an error.
cudaError_t make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d, int S, int BH, int box_w,
                              int box_rows);

// Same over the first `rows` rows of each head of a [BH, pitch, d] bf16
// array (base may point inside the first head: a window of key rows).
cudaError_t make_tmap_bf16_3d_rows(CUtensorMap* map, const void* base, int d, int rows, int pitch, int BH,
                                   int box_w, int box_rows);

// Same over a contiguous [BH, S, d] fp32 array (box inner extent 64 or 128
// bytes, matching swizzle), used to reduce-add tiles into it.
cudaError_t make_tmap_f32_3d(CUtensorMap* map, const void* base, int d, int S, int BH, int box_w, int box_rows);

}  // namespace fa
