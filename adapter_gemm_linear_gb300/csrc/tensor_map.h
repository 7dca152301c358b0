// Host helpers that encode TMA tensor maps (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry point, so the library needs no link
// against the driver library).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace lora {

// Row-major bf16 matrix [rows][cols] with row stride `ld` elements, tiled in
// boxes of box_rows x box_cols; `swizzle_bytes` 128 (box_cols 64: one
// 128-byte row of the swizzle atom per box row) or 32 (box_cols 16).
// Out-of-range elements of a box read as zero.
bool make_tmap_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint64_t ld,
                    uint32_t box_rows, uint32_t box_cols = 64, int swizzle_bytes = 128);

// Row-major byte matrix [rows][cols] (row stride `cols` bytes, a multiple of
// 16) in boxes of box_rows x box_cols bytes without swizzle; out-of-range
// elements read as zero.
bool make_tmap_u8(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                  uint32_t box_cols);

}  // namespace lora
