// Host helpers for the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace jfa {

// 2-D bf16 tensor map over a row-major [rows, cols] buffer with a box of
// box_cols x box_rows elements and 128-byte swizzle; rows past the end read as 0.
bool make_tile_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_cols,
                   int box_rows);

}  // namespace jfa
