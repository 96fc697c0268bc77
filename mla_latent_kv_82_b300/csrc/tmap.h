// Host-side TMA tensor-map helper.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace mla {

// Tiled map of a row-major bf16 matrix [rows, cols] (row stride ld_elems),
// box = box_rows x box_cols elements, 128-byte swizzle, zero fill out of
// bounds.  box_cols * 2 must be 128 (one swizzle row).  Returns false if the
// driver rejects it.
bool make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t ld_elems, uint32_t box_cols, uint32_t box_rows, bool weights);

}  // namespace mla
