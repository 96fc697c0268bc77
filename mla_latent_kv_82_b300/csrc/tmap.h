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

// Views of the latent cache pool [rows, 576] bf16 (row stride 1152 bytes)
// that let one copy fetch several 64-column blocks, each landing as its own
// 128-byte-swizzled block in shared memory (block after block):
//   blocks: dims {64 columns, rows, 9 blocks}, box {64, box_rows, nb} ->
//           [nb][box_rows][64]; coordinates (0, row, first block);
//   slabs:  dims {64 columns, 32 rows, 9 blocks, rows / 32 slabs},
//           box {64, 32, nb, 2} -> [2 slabs][nb][32][64]; coordinates
//           (0, 0, first block, first slab).
bool make_tmap_pool_blocks(CUtensorMap* tm, const void* base, uint64_t rows, uint32_t box_rows,
                           uint32_t nb);
bool make_tmap_pool_slabs(CUtensorMap* tm, const void* base, uint64_t rows, uint32_t nb);

// Tiled map of a byte matrix [rows, row_bytes] (row stride row_bytes, a
// multiple of 16), box = box_rows x box_bytes; swizzle128 selects the
// 128-byte swizzle (box_bytes must then be 128), else no swizzle (box_bytes a
// multiple of 16).  Zero fill out of bounds.
bool make_tmap_u8_2d(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t row_bytes,
                     uint32_t box_bytes, uint32_t box_rows, bool swizzle128);

}  // namespace mla
