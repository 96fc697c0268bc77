// Weight-streaming tcgen05 GEMM: launch interface (see wgemm.cu).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "plan_device.cuh"

namespace mla {

enum WgEpi { WG_ROWMAJOR = 0, WG_APPEND = 1, WG_QIMG = 2 };

struct WgArgs {
  int n_tokens;          // valid tokens (N extent)
  int k_chunks;          // K / 64
  int splits;            // K splits (1 .. k_chunks)
  int tiles_per_head;    // 128-row weight tiles per head (1 if not batched)
  int a_tiles_main;      // tiles below this come from map A, the rest from map A2
  int a_head_rows;       // A row offset per head
  int b_head_cols;       // B column offset per head
  int valid_rows_last;   // rows written for the last tile of a head
  // WG_ROWMAJOR: out[t * ld_out + head * out_head_cols + tile * 128 + f]; with
  // out_rows_per_head > 0 instead weight row r = tile * 128 + f (head 0) goes
  // to out[t * ld_out + (r / out_rows_per_head) * out_head_cols +
  // r % out_rows_per_head] (several output heads per weight tile)
  __nv_bfloat16* out;
  int ld_out, out_head_cols, out_rows_per_head;
  // WG_APPEND: cache row of token t; RoPE on rows of tile append_rope_tile
  __nv_bfloat16* cache;
  const int32_t* pos;
  const int32_t* bt;
  int max_pages, num_pages, T, max_position, append_rope_tile;
  int stage_rows;        // write token t's row to cache + t * 576 (no paging)
  const float2* rope_cs;
  // WG_QIMG: absorbed-query image per token; RoPE of q^R by tile-0 CTAs at
  // the position plan_len(seq_lens) - T + t; with do_plan, the epilogue
  // warps of CTA 0 also build the split-KV plan while the MMAs run
  __nv_bfloat16* qimg;
  const __nv_bfloat16* q;
  PlanArgs plan;
  int do_plan;
  // split-K scratch: partials [m_tiles * n_tiles * splits * NT * 128] fp32,
  // counters [m_tiles * n_tiles] (zero between launches)
  float* partials;
  int* counters;
  int* status;
};

struct WgPlan {
  CUtensorMap tmA, tmA2, tmB;
  int m_tiles, n_tiles, nt;
  WgArgs args;
};

int wgemm_token_tile(int n_tokens);
int wgemm_ctas_per_sm(int nt);
cudaError_t wgemm_launch(const WgPlan& p, int epi, bool a_mn_major, cudaStream_t st, bool pdl);
// A WG_APPEND plan (token tile 16 or 32) and a WG_QIMG plan (MN-major) in one
// launch; cudaErrorInvalidValue for another append token tile.
cudaError_t wgemm_launch_dual(const WgPlan& append, const WgPlan& qimg, cudaStream_t st, bool pdl);

}  // namespace mla
