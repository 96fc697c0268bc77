// Weight-streaming GEMV for few query tokens: launch interface (see gemv.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "plan_device.cuh"

namespace mla {

constexpr int kGemvMaxTokens = 2;

// out[t * ldo + col(r)] = bf16(sum_k W[r * K + k] * x[t * ldx + seg(r) * seg_stride + k])
// for rows r < R and tokens t < M, seg(r) = r / rows_per_seg (rows_per_seg >= R:
// one x for all rows); col(r) = r, or with out_rows_per_head > 0 row r is
// feature r % out_rows_per_head of output head r / out_rows_per_head:
// col(r) = (r / out_rows_per_head) * out_head_stride + r % out_rows_per_head.
// W, x, out device, 16-byte aligned rows; fp32 sums.
struct GemvArgs {
  const __nv_bfloat16* W;
  int R, K, M;
  const __nv_bfloat16* x;
  long long ldx;
  int rows_per_seg;
  long long seg_stride;
  __nv_bfloat16* out;
  long long ldo;
  int out_rows_per_head;
  long long out_head_stride;
};

// Log-sum-exp combine of the split results and the value up-projection, for
// M = B * T <= 2 query tokens: o_lat[m, h, :] = merged split results (bf16),
// out[m, h * 128 + r] = bf16(W[h * 128 + r, :] . o_lat[m, h, :]).  W is
// W^UV [n_heads * 128, 512]; part_o [slot][T][n_heads][512] and part_lse
// [slot][T][n_heads] (log2 units) as the attention writes them; slot_base
// [B + 1] the sequences' first slots.  A sequence held by one split has its
// o_lat written by the attention already.  max_slots bounds the slots of
// one sequence.  Errors go to *status.
struct CombineValueArgs {
  const __nv_bfloat16* W;
  int n_heads, M, T, max_slots;
  const float* part_o;
  const float* part_lse;
  const int* slot_base;
  __nv_bfloat16* o_lat;
  __nv_bfloat16* out;
  int* status;
};

// The compress + RoPE + paged append of M <= 2 new tokens (h != nullptr) and
// their absorbed query image (q != nullptr), one launch on CUDA cores:
//   row f of [W^DKV; W^KR] . h_m, RoPE on the k^R pairs at pos[m], stored in
//   the cache slot of pos[m] (block table bt, token m in sequence m / T), or
//   with stage_rows in row m of a [M, 576] buffer;
//   q~ of head i = W^UK_i^T q^C_i (q [M, 128, 192], q^C its first 128) and
//   RoPE(q^R) at position plan_len - T + t, as the query image qimg [M][147456];
//   with do_plan, the split-KV plan too.
// rows_head, max_rows and w_bytes are filled by the launch.  Pointers are
// device pointers; index errors go to *status.
struct SmallProjArgs {
  int M, T, D;
  const __nv_bfloat16* h;
  const __nv_bfloat16* w_dkv;
  const __nv_bfloat16* w_kr;
  const int32_t* pos;
  const int32_t* bt;
  int max_pages, num_pages, stage_rows;
  __nv_bfloat16* cache;
  const __nv_bfloat16* q;
  const __nv_bfloat16* w_uk;
  __nv_bfloat16* qimg;
  PlanArgs plan;
  int do_plan;
  const float2* rope_cs;
  int max_position;
  int* status;
  int rows_head, max_rows;
  uint32_t w_bytes;
};

bool gemv_supported(const GemvArgs& g, int num_sms);
cudaError_t gemv_launch(const GemvArgs& g, int num_sms, cudaStream_t st, bool pdl);
bool combine_value_supported(const CombineValueArgs& g, int num_sms);
bool proj_small_supported(const SmallProjArgs& a, int num_sms);
cudaError_t proj_small_launch(const SmallProjArgs& a, int num_sms, cudaStream_t st);
cudaError_t combine_value_launch(const CombineValueArgs& g, int num_sms, cudaStream_t st);

}  // namespace mla
