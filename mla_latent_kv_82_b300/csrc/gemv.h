// Weight-streaming GEMV for few query tokens: launch interface (see gemv.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mla {

constexpr int kGemvMaxTokens = 2;

// out[t * ldo + r] = bf16(sum_k W[r * K + k] * x[t * ldx + seg(r) * seg_stride + k])
// for rows r < R and tokens t < M, seg(r) = r / rows_per_seg (rows_per_seg >= R:
// one x for all rows).  W, x, out device, 16-byte aligned rows; fp32 sums.
struct GemvArgs {
  const __nv_bfloat16* W;
  int R, K, M;
  const __nv_bfloat16* x;
  long long ldx;
  int rows_per_seg;
  long long seg_stride;
  __nv_bfloat16* out;
  long long ldo;
};

bool gemv_supported(const GemvArgs& g, int num_sms);
cudaError_t gemv_launch(const GemvArgs& g, int num_sms, cudaStream_t st, bool pdl);

}  // namespace mla
