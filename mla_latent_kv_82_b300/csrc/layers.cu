// A decode step through a stack of MLA attention layers
// (mla_multi_layer_step): layer j runs mla_layer_step on h_j with its own
// weights and cache, then h_{j+1} = h_j + u_j (the residual connection
// around the attention output of a transformer block).  The pages count the
// cache over all l layers of the model (page "DeepSeek-V2：在“大力出奇迹”的AI
// 军备竞赛中，四两拨千斤", liang.world, 第二章 §2: (d_c + d_h^R) x l elements
// per token); they give no normalisation, and the FFN sublayer is outside
// this library.
#include "mla_internal.h"
#include "device_util.cuh"

namespace mla {
namespace {

// h[i] = round(h[i] + u[i]) in the buffer's type, fp32 addition; 8 elements
// per thread for bf16, 4 for fp32.
template <typename T>
__global__ void __launch_bounds__(256) residual_kernel(T* __restrict__ h,
                                                       const T* __restrict__ u, size_t n) {
  asm volatile("griddepcontrol.wait;" ::: "memory");   // u comes from the kernel before
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kVec = 16 / sizeof(T);
  const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * kVec;
  if (i + kVec <= n) {
    uint4 hv = *reinterpret_cast<const uint4*>(h + i);
    const uint4 uv = *reinterpret_cast<const uint4*>(u + i);
    T* hp = reinterpret_cast<T*>(&hv);
    const T* up = reinterpret_cast<const T*>(&uv);
#pragma unroll
    for (int j = 0; j < kVec; ++j) hp[j] = from_f<T>(to_f(hp[j]) + to_f(up[j]));
    *reinterpret_cast<uint4*>(h + i) = hv;
  } else {
    for (size_t j = i; j < n; ++j) h[j] = from_f<T>(to_f(h[j]) + to_f(u[j]));
  }
}

}  // namespace

bool launch_residual(mla_ctx* ctx, void* h, const void* u, size_t n, cudaStream_t st) {
  const bool bf = ctx->cfg.dtype == MLA_BF16;
  const size_t per = bf ? 8 : 4;
  const size_t threads = (n + per - 1) / per;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((threads + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_mark(ctx, st, "residual");
  ctx->launches += 1;
  const cudaError_t e =
      bf ? cudaLaunchKernelEx(&cfg, residual_kernel<__nv_bfloat16>,
                              static_cast<__nv_bfloat16*>(h), static_cast<const __nv_bfloat16*>(u), n)
         : cudaLaunchKernelEx(&cfg, residual_kernel<float>, static_cast<float*>(h),
                              static_cast<const float*>(u), n);
  return e == cudaSuccess;
}

}  // namespace mla

extern "C" mla_status mla_multi_layer_step(mla_ctx* const* ctxs, int n_layers, void* h,
                                           const int32_t* positions, void* const* caches,
                                           int num_pages, const int32_t* block_table,
                                           int max_pages, const int32_t* seq_lens, int batch,
                                           int T, void* u_scratch, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  if (!ctxs || n_layers < 1 || !h || !caches || !u_scratch) return MLA_ERR_INVALID_ARG;
  const mla_ctx* c0 = ctxs[0];
  if (!c0) return MLA_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const mla_ctx* c = ctxs[l];
    if (!c || !caches[l]) return MLA_ERR_INVALID_ARG;
    if (c->cfg.dtype != c0->cfg.dtype || c->cfg.d_model != c0->cfg.d_model ||
        c->device != c0->device)
      return MLA_ERR_INVALID_ARG;
    if (c->cfg.d_cq <= 0) return MLA_ERR_UNSUPPORTED;
    if (workspace_bytes < mla_decode_workspace_size(c, batch, T, max_pages))
      return MLA_ERR_WORKSPACE;
  }
  const size_t a = c0->cfg.dtype == MLA_BF16 ? 16 : 4;
  auto misaligned = [&](const void* p) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if (misaligned(u_scratch) || misaligned(h)) return MLA_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l)
    if (misaligned(caches[l])) return MLA_ERR_INVALID_ARG;
  const size_t n = (size_t)batch * T * c0->cfg.d_model;
  for (int l = 0; l < n_layers; ++l) {
    mla_ctx* c = ctxs[l];
    mla_status s = mla_layer_step(c, h, positions, caches[l], num_pages, block_table, max_pages,
                                  seq_lens, batch, T, u_scratch, workspace, workspace_bytes,
                                  stream);
    if (s != MLA_OK) return s;
    if (cudaSetDevice(c->device) != cudaSuccess) { cudaGetLastError(); return MLA_ERR_CUDA; }
    if (!mla::launch_residual(c, h, u_scratch, n, static_cast<cudaStream_t>(stream))) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    mla::prof_mark(c, static_cast<cudaStream_t>(stream), nullptr);
  }
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
