// Decode without a caller-provided workspace (mla_decode_static_workspace).
//
// Some callers cannot allocate device memory at the point where they decode:
// code running under a fixed memory budget that was reserved up front, a
// host runtime whose allocator is not reachable from the thread that issues
// the step, or a plugin that is only handed input and output buffers.  For
// them this entry point runs the same decode as mla_decode, with its scratch
// in a statically sized device array that the library owns.  It calls no
// cudaMalloc, cudaFree or allocating library routine.
//
// The array costs kStaticWorkspaceBytes of device memory on every GPU where
// the library's device code is loaded, for the life of the process.  All
// calls share it: calls that overlap on the GPU (two streams, two contexts,
// two threads) race on it and give wrong results.  Nothing in it needs to
// start at zero: every byte a decode reads was written earlier by the same
// call (the split-K tile counters live in the context, not here).
#include <mutex>

#include "mla_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

// Device-side scratch.  Host code must not use this name as an address:
// on the host it is a stand-in for the symbol, and only the address that
// cudaGetSymbolAddress returns for the current device is valid on the GPU.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_workspace on `device` (which must be current),
// looked up once per device and cached.
mla_status static_workspace_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_addr[device] = p;
  }
  *out = g_addr[device];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_static_workspace(mla_ctx* ctx, const void* q, const void* cache,
                                                  int num_pages, const int32_t* block_table,
                                                  int max_pages, const int32_t* seq_lens,
                                                  int batch, int T, void* out, void* stream) {
  if (!ctx || batch < 1 || T < 1 || max_pages < 1) return MLA_ERR_INVALID_ARG;
  const size_t need = mla_decode_workspace_size(ctx, batch, T, max_pages);
  if (need == 0) return MLA_ERR_INVALID_ARG;
  if (need > kStaticWorkspaceBytes) return MLA_ERR_WORKSPACE;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) {
    cudaGetLastError();
    prev = -1;
  }
  if (cudaSetDevice(ctx->device) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  void* ws = nullptr;
  mla_status s = static_workspace_address(ctx->device, &ws);
  if (s == MLA_OK)
    s = mla_decode(ctx, q, cache, num_pages, block_table, max_pages, seq_lens, batch, T, out, ws,
                   kStaticWorkspaceBytes, stream);
  if (prev >= 0 && prev != ctx->device) cudaSetDevice(prev);
  return s;
}
