// Device helpers: status reporting, bounded mbarrier waits, small maths.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "mla_internal.h"

namespace mla {

// Record the first device-side error; later ones only bump the count.
__device__ __forceinline__ void report(int* status, int code, int detail) {
  if (atomicCAS(&status[MLA_ST_CODE], 0, code) == 0) status[MLA_ST_DETAIL] = detail;
  atomicAdd(&status[MLA_ST_COUNT], 1);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of the same condition.  When the phase has already
// completed this returns in a fraction of the time try_wait takes, which
// matters on the tensor-core issue path (one check per ring stage).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, polling at most `max_polls`
// times and for at most `max_ns` nanoseconds.  On giving up, records
// MLA_ERR_TIMEOUT with `where` as detail and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status, int where,
                                          long long max_polls = (1LL << 40),
                                          uint64_t max_ns = 2000000000ull) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (long long i = 1; i < max_polls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 0 && global_ns() - t0 > max_ns) break;
  }
  report(status, MLA_ERR_TIMEOUT, where);
  return false;
}

// Wait on a barrier that other CTAs of the cluster arrive on (remote arrive,
// multicast commit, or a copy issued by the other CTA): acquire at cluster
// scope.  Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_test_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int* status,
                                                  int where, uint64_t max_ns = 2000000000ull) {
  if (mbar_test_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (long long i = 1;; ++i) {
    // the potentially blocking probe suspends the thread in hardware until
    // the phase completes or a time limit passes
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 255) == 0 && global_ns() - t0 > max_ns) break;
  }
  report(status, MLA_ERR_TIMEOUT, where);
  return false;
}

// Copy `bytes` (a multiple of 16, both ends 16-byte aligned) from global to
// shared memory with 16-byte asynchronous copies strided over `nthreads`
// threads (each thread's share; complete with cp_async_wait_all and a block
// barrier).  Many independent requests per thread keep the copy near the
// HBM rate without holding registers.
__device__ __forceinline__ void cp_async_block(void* dst, const void* src, size_t bytes, int tid,
                                               int nthreads) {
  const uint32_t d = smem_u32(dst);
  const char* s = static_cast<const char*>(src);
  for (size_t o = (size_t)tid * 16; o < bytes; o += (size_t)nthreads * 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + (uint32_t)o), "l"(s + o)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

// 32-byte global accesses (a whole L2 sector per thread), caching in L2
// only: the split results are written and read 8 fp32 columns at a time.
__device__ __forceinline__ void st_v8(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.cg.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// 32 bytes of read-only data through the non-coherent path.
__device__ __forceinline__ void ld_nc_v8(const void* p, uint32_t* v) {
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                 "=r"(v[6]), "=r"(v[7])
               : "l"(p));
}

__device__ __forceinline__ void ld_cg_v8(const float* p, float (&v)[8]) {
  asm volatile("ld.global.cg.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                 "=f"(v[6]), "=f"(v[7])
               : "l"(p));
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Global page range [g0, g1) of split c when P pages are cut into G splits.
__device__ __forceinline__ void split_range(int c, long long P, int G, long long* g0,
                                            long long* g1) {
  *g0 = (long long)c * P / G;
  *g1 = (long long)(c + 1) * P / G;
}

// Largest b in [0, B) with prefix[b] <= g (prefix strictly increasing).
__device__ __forceinline__ int seq_of_page(const int* prefix, int B, long long g) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (prefix[mid] <= g) lo = mid; else hi = mid;
  }
  return lo;
}

}  // namespace mla
