// Weight-streaming GEMV for a projection of a decode step with few query
// tokens (M <= 2): D[t, r] = sum_k W[r, k] x_seg(r)[t, k].  Used for the
// output projection u = W_O [o_1; ...; o_{n_h}] (page "DeepSeek-V2：在“大力
// 出奇迹”的AI军备竞赛中，四两拨千斤", liang.world, 第二章 §1), where every row
// reads the same x = o; rows may also read per-segment x (x_seg(r)).
// With one token the product is a matrix-vector product: the weights are
// read once and each feeds a single multiply-add, so the kernel is bound by
// HBM reads, not by arithmetic.  On B300 plain 16-byte loads stream a
// matrix at ~5.6 TB/s where TMA tiles reach ~4.5-4.8 TB/s, so this kernel
// uses CUDA cores.
//
// One CTA per SM (its shared-memory request keeps a second one off the SM,
// also when it is launched early behind the previous kernel) owns a
// contiguous range of rows; the range is cut into segments of at most 1024
// columns, and the 32 warps take segments in turn, two at a time (eight
// 16-byte loads in flight per lane).  Each segment's dot product is reduced
// across the warp, the per-segment sums of a row are added in column order
// in shared memory, so results do not depend on timing.
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "gemv.h"
#include "launch_util.h"

namespace mla {
namespace {

constexpr int kWarps = 32;
constexpr int kThreads = 32 * kWarps;
constexpr int kSegCols = 1024;                 // columns per segment
constexpr int kSegChunks = kSegCols / 8;       // 16-byte chunks per segment (128)
constexpr int kPerLane = kSegChunks / 32;      // chunks per lane and segment (4)
constexpr int kMaxRowsPerCta = 256;
constexpr int kMaxSegsPerRow = 32;             // K <= 32768
constexpr uint32_t kSmemX = kGemvMaxTokens * 32768 * 2;   // x staged for one segment
constexpr uint32_t kSmemPart = kMaxRowsPerCta * kMaxSegsPerRow * kGemvMaxTokens * 4;
// enough that two CTAs never share an SM
constexpr uint32_t kSmem = 120 * 1024 > kSmemX + kSmemPart ? 120 * 1024 : kSmemX + kSmemPart;

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// bf16 pair (low, high) of a 32-bit word -> two floats (exact)
__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void fma8(float& acc, const uint4& w, const uint4& x) {
  acc = fmaf(lo_f(w.x), lo_f(x.x), acc);
  acc = fmaf(hi_f(w.x), hi_f(x.x), acc);
  acc = fmaf(lo_f(w.y), lo_f(x.y), acc);
  acc = fmaf(hi_f(w.y), hi_f(x.y), acc);
  acc = fmaf(lo_f(w.z), lo_f(x.z), acc);
  acc = fmaf(hi_f(w.z), hi_f(x.z), acc);
  acc = fmaf(lo_f(w.w), lo_f(x.w), acc);
  acc = fmaf(hi_f(w.w), hi_f(x.w), acc);
}

template <int M>
__global__ void __launch_bounds__(kThreads, 1)
gemv_kernel(const __nv_bfloat16* __restrict__ W, int R, int K, const __nv_bfloat16* __restrict__ x,
            long long ldx, int rows_per_seg, long long seg_stride, __nv_bfloat16* __restrict__ out,
            long long ldo) {
  extern __shared__ __align__(16) uint8_t smem[];
  float* part = reinterpret_cast<float*>(smem + kSmemX);   // [row][seg][M]
  uint4* xs = reinterpret_cast<uint4*>(smem);               // [M][K / 8] (one x segment)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r_lo = (int)((long long)blockIdx.x * R / gridDim.x);
  const int r_hi = (int)((long long)(blockIdx.x + 1) * R / gridDim.x);
  const int kq = K / 8;                          // 16-byte chunks per row
  const int nseg = (kq + kSegChunks - 1) / kSegChunks;
  const int items = (r_hi - r_lo) * nseg;        // (row, segment) pairs of this CTA
  const bool one_x = rows_per_seg >= R;          // every row reads the same x

  // weights of the warp's first two segments: independent of the previous kernel
  uint4 w[2][kPerLane];
  auto load = [&](int it, uint4* dst) {
    const int row = r_lo + it / nseg, sg = it % nseg;
    const uint4* p = reinterpret_cast<const uint4*>(W + (size_t)row * K) + sg * kSegChunks;
#pragma unroll
    for (int u = 0; u < kPerLane; ++u) {
      const int c = sg * kSegChunks + lane + 32 * u;
      dst[u] = (it < items && c < kq) ? ld_stream(p + lane + 32 * u) : make_uint4(0, 0, 0, 0);
    }
  };
  load(warp, w[0]);
  load(warp + kWarps, w[1]);
  asm volatile("griddepcontrol.wait;" ::: "memory");   // x comes from the previous kernel
  if (one_x) {
    for (int e = threadIdx.x; e < M * kq; e += kThreads) {
      const int t = e / kq, c = e % kq;
      xs[e] = *reinterpret_cast<const uint4*>(x + t * ldx + (size_t)c * 8);
    }
  }
  __syncthreads();
  for (int it0 = warp; it0 < items; it0 += 2 * kWarps) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int it = it0 + h * kWarps;
      if (it >= items) break;
      const int row = r_lo + it / nseg, sg = it % nseg;
      const __nv_bfloat16* xr = x + (size_t)(row / rows_per_seg) * seg_stride;
      float acc[M];
#pragma unroll
      for (int t = 0; t < M; ++t) acc[t] = 0.f;
#pragma unroll
      for (int u = 0; u < kPerLane; ++u) {
        const int c = sg * kSegChunks + lane + 32 * u;
        if (c < kq)
#pragma unroll
          for (int t = 0; t < M; ++t) {
            const uint4 xv = one_x ? xs[t * kq + c]
                                   : *reinterpret_cast<const uint4*>(xr + t * ldx + (size_t)c * 8);
            fma8(acc[t], w[h][u], xv);
          }
      }
#pragma unroll
      for (int t = 0; t < M; ++t) {
        float v = acc[t];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) part[((row - r_lo) * nseg + sg) * M + t] = v;
      }
    }
    load(it0 + 2 * kWarps, w[0]);
    load(it0 + 3 * kWarps, w[1]);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < (r_hi - r_lo) * M; e += kThreads) {
    const int i = e / M, t = e % M;
    float v = 0.f;
    for (int sg = 0; sg < nseg; ++sg) v += part[(i * nseg + sg) * M + t];
    out[t * ldo + r_lo + i] = __float2bfloat16_rn(v);
  }
}

template <int M>
cudaError_t launch_m(const GemvArgs& g, int ctas, cudaStream_t st, bool pdl) {
  auto kern = gemv_kernel<M>;
  static std::atomic<uint64_t> attr_done{0};   // per instantiation
  if (const cudaError_t e = smem_attr_once(attr_done, kern, (int)kSmem); e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, g.W, g.R, g.K, g.x, g.ldx, g.rows_per_seg, g.seg_stride,
                            g.out, g.ldo);
}

}  // namespace

bool gemv_supported(const GemvArgs& g, int num_sms) {
  return g.M >= 1 && g.M <= kGemvMaxTokens && g.K % 8 == 0 && g.K >= 8 && g.K <= 32768 &&
         g.R >= num_sms && (g.R + num_sms - 1) / num_sms <= kMaxRowsPerCta &&
         g.rows_per_seg > 0;
}

cudaError_t gemv_launch(const GemvArgs& g, int num_sms, cudaStream_t st, bool pdl) {
  if (!gemv_supported(g, num_sms)) return cudaErrorInvalidValue;
  return g.M == 1 ? launch_m<1>(g, num_sms, st, pdl) : launch_m<2>(g, num_sms, st, pdl);
}

}  // namespace mla
