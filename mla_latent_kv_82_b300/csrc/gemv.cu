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
#include "layouts.cuh"
#include "tc_util.cuh"
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
            long long ldo, int out_rph, long long out_hs) {
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
    const int r = r_lo + i;
    const long long col = out_rph > 0 ? (long long)(r / out_rph) * out_hs + r % out_rph : r;
    out[t * ldo + col] = __float2bfloat16_rn(v);
  }
}

// ---------------------------------------------------------------------------
// Log-sum-exp combine fused with the value up-projection, for one or two
// query tokens: o_lat[m, h] = sum_s w_s O_s[m, h] / sum_s w_s (w_s = 2^(lse_s
// - max), the splits of token m's sequence), rounded to bf16 as stored, then
// o[m, h*128 + r] = W^UV[h*128 + r, :] . o_lat[m, h] (page "DeepSeek-V2：在
// “大力出奇迹”的AI军备竞赛中，四两拨千斤", liang.world, 第二章 §2: the value
// half of the absorbed form applies W^UV_i to the attention-weighted latent).
//
// One CTA per SM owns a contiguous range of at most 128 rows of W^UV (so at
// most two heads).  Its rows are one contiguous block of memory, fetched
// with 16-byte asynchronous copies into shared memory before the kernel
// waits for the attention;
// then the CTA merges the split results of its heads from L2 (thread = 4
// columns x a subset of the splits, eight loads in flight, subsets added in
// order), and each warp reduces its rows' dot products.  The CTA holding a
// head's first row writes that head's o_lat.
constexpr int kUvRows = 128;      // rows (and value features) per head
constexpr int kUvK = 512;         // latent width
constexpr int kUvMaxRows = 128;   // rows per CTA
constexpr int kUvMaxPairs = kGemvMaxTokens * 2;   // (token, head) pairs per CTA
constexpr int kUvMaxSlots = 256;  // splits per sequence
constexpr int kUvLoads = 8;       // split results in flight per thread
constexpr uint32_t kUvOffW = 0;                                    // weights [row][512]
constexpr uint32_t kUvOffSl = kUvMaxRows * kUvK * 2;               // split weights [pair][slot]
constexpr uint32_t kUvOffRed = kUvOffSl + kUvMaxPairs * kUvMaxSlots * 4;   // [thread][8] fp32
constexpr uint32_t kUvOffX = kUvOffRed + kThreads * 32;            // o_lat [pair][512] bf16
constexpr uint32_t kUvOffSum = kUvOffX + kUvMaxPairs * kUvK * 2;   // [pair] float
constexpr uint32_t kUvOffBar = kUvOffSum + kUvMaxPairs * 4;
constexpr uint32_t kUvSmem = kUvOffBar + 16;
static_assert(kUvSmem <= 232448 && kUvOffBar % 8 == 0, "shared memory");

template <int M>
__global__ void __launch_bounds__(kThreads, 1)
combine_value_kernel(const __nv_bfloat16* __restrict__ W, int R, const float* __restrict__ part_o,
                     const float* __restrict__ part_lse, const int* __restrict__ slot_base, int T,
                     int n_heads, __nv_bfloat16* __restrict__ o_lat, __nv_bfloat16* __restrict__ out,
                     int* status) {
  extern __shared__ __align__(16) uint8_t smem[];
  const uint4* wsm = reinterpret_cast<const uint4*>(smem + kUvOffW);
  float* wsl = reinterpret_cast<float*>(smem + kUvOffSl);
  float4* red = reinterpret_cast<float4*>(smem + kUvOffRed);
  uint4* xs = reinterpret_cast<uint4*>(smem + kUvOffX);
  float* wsum = reinterpret_cast<float*>(smem + kUvOffSum);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r_lo = (int)((long long)blockIdx.x * R / gridDim.x);
  const int r_hi = (int)((long long)(blockIdx.x + 1) * R / gridDim.x);
  const int h0 = r_lo / kUvRows;
  const int nh = r_hi > r_lo ? (r_hi - 1) / kUvRows - h0 + 1 : 0;
  const int np = M * nh;                  // (token, head) pairs, token-major

  // this CTA's weight rows: independent of the previous kernel
  cp_async_block(smem + kUvOffW, W + (size_t)r_lo * kUvK, (size_t)(r_hi - r_lo) * kUvK * 2, tid,
                 kThreads);
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the split results

  // weights of the splits, one warp per pair
  if (warp < np) {
    const int m = warp / nh, head = h0 + warp % nh;
    const int b = m / T, t = m % T;
    const int s0 = slot_base[b];
    int n = slot_base[b + 1] - s0;
    if (n > kUvMaxSlots) {   // cannot happen with the planner's split counts
      if (lane == 0) report(status, MLA_ERR_INVALID_ARG, 61);
      n = kUvMaxSlots;
    }
    float* wp = wsl + warp * kUvMaxSlots;
    float lmax = -INFINITY;
    for (int i = lane; i < n; i += 32) {
      const float v = part_lse[((size_t)(s0 + i) * T + t) * n_heads + head];
      wp[i] = v;
      lmax = fmaxf(lmax, v);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
    __syncwarp();
    for (int i = lane; i < n; i += 32) wp[i] = exp2f(wp[i] - lmax);
    __syncwarp();
    if (lane == 0) {   // in slot order
      float s = 0.f;
      for (int i = 0; i < n; ++i) s += wp[i];
      wsum[warp] = s;
    }
  }
  __syncthreads();

  // merge: thread = (pair, subset of the splits, 8-column chunk)
  const int subs = kThreads / (np * 64);
  const int pr = tid / (subs * 64), sub = (tid / 64) % subs, c8 = tid % 64;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  if (pr < np) {
    const int m = pr / nh, head = h0 + pr % nh;
    const int b = m / T, t = m % T;
    const int s0 = slot_base[b];
    const int n = min(slot_base[b + 1] - s0, kUvMaxSlots);
    if (n > 1) {
      const float* wp = wsl + pr * kUvMaxSlots;
      for (int i0 = sub; i0 < n; i0 += kUvLoads * subs) {
        float x[kUvLoads][8];
        float ws[kUvLoads];
#pragma unroll
        for (int j = 0; j < kUvLoads; ++j) {
          const int i = i0 + j * subs;
          ws[j] = i < n ? wp[i] : 0.f;
          // an empty split (no visible token) has weight 0 and no result
          if (ws[j] != 0.f) {
            ld_cg_v8(part_o + part_off((size_t)(s0 + i) * T + t, head, c8 * 8), x[j]);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[j][e] = 0.f;
          }
        }
#pragma unroll
        for (int j = 0; j < kUvLoads; ++j)
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] = fmaf(ws[j], x[j][e], acc[e]);
      }
    }
  }
  float4* red4 = reinterpret_cast<float4*>(red);
  red4[2 * tid] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  red4[2 * tid + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  if (tid < np * 64) {
    const int p = tid / 64, c = tid % 64;
    const int m = p / nh, head = h0 + p % nh;
    const int b = m / T;
    const int n = slot_base[b + 1] - slot_base[b];
    __nv_bfloat16* dst = o_lat + ((size_t)m * n_heads + head) * kUvK + c * 8;
    uint4 v;
    if (n > 1) {
      float a[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) a[e] = 0.f;
      for (int sb = 0; sb < subs; ++sb) {   // the subsets in order
        const int u = (p * subs + sb) * 64 + c;
        const float4 y0 = red4[2 * u], y1 = red4[2 * u + 1];
        a[0] += y0.x; a[1] += y0.y; a[2] += y0.z; a[3] += y0.w;
        a[4] += y1.x; a[5] += y1.y; a[6] += y1.z; a[7] += y1.w;
      }
      const float inv = 1.f / wsum[p];
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(a[e] * inv, a[e + 1] * inv);
        o[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      v = make_uint4(o[0], o[1], o[2], o[3]);
      if (head * kUvRows >= r_lo) *reinterpret_cast<uint4*>(dst) = v;   // the head's first row is here
    } else {
      // one split held the whole sequence: it wrote o_lat itself
      v = __ldcg(reinterpret_cast<const uint4*>(dst));
    }
    xs[p * (kUvK / 8) + c] = v;
  }
  cp_async_wait_all();
  __syncthreads();

  // o = W^UV o_lat: a warp per row, two chunks of 8 columns per lane
  for (int row = r_lo + warp; row < r_hi; row += kWarps) {
    const int hl = row / kUvRows - h0;
    const uint4* wr = wsm + (size_t)(row - r_lo) * (kUvK / 8);
    const uint4 w0 = wr[lane], w1 = wr[lane + 32];
    float acc_t[M];
#pragma unroll
    for (int t = 0; t < M; ++t) {
      acc_t[t] = 0.f;
      fma8(acc_t[t], w0, xs[(t * nh + hl) * (kUvK / 8) + lane]);
      fma8(acc_t[t], w1, xs[(t * nh + hl) * (kUvK / 8) + lane + 32]);
#pragma unroll
      for (int o = 16; o; o >>= 1) acc_t[t] += __shfl_xor_sync(0xffffffffu, acc_t[t], o);
    }
    if (lane == 0)
#pragma unroll
      for (int t = 0; t < M; ++t) out[(size_t)t * R + row] = __float2bfloat16_rn(acc_t[t]);
  }
}

template <int M>
cudaError_t launch_uv(const CombineValueArgs& g, int ctas, cudaStream_t st) {
  auto kern = combine_value_kernel<M>;
  static std::atomic<uint64_t> attr_done{0};   // per instantiation
  if (const cudaError_t e = smem_attr_once(attr_done, kern, (int)kUvSmem); e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kUvSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, g.W, g.n_heads * kUvRows, g.part_o, g.part_lse,
                            g.slot_base, g.T, g.n_heads, g.o_lat, g.out, g.status);
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
                            g.out, g.ldo, g.out_rows_per_head, g.out_head_stride);
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

bool combine_value_supported(const CombineValueArgs& g, int num_sms) {
  const int R = g.n_heads * kUvRows;
  return g.M >= 1 && g.M <= kGemvMaxTokens && g.T >= 1 && g.M % g.T == 0 && R >= num_sms &&
         (R + num_sms - 1) / num_sms <= kUvMaxRows && g.max_slots <= kUvMaxSlots;
}

cudaError_t combine_value_launch(const CombineValueArgs& g, int num_sms, cudaStream_t st) {
  if (!combine_value_supported(g, num_sms)) return cudaErrorInvalidValue;
  return g.M == 1 ? launch_uv<1>(g, num_sms, st) : launch_uv<2>(g, num_sms, st);
}

}  // namespace mla
