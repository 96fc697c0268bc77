// Compress + RoPE + paged append and the absorbed query image for one or two
// query tokens, as matrix-vector products on CUDA cores.
//
// Page "DeepSeek-V2：在“大力出奇迹”的AI军备竞赛中，四两拨千斤" (liang.world),
// 第二章 §2-§3: every new token caches c^KV = W^DKV h and k^R = RoPE(W^KR h);
// the absorbed query of head i is q~_i = W^UK_i^T q^C_i next to RoPE(q^R_i),
// written as the attention kernel's query image.
//
// With one or two tokens each weight element feeds one or two multiply-adds,
// so the launch is bound by reading the weights (W^UK 16 MB, [W^DKV; W^KR]
// 5.6 MB at V2 widths).  One CTA per SM: when the absorbed query is computed
// CTA i < 128 owns head i's W^UK block (128 x 512, contiguous) and a few
// rows of [W^DKV; W^KR]; the other CTAs share the remaining rows.  Each CTA
// fetches its weights into shared memory with 16-byte asynchronous copies
// (many in flight per thread) before it waits for the previous kernel (h and
// q may come from it), then computes:
//   * W^UK_i^T q^C_i: eight warps, 16 weight rows each, lane = 16 latent
//     columns; the eight partial sums added in warp order;
//   * a row of [W^DKV; W^KR] . h: the row is cut into 8 fixed K segments (a
//     warp each, lane-strided 16-byte chunks, xor-shuffle sum) whose sums
//     are added in segment order, so a row's value depends neither on the
//     CTA that computes it nor on whether the query runs in the same launch;
//     RoPE pairs (2j, 2j+1) of k^R always sit in the same CTA.
// The last CTA also builds the split-KV plan.
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "gemv.h"
#include "layouts.cuh"
#include "launch_util.h"
#include "tc_util.cuh"

namespace mla {
namespace {

constexpr int kPsThreads = 1024;
constexpr int kPsWarps = kPsThreads / 32;
constexpr int kPsSegs = 8;               // K segments of an append row
constexpr int kPsAbsWarps = 8;           // warps of the absorbed query
constexpr int kPsAppendRows = kLat + kRope;   // 576
constexpr uint32_t kPsHeadBytes = kNope * kLat * 2;   // one head of W^UK (128 KB)

// Shared-memory layout, the same on the host and the device.
struct PsLayout {
  uint32_t w_bytes;    // weights: head block (head CTAs) then append rows
  uint32_t off_x, off_q, off_red, off_part, off_tmp, off_bar, total;
};

__host__ __device__ inline uint32_t ps_align(uint32_t x) { return (x + 127u) & ~127u; }

__host__ __device__ inline PsLayout ps_layout(int M, int D, uint32_t w_bytes, int max_rows,
                                              bool absorb) {
  PsLayout L;
  L.w_bytes = ps_align(w_bytes);
  L.off_x = L.w_bytes;
  L.off_q = ps_align(L.off_x + (uint32_t)M * D * 2u);
  L.off_red = ps_align(L.off_q + (uint32_t)M * kNope * 4u);
  L.off_part = ps_align(L.off_red + (absorb ? (uint32_t)kPsAbsWarps * M * kLat * 4u : 0u));
  L.off_tmp = ps_align(L.off_part + (uint32_t)max_rows * kPsSegs * M * 4u);
  L.off_bar = ps_align(L.off_tmp + 33u * 4u);
  L.total = L.off_bar + 16u;
  return L;
}

// Append rows [lo, hi) of CTA i: rows_head each for the head CTAs (i < H),
// the rest shared in pairs by the others.
__host__ __device__ inline void ps_rows(int i, int G, int H, int rows_head, int* lo, int* hi) {
  if (i < H) {
    *lo = i * rows_head;
    *hi = *lo + rows_head;
    return;
  }
  const int base = H * rows_head, pairs = (kPsAppendRows - base) / 2, n = G - H, j = i - H;
  *lo = base + 2 * (int)((long long)j * pairs / n);
  *hi = base + 2 * (int)((long long)(j + 1) * pairs / n);
}

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

// acc[0..7] += (8 bf16 of w) * s
__device__ __forceinline__ void axpy8(float* acc, const uint4& w, float s) {
  acc[0] = fmaf(lo_f(w.x), s, acc[0]);
  acc[1] = fmaf(hi_f(w.x), s, acc[1]);
  acc[2] = fmaf(lo_f(w.y), s, acc[2]);
  acc[3] = fmaf(hi_f(w.y), s, acc[3]);
  acc[4] = fmaf(lo_f(w.z), s, acc[4]);
  acc[5] = fmaf(hi_f(w.z), s, acc[5]);
  acc[6] = fmaf(lo_f(w.w), s, acc[6]);
  acc[7] = fmaf(hi_f(w.w), s, acc[7]);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int M>
__global__ void __launch_bounds__(kPsThreads, 1) proj_small_kernel(const SmallProjArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, i = blockIdx.x;
  const bool absorb = a.q != nullptr, append = a.h != nullptr;
  const int H = absorb ? kHeads : 0;
  const bool has_head = i < H;
  int rlo = 0, rhi = 0;
  if (append) ps_rows(i, G, H, a.rows_head, &rlo, &rhi);
  const int nrows = rhi - rlo;
  const PsLayout L = ps_layout(M, a.D, a.w_bytes, a.max_rows, absorb);
  const uint32_t rows_off = absorb && has_head ? kPsHeadBytes : 0u;
  const size_t row_bytes = (size_t)a.D * 2;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // ---- this CTA's weights (independent of the previous kernel)
  {
    if (has_head) cp_async_block(smem, a.w_uk + (size_t)i * kNope * kLat, kPsHeadBytes, tid, kPsThreads);
    // rows below 512 come from W^DKV, the others from W^KR
    const int d_hi = min(rhi, kLat), r_lo = max(rlo, kLat);
    if (d_hi > rlo)
      cp_async_block(smem + rows_off, a.w_dkv + (size_t)rlo * a.D, (d_hi - rlo) * row_bytes, tid,
                     kPsThreads);
    if (rhi > r_lo)
      cp_async_block(smem + rows_off + (size_t)(r_lo - rlo) * row_bytes,
                     a.w_kr + (size_t)(r_lo - kLat) * a.D, (rhi - r_lo) * row_bytes, tid, kPsThreads);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");   // h, q and seq_lens

  // ---- inputs into shared memory
  uint4* xs = reinterpret_cast<uint4*>(smem + L.off_x);      // h [M][D]
  float* qs = reinterpret_cast<float*>(smem + L.off_q);      // q^C of this head [M][128] (fp32)
  if (append && nrows > 0) {
    const int nq = a.D / 8;
    for (int e = tid; e < M * nq; e += kPsThreads)
      xs[e] = *reinterpret_cast<const uint4*>(a.h + (size_t)(e / nq) * a.D + (size_t)(e % nq) * 8);
  }
  if (has_head && tid < M * kNope) {
    const int m = tid / kNope, r = tid % kNope;
    qs[tid] = __bfloat162float(a.q[((size_t)m * kHeads + i) * (kNope + kRope) + r]);
  }
  cp_async_wait_all();
  __syncthreads();

  float* red = reinterpret_cast<float*>(smem + L.off_red);    // [warp][M][512]
  float* part = reinterpret_cast<float*>(smem + L.off_part);  // [row][seg][M]
  const int app_w0 = has_head ? kPsAbsWarps : 0;              // first append warp
  if (has_head && warp < kPsAbsWarps) {
    // ---- q~ = W^UK_i^T q^C_i: rows warp*16 .. +15, columns lane*8.. and (lane+32)*8..
    const uint4* ws = reinterpret_cast<const uint4*>(smem);
    float acc[M][16];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[m][e] = 0.f;
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
      const int r = warp * 16 + j;
      const uint4 w0 = ws[r * (kLat / 8) + lane], w1 = ws[r * (kLat / 8) + lane + 32];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const float s = qs[m * kNope + r];
        axpy8(acc[m], w0, s);
        axpy8(acc[m] + 8, w1, s);
      }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float4* dst = reinterpret_cast<float4*>(red + ((size_t)warp * M + m) * kLat);
      dst[lane * 2] = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
      dst[lane * 2 + 1] = make_float4(acc[m][4], acc[m][5], acc[m][6], acc[m][7]);
      dst[(lane + 32) * 2] = make_float4(acc[m][8], acc[m][9], acc[m][10], acc[m][11]);
      dst[(lane + 32) * 2 + 1] = make_float4(acc[m][12], acc[m][13], acc[m][14], acc[m][15]);
    }
  } else if (warp >= app_w0 && nrows > 0) {
    // ---- append rows: unit = (row, K segment), one warp per unit
    const int seg_q = a.D / (8 * kPsSegs);   // 16-byte chunks per segment
    const uint4* wr = reinterpret_cast<const uint4*>(smem + rows_off);
    for (int u = warp - app_w0; u < nrows * kPsSegs; u += kPsWarps - app_w0) {
      const int rl = u / kPsSegs, sg = u % kPsSegs;
      const uint4* w = wr + (size_t)rl * (a.D / 8) + sg * seg_q;
      const uint4* x = xs + sg * seg_q;
      float acc[M];
#pragma unroll
      for (int m = 0; m < M; ++m) acc[m] = 0.f;
      for (int c = lane; c < seg_q; c += 32) {
        const uint4 wv = w[c];
#pragma unroll
        for (int m = 0; m < M; ++m) fma8(acc[m], wv, x[(size_t)m * (a.D / 8) + c]);
      }
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float v = acc[m];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) part[(rl * kPsSegs + sg) * M + m] = v;
      }
    }
  }
  __syncthreads();

  if (has_head) {
    uint8_t* img = reinterpret_cast<uint8_t*>(a.qimg);
    if (tid < M * (kLat / 8)) {
      // ---- q~ of this head: 8 columns per thread, the warps' sums in order
      const int m = tid / (kLat / 8), kq = tid % (kLat / 8);
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = 0.f;
      for (int w = 0; w < kPsAbsWarps; ++w) {
        const float4* src = reinterpret_cast<const float4*>(red + ((size_t)w * M + m) * kLat + kq * 8);
        const float4 p0 = src[0], p1 = src[1];
        v[0] += p0.x; v[1] += p0.y; v[2] += p0.z; v[3] += p0.w;
        v[4] += p1.x; v[5] += p1.y; v[6] += p1.z; v[7] += p1.w;
      }
      *reinterpret_cast<uint4*>(img + (size_t)m * kQImgBytes + qimg_off(i, kq * 8)) =
          make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                     pack_bf16(v[6], v[7]));
    } else if (tid >= 512 && tid < 512 + M * (kRope / 2)) {
      // ---- RoPE(q^R) of this head at the token's position -> features 512..575
      const int e = tid - 512, m = e / (kRope / 2), p = e % (kRope / 2);
      const int b = m / a.T, t = m % a.T;
      const int pos = plan_len(a.plan.seq_lens, b, a.T, kPage, a.plan.max_pages, a.max_position) -
                      a.T + t;
      const __nv_bfloat16* x = a.q + ((size_t)m * kHeads + i) * (kNope + kRope) + kNope + 2 * p;
      const float x0 = __bfloat162float(x[0]), x1 = __bfloat162float(x[1]);
      const float2 cs = a.rope_cs[(size_t)pos * (kRope / 2) + p];
      *reinterpret_cast<uint32_t*>(img + (size_t)m * kQImgBytes + qimg_off(i, kLat + 2 * p)) =
          pack_bf16(x0 * cs.x - x1 * cs.y, x0 * cs.y + x1 * cs.x);
    }
  }
  if (nrows > 0 && tid < nrows * M) {
    // ---- finish append rows: segment sums in order, RoPE on k^R, store
    const int rl = tid / M, m = tid % M;
    const int row = rlo + rl;
    float v = 0.f, other = 0.f;
#pragma unroll
    for (int sg = 0; sg < kPsSegs; ++sg) v += part[(rl * kPsSegs + sg) * M + m];
    const int pos = a.pos[m];
    const bool pos_ok = pos >= 0 && pos < a.max_position;
    if (row >= kLat) {
      const int pr = rl ^ 1;   // the pair partner, in this CTA (even row boundaries)
#pragma unroll
      for (int sg = 0; sg < kPsSegs; ++sg) other += part[(pr * kPsSegs + sg) * M + m];
      if (pos_ok) {
        const float2 cs = a.rope_cs[(size_t)pos * (kRope / 2) + ((row - kLat) >> 1)];
        v = (row & 1) ? fmaf(other, cs.y, v * cs.x) : fmaf(-other, cs.y, v * cs.x);
      }
    }
    __nv_bfloat16* dst = nullptr;
    if (a.stage_rows) {
      dst = a.cache + (size_t)m * kRow + row;
    } else if (!pos_ok || pos / kPage >= a.max_pages) {
      if (rlo == 0 && rl == 0) report(a.status, MLA_ERR_DEVICE_INDEX, 2000000 + m);
    } else {
      const int b = m / a.T;
      const int pg = a.bt[(size_t)b * a.max_pages + pos / kPage];
      if (pg < 0 || pg >= a.num_pages) {
        if (rlo == 0 && rl == 0) report(a.status, MLA_ERR_DEVICE_INDEX, 3000000 + m);
      } else {
        dst = a.cache + ((size_t)pg * kPage + pos % kPage) * kRow + row;
      }
    }
    if (dst) *dst = __float2bfloat16_rn(v);
  }
  if (a.do_plan && i == G - 1) {
    __syncthreads();
    build_plan<kPsThreads>(tid, [] { __syncthreads(); }, reinterpret_cast<int*>(smem + L.off_tmp),
                           a.plan);
  }
}

}  // namespace

// Append rows per head CTA that balance the bytes each CTA reads (even), the
// largest row count of any CTA and the largest weight bytes of any CTA.
static void ps_balance(const SmallProjArgs& a, int G, int* rows_head, int* max_rows,
                       uint32_t* w_bytes) {
  const bool absorb = a.q != nullptr, append = a.h != nullptr;
  const int H = absorb ? kHeads : 0;
  const long long row_bytes = 2LL * a.D;
  int rh = 0;
  if (append && absorb) {
    const long long total = (long long)H * kPsHeadBytes + kPsAppendRows * row_bytes;
    const long long target = total / G;
    rh = target > (long long)kPsHeadBytes ? (int)((target - kPsHeadBytes) / row_bytes) : 0;
    rh &= ~1;
    while (H * rh > kPsAppendRows) rh -= 2;
  }
  int mx = 0;
  long long wb = absorb ? kPsHeadBytes : 0;
  if (append) {
    for (int i = 0; i < G; ++i) {
      int lo, hi;
      ps_rows(i, G, H, rh, &lo, &hi);
      mx = hi - lo > mx ? hi - lo : mx;
      const long long b = (i < H ? (long long)kPsHeadBytes : 0LL) + (hi - lo) * row_bytes;
      wb = b > wb ? b : wb;
    }
  }
  *rows_head = rh;
  *max_rows = mx;
  *w_bytes = (uint32_t)(wb < (1LL << 30) ? wb : (1LL << 30));
}

bool proj_small_supported(const SmallProjArgs& a, int num_sms) {
  if (a.M < 1 || a.M > kGemvMaxTokens || a.D % (8 * kPsSegs) != 0 || a.D <= 0) return false;
  if (a.q == nullptr && a.h == nullptr) return false;
  if (a.q != nullptr && num_sms < kHeads + (a.h != nullptr ? 1 : 0)) return false;
  int rh, mx;
  uint32_t wb;
  ps_balance(a, num_sms, &rh, &mx, &wb);
  const PsLayout L = ps_layout(a.M, a.D, wb, mx, a.q != nullptr);
  return L.total <= 232448u && mx <= 64;
}

cudaError_t proj_small_launch(const SmallProjArgs& a0, int num_sms, cudaStream_t st) {
  if (!proj_small_supported(a0, num_sms)) return cudaErrorInvalidValue;
  SmallProjArgs a = a0;
  ps_balance(a, num_sms, &a.rows_head, &a.max_rows, &a.w_bytes);
  const PsLayout L = ps_layout(a.M, a.D, a.w_bytes, a.max_rows, a.q != nullptr);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kPsThreads);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.M == 1) {
    static std::atomic<uint64_t> done1{0};
    if (const cudaError_t e = smem_attr_once(done1, proj_small_kernel<1>, 232448); e != cudaSuccess)
      return e;
    return cudaLaunchKernelEx(&cfg, proj_small_kernel<1>, a);
  }
  static std::atomic<uint64_t> done2{0};
  if (const cudaError_t e = smem_attr_once(done2, proj_small_kernel<2>, 232448); e != cudaSuccess)
    return e;
  return cudaLaunchKernelEx(&cfg, proj_small_kernel<2>, a);
}

}  // namespace mla
