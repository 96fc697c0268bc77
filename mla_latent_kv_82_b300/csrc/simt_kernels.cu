// Plain SIMT kernels for every step of MLA decode, for any small widths.
//
// These serve fp32 contexts only (fp32 FMA throughout: the tensor cores
// cannot meet an fp32 tolerance); bf16 contexts run the tcgen05 kernels.
// Steps, following the page "DeepSeek-V2：在“大力出奇迹”的AI军备竞赛中，四两拨
// 千斤" (liang.world), 第二章 §1-§3:
//   compress_append  [c ; k^R] = [W^DKV h ; RoPE_pos(W^KR h)] -> paged pool
//   absorb_q         q~_i = W^UK_i^T q^C_i, q^R_i rotated at its position
//   attend           split-KV online softmax over the latent rows
//   combine_uv       log-sum-exp merge of the splits, o_i = W^UV_i o~_i
//   out_proj         u = W_O [o_1; ...; o_{n_h}]
#include "device_util.cuh"

namespace mla {
namespace {

constexpr int kTM = 64, kTN = 64, kTK = 16, kGemmThreads = 256;

enum EpiMode { EPI_STORE = 0, EPI_APPEND = 1 };

struct AppendArgs {
  const int32_t* pos;
  const int32_t* bt;
  int max_pages, num_pages, page, T, d_latent, d_rope, max_position;
  const float2* rope_cs;
  int* status;
};

// C[m, n] = sum_k A[m, k] * B[n, k], B's rows n < n_split from B0, the rest
// from B1 (row n - n_split).  fp32 accumulation.  64x64 tiles, 4x4 per thread.
// EPI_STORE writes C[m, n] at m * ldc + (n / col_group) * col_stride +
// n % col_group (col_group = N, col_stride = 0: plain row-major).
template <typename T, int MODE>
__global__ void __launch_bounds__(kGemmThreads)
gemm_tn_kernel(int M, int N, int K, const T* __restrict__ A, int lda,
               const T* __restrict__ B0, const T* __restrict__ B1, int n_split, int ldb,
               T* __restrict__ C, int ldc, AppendArgs ap, int col_group, int col_stride) {
  __shared__ float As[kTK][kTM + 4];
  __shared__ float Bs[kTK][kTN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * kTM, n0 = blockIdx.x * kTN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kTK) {
    for (int i = threadIdx.x; i < kTM * kTK; i += kGemmThreads) {
      const int r = i / kTK, kk = i % kTK;
      const int m = m0 + r, k = k0 + kk;
      As[kk][r] = (m < M && k < K) ? to_f(A[(size_t)m * lda + k]) : 0.f;
      const int n = n0 + r;
      float bv = 0.f;
      if (n < N && k < K) {
        const T* row = n < n_split ? B0 + (size_t)n * ldb : B1 + (size_t)(n - n_split) * ldb;
        bv = to_f(row[k]);
      }
      Bs[kk][r] = bv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
    const int nb = n0 + tx * 4;
    if (MODE == EPI_STORE) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = nb + j;
        if (n < N)
          C[(size_t)m * ldc + (size_t)(n / col_group) * col_stride + n % col_group] =
              from_f<T>(acc[i][j]);
      }
    } else {
      // compress + RoPE + paged append of token m
      const int pos = ap.pos[m];
      const int b = m / ap.T;
      const int lp = pos / ap.page;
      if (pos < 0 || pos >= ap.max_position || lp >= ap.max_pages) {
        if (tx == 0 && blockIdx.x == 0) report(ap.status, MLA_ERR_DEVICE_INDEX, 2000000 + m);
        continue;
      }
      const int pg = ap.bt[(size_t)b * ap.max_pages + lp];
      if (pg < 0 || pg >= ap.num_pages) {
        if (tx == 0 && blockIdx.x == 0) report(ap.status, MLA_ERR_DEVICE_INDEX, 3000000 + m);
        continue;
      }
      const size_t row = (size_t)pg * ap.page + pos % ap.page;
      float v[4] = {acc[i][0], acc[i][1], acc[i][2], acc[i][3]};
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        const int n = nb + j;
        if (n >= ap.d_latent && n + 1 < N) {   // an interleaved RoPE pair of k^R
          const int pair = (n - ap.d_latent) >> 1;
          const float2 cs = ap.rope_cs[(size_t)pos * (ap.d_rope >> 1) + pair];
          const float x0 = v[j], x1 = v[j + 1];
          v[j] = x0 * cs.x - x1 * cs.y;
          v[j + 1] = x0 * cs.y + x1 * cs.x;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (nb + j < N) C[row * ldc + nb + j] = from_f<T>(v[j]);
    }
  }
}

// q~ and the rotated q^R of one (token, head): Q[m, i, :] = [W^UK_i^T q^C ; RoPE(q^R)].
template <typename T>
__global__ void absorb_q_kernel(const T* __restrict__ q, const T* __restrict__ w_uk,
                                const int* __restrict__ lens, int T_, int H, int dn, int dc,
                                int dr, const float2* __restrict__ rope_cs,
                                T* __restrict__ Q) {
  extern __shared__ float qs[];   // [dn + dr]
  const int i = blockIdx.x, m = blockIdx.y;
  const int b = m / T_, t = m % T_;
  const T* qrow = q + ((size_t)m * H + i) * (dn + dr);
  for (int k = threadIdx.x; k < dn + dr; k += blockDim.x) qs[k] = to_f(qrow[k]);
  __syncthreads();
  const int R = dc + dr;
  T* out = Q + ((size_t)m * H + i) * R;
  const T* W = w_uk + (size_t)i * dn * dc;
  for (int j = threadIdx.x; j < dc; j += blockDim.x) {
    float acc = 0.f;
    for (int k = 0; k < dn; ++k) acc = fmaf(to_f(W[(size_t)k * dc + j]), qs[k], acc);
    out[j] = from_f<T>(acc);
  }
  const int pos = lens[b] - T_ + t;
  for (int j = threadIdx.x; j < dr / 2; j += blockDim.x) {
    const float2 cs = rope_cs[(size_t)pos * (dr >> 1) + j];
    const float x0 = qs[dn + 2 * j], x1 = qs[dn + 2 * j + 1];
    out[dc + 2 * j] = from_f<T>(x0 * cs.x - x1 * cs.y);
    out[dc + 2 * j + 1] = from_f<T>(x0 * cs.y + x1 * cs.x);
  }
}

constexpr int kAttWarps = 8, kAttRows = 8, kMaxR = 576, kMaxRegs = kMaxR / 32, kMaxC = 16;

// One CTA per (split, query token, group of 8 heads); one warp per head.
// Online softmax in the log2 domain; writes O/l and m + log2(l) per split.
template <typename T>
__global__ void __launch_bounds__(kAttWarps * 32)
attend_kernel(const T* __restrict__ Q, const T* __restrict__ cache, int num_pages,
              const int32_t* __restrict__ bt, int max_pages, const int* __restrict__ lens,
              const int* __restrict__ prefix, const int* __restrict__ first_split,
              const int* __restrict__ slot_base, const int* __restrict__ meta, int B, int T_,
              int H, int dc, int dr, int page, float scale_log2, float* __restrict__ part_o,
              float* __restrict__ part_lse, int* status) {
  __shared__ float rows[kAttRows][kMaxR];
  const int c = blockIdx.x, t = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = blockIdx.z * kAttWarps + warp;
  const bool active = head < H;
  const int R = dc + dr;
  const int G = meta[0];
  if (c >= G) return;
  long long g0, g1;
  split_range(c, prefix[B], G, &g0, &g1);
  for (int b = seq_of_page(prefix, B, g0); b < B && prefix[b] < g1; ++b) {
    const long long lo = g0 > prefix[b] ? g0 : prefix[b];
    const long long hi = g1 < prefix[b + 1] ? g1 : prefix[b + 1];
    const int vis = lens[b] - T_ + t + 1;
    const int p_begin = (int)(lo - prefix[b]) * page;
    int p_end = (int)(hi - prefix[b]) * page;
    if (p_end > vis) p_end = vis;
    const int slot = slot_base[b] + (c - first_split[b]);
    float qr[kMaxRegs];
    const size_t mrow = (size_t)b * T_ + t;
#pragma unroll
    for (int k = 0; k < kMaxRegs; ++k) {
      const int f = lane + 32 * k;
      qr[k] = (active && f < R) ? to_f(Q[(mrow * H + head) * R + f]) : 0.f;
    }
    float acc[kMaxC];
#pragma unroll
    for (int k = 0; k < kMaxC; ++k) acc[k] = 0.f;
    float mx = -INFINITY, l = 0.f;
    for (int p0 = p_begin; p0 < p_end; p0 += kAttRows) {
      const int nrow = min(kAttRows, p_end - p0);
      __syncthreads();
      for (int idx = threadIdx.x; idx < nrow * R; idx += blockDim.x) {
        const int r = idx / R, f = idx % R;
        const int p = p0 + r;
        const int pg = bt[(size_t)b * max_pages + p / page];
        float v = 0.f;
        if (pg >= 0 && pg < num_pages) {
          v = to_f(cache[((size_t)pg * page + p % page) * R + f]);
        } else if (f == 0) {
          report(status, MLA_ERR_DEVICE_INDEX, 4000000 + b);
        }
        rows[r][f] = v;
      }
      __syncthreads();
      if (!active) continue;
      for (int r = 0; r < nrow; ++r) {
        float s = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxRegs; ++k) {
          const int f = lane + 32 * k;
          if (f < R) s = fmaf(qr[k], rows[r][f], s);
        }
        s = warp_sum(s) * scale_log2;
        const float mn = fmaxf(mx, s);
        const float corr = exp2f(mx - mn);
        const float p = exp2f(s - mn);
        l = l * corr + p;
#pragma unroll
        for (int k = 0; k < kMaxC; ++k) {
          const int j = lane + 32 * k;
          if (j < dc) acc[k] = acc[k] * corr + p * rows[r][j];
        }
        mx = mn;
      }
    }
    if (active) {
      const size_t o = ((size_t)slot * T_ + t) * H + head;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int k = 0; k < kMaxC; ++k) {
        const int j = lane + 32 * k;
        if (j < dc) part_o[o * dc + j] = acc[k] * inv;
      }
      if (lane == 0) part_lse[o] = l > 0.f ? mx + log2f(l) : -INFINITY;
    }
  }
}

// One CTA per (token, head): merge the splits into o~, then o = W^UV_i o~.
template <typename T>
__global__ void combine_uv_kernel(const float* __restrict__ part_o,
                                  const float* __restrict__ part_lse,
                                  const int* __restrict__ slot_base, const T* __restrict__ w_uv,
                                  int T_, int H, int dc, int dv, T* __restrict__ o_lat,
                                  T* __restrict__ o) {
  extern __shared__ float ol[];   // [dc]
  __shared__ float wsum_s;
  const int i = blockIdx.x, m = blockIdx.y;
  const int b = m / T_, t = m % T_;
  const int s0 = slot_base[b], s1 = slot_base[b + 1];
  float lmax = -INFINITY;
  for (int s = s0; s < s1; ++s) lmax = fmaxf(lmax, part_lse[((size_t)s * T_ + t) * H + i]);
  if (threadIdx.x == 0) {
    float ws = 0.f;
    for (int s = s0; s < s1; ++s) ws += exp2f(part_lse[((size_t)s * T_ + t) * H + i] - lmax);
    wsum_s = ws;
  }
  __syncthreads();
  const float inv = 1.f / wsum_s;
  for (int j = threadIdx.x; j < dc; j += blockDim.x) {
    float acc = 0.f;
    for (int s = s0; s < s1; ++s) {
      const size_t r = ((size_t)s * T_ + t) * H + i;
      const float w = exp2f(part_lse[r] - lmax);
      if (w > 0.f) acc = fmaf(w, part_o[r * dc + j], acc);
    }
    const float v = acc * inv;
    o_lat[((size_t)m * H + i) * dc + j] = from_f<T>(v);
    ol[j] = to_f(from_f<T>(v));   // the value the up-projection sees
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int v = warp; v < dv; v += nw) {
    const T* W = w_uv + ((size_t)i * dv + v) * dc;
    float acc = 0.f;
    for (int j = lane; j < dc; j += 32) acc = fmaf(to_f(W[j]), ol[j], acc);
    acc = warp_sum(acc);
    if (lane == 0) o[(size_t)m * H * dv + (size_t)i * dv + v] = from_f<T>(acc);
  }
}

template <typename T>
void compress_append_impl(mla_ctx* ctx, const T* h, int B, int T_, const int32_t* pos,
                          const int32_t* bt, int max_pages, T* cache, int num_pages,
                          cudaStream_t st) {
  const mla_config& c = ctx->cfg;
  const int M = B * T_, N = c.d_latent + c.d_rope, K = c.d_model;
  AppendArgs ap{pos, bt, max_pages, num_pages, c.page_size, T_, c.d_latent, c.d_rope,
                c.max_position, ctx->rope_cs, ctx->status};
  dim3 grid((N + kTN - 1) / kTN, (M + kTM - 1) / kTM);
  prof_mark(ctx, st, "compress_append");
  ctx->launches += 1;
  gemm_tn_kernel<T, EPI_APPEND><<<grid, kGemmThreads, 0, st>>>(
      M, N, K, h, K, static_cast<const T*>(ctx->w.w_dkv), static_cast<const T*>(ctx->w.w_kr),
      c.d_latent, K, cache, N, ap, N, 0);
}

// q = [W^UQ W^DQ h ; W^QR h] per head, in mla_decode's q layout.
template <typename T>
void query_impl(mla_ctx* ctx, const T* h, int M, char* ws, const WsLayout& L, cudaStream_t st) {
  const mla_config& c = ctx->cfg;
  const int H = c.n_heads, dn = c.d_nope, dr = c.d_rope, D = c.d_model, dcq = c.d_cq;
  T* cq = reinterpret_cast<T*>(ws + L.c_q);
  T* q = reinterpret_cast<T*>(ws + L.q_in);
  AppendArgs none{};
  auto grid = [&](int N) { return dim3((N + kTN - 1) / kTN, (M + kTM - 1) / kTM); };
  prof_mark(ctx, st, "query_down");
  ctx->launches += 1;
  gemm_tn_kernel<T, EPI_STORE><<<grid(dcq), kGemmThreads, 0, st>>>(
      M, dcq, D, h, D, static_cast<const T*>(ctx->w.w_dq), nullptr, dcq, D, cq, dcq, none, dcq, 0);
  prof_mark(ctx, st, "query_rope");
  ctx->launches += 1;
  gemm_tn_kernel<T, EPI_STORE><<<grid(H * dr), kGemmThreads, 0, st>>>(
      M, H * dr, D, h, D, static_cast<const T*>(ctx->w.w_qr), nullptr, H * dr, D, q + dn,
      H * (dn + dr), none, dr, dn + dr);
  prof_mark(ctx, st, "query_up");
  ctx->launches += 1;
  gemm_tn_kernel<T, EPI_STORE><<<grid(H * dn), kGemmThreads, 0, st>>>(
      M, H * dn, dcq, cq, dcq, static_cast<const T*>(ctx->w.w_uq), nullptr, H * dn, dcq, q,
      H * (dn + dr), none, dn, dn + dr);
}

template <typename T>
void decode_impl(mla_ctx* ctx, const T* q, const T* cache, int num_pages,
                 const int32_t* bt, int max_pages, int B, int T_, T* out, char* ws,
                 const WsLayout& L, cudaStream_t st) {
  const mla_config& c = ctx->cfg;
  const int M = B * T_, H = c.n_heads;
  const int* lens = reinterpret_cast<const int*>(ws + L.lens);
  const int* prefix = reinterpret_cast<const int*>(ws + L.page_prefix);
  const int* first = reinterpret_cast<const int*>(ws + L.first_split);
  const int* sbase = reinterpret_cast<const int*>(ws + L.slot_base);
  const int* meta = reinterpret_cast<const int*>(ws + L.meta);
  T* Q = reinterpret_cast<T*>(ws + L.qfull);
  float* po = reinterpret_cast<float*>(ws + L.part_o);
  float* pl = reinterpret_cast<float*>(ws + L.part_lse);
  T* olat = reinterpret_cast<T*>(ws + L.o_lat);
  T* o = reinterpret_cast<T*>(ws + L.o);
  prof_mark(ctx, st, "absorb_q");
  ctx->launches += 1;
  absorb_q_kernel<T><<<dim3(H, M), 128, sizeof(float) * (c.d_nope + c.d_rope), st>>>(
      q, static_cast<const T*>(ctx->w.w_uk), lens, T_, H, c.d_nope, c.d_latent, c.d_rope,
      ctx->rope_cs, Q);
  const float scale_log2 = c.softmax_scale * 1.4426950408889634f;
  prof_mark(ctx, st, "attend");
  ctx->launches += 1;
  attend_kernel<T><<<dim3(L.G, T_, (H + kAttWarps - 1) / kAttWarps), kAttWarps * 32, 0, st>>>(
      Q, cache, num_pages, bt, max_pages, lens, prefix, first, sbase, meta, B, T_, H,
      c.d_latent, c.d_rope, c.page_size, scale_log2, po, pl, ctx->status);
  prof_mark(ctx, st, "combine_uv");
  ctx->launches += 1;
  combine_uv_kernel<T><<<dim3(H, M), 256, sizeof(float) * c.d_latent, st>>>(
      po, pl, sbase, static_cast<const T*>(ctx->w.w_uv), T_, H, c.d_latent, c.d_v, olat, o);
  const int N = c.d_model, K = H * c.d_v;
  AppendArgs none{};
  prof_mark(ctx, st, "out_proj");
  ctx->launches += 1;
  gemm_tn_kernel<T, EPI_STORE><<<dim3((N + kTN - 1) / kTN, (M + kTM - 1) / kTM), kGemmThreads, 0,
                                 st>>>(M, N, K, o, K, static_cast<const T*>(ctx->w.w_o), nullptr,
                                       N, K, out, N, none, N, 0);
}

}  // namespace

void f32_compress_append(mla_ctx* ctx, const float* h, int B, int T, const int32_t* pos,
                         const int32_t* bt, int max_pages, float* cache, int num_pages,
                         cudaStream_t st) {
  compress_append_impl<float>(ctx, h, B, T, pos, bt, max_pages, cache, num_pages, st);
}

void f32_query(mla_ctx* ctx, const float* h, int M, char* ws, const WsLayout& L,
               cudaStream_t st) {
  query_impl<float>(ctx, h, M, ws, L, st);
}

void f32_decode(mla_ctx* ctx, const float* q, const float* cache, int num_pages,
                const int32_t* bt, int max_pages, int B, int T, float* out, char* ws,
                const WsLayout& L, cudaStream_t st) {
  decode_impl<float>(ctx, q, cache, num_pages, bt, max_pages, B, T, out, ws, L, st);
}

}  // namespace mla
