// bf16 decode step at DeepSeek-V2 head widths: launches and small kernels.
//
//   append   : wgemm [W^DKV; W^KR] h  (+RoPE, paged 16-byte stores)
//   decode   : wgemm absorb (query image; CTA 0 also builds the split plan)
//              -> attend (split-KV) -> combine (o_lat, bf16) -> wgemm W^UV
//              -> wgemm W_O
// Every launch after the first of a call uses programmatic dependent launch.
#include <algorithm>

#include "gemv.h"
#include "layouts.cuh"
#include "tmap.h"
#include "wgemm.h"
#include "device_util.cuh"

namespace mla {
namespace {

// Merge the split partials of one (token, head) into o_lat = sum_s w_s O_s /
// sum_s w_s with w_s = 2^(lse_s - max lse): the log-sum-exp combine of
// flash-decoding.  A sequence held by one split alone is skipped: the
// attention kernel wrote its o_lat directly.  For sequences cut into many splits (a few long
// sequences), one CTA per (token, head): the split weights are formed
// once in shared memory, then four groups of 64 threads (one 8-column chunk
// of the 512 latent columns per thread, 32-byte loads) each sum every fourth
// split with eight independent loads in flight, and the four sums are added
// in a fixed order.
constexpr int kCombineThreads = 256;
constexpr int kCombineMaxSlots = 1024;
constexpr int kCombineGroups = kCombineThreads / (kLat / 8);   // 4

__global__ void __launch_bounds__(kCombineThreads)
combine_heads_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                     const int* __restrict__ slot_base, int T, __nv_bfloat16* __restrict__ o_lat,
                     int* status) {
  __shared__ float w[kCombineMaxSlots];
  __shared__ float red[2];
  __shared__ float acc1[kCombineGroups - 1][kLat];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int mh = blockIdx.x;                   // token row * kHeads + head
  const int m = mh / kHeads, head = mh % kHeads;
  const int b = m / T, t = m % T;
  const int s0 = slot_base[b];
  int n = slot_base[b + 1] - s0;
  if (n == 1) return;   // one split held the whole sequence: it wrote o_lat itself
  if (n > kCombineMaxSlots) {   // cannot happen with the planner's slot counts
    if (threadIdx.x == 0) report(status, MLA_ERR_INVALID_ARG, 60);
    n = kCombineMaxSlots;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // weights: w_s = 2^(lse_s - max); empty splits have lse = -inf, weight 0
  float lmax = -INFINITY;
  for (int i = tid; i < n; i += kCombineThreads) {
    const float v = part_lse[((size_t)(s0 + i) * T + t) * kHeads + head];
    w[i] = v;
    lmax = fmaxf(lmax, v);
  }
  for (int o = 16; o; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  __shared__ float wmax[kCombineThreads / 32];
  if (lane == 0) wmax[warp] = lmax;
  __syncthreads();
  lmax = wmax[0];
#pragma unroll
  for (int i = 1; i < kCombineThreads / 32; ++i) lmax = fmaxf(lmax, wmax[i]);
  for (int i = tid; i < n; i += kCombineThreads) w[i] = exp2f(w[i] - lmax);
  __syncthreads();
  if (tid == 0) {
    float sum = 0.f;
    for (int i = 0; i < n; ++i) sum += w[i];
    red[0] = sum;
  }
  const int g = tid / (kLat / 8), c8 = tid % (kLat / 8);
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int i0 = g; i0 < n; i0 += 8 * kCombineGroups) {
    float x[8][8];
    float ws[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + kCombineGroups * j;
      ws[j] = i < n ? w[i] : 0.f;
      if (ws[j] != 0.f) {
        ld_cg_v8(part_o + part_off((size_t)(s0 + i) * T + t, head, c8 * 8), x[j]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[j][e] = 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(ws[j], x[j][e], acc[e]);
  }
  if (g > 0)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc1[g - 1][c8 * 8 + e] = acc[e];
  __syncthreads();
  if (g > 0) return;
  const float inv = 1.f / red[0];
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    float a0 = acc[e], a1 = acc[e + 1];
#pragma unroll
    for (int gg = 0; gg < kCombineGroups - 1; ++gg) {
      a0 += acc1[gg][c8 * 8 + e];
      a1 += acc1[gg][c8 * 8 + e + 1];
    }
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(a0 * inv, a1 * inv);
    o[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  *reinterpret_cast<uint4*>(o_lat + (size_t)mh * kLat + c8 * 8) = make_uint4(o[0], o[1], o[2], o[3]);
}

// The same merge for sequences split into a few pieces only: one CTA per
// (token, 16 heads), so that a token whose sequence one split held (it wrote
// o_lat itself) costs one small CTA that leaves at once; a thread takes one
// head and four 8-column chunks (32-byte loads, the four of a split in flight
// together; the 16 heads of a chunk are 512 contiguous bytes).
constexpr int kCombineHeads = 16;
__global__ void __launch_bounds__(256)
combine_rows_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                    const int* __restrict__ slot_base, int T, __nv_bfloat16* __restrict__ o_lat) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int m = blockIdx.x / (kHeads / kCombineHeads);
  const int head = (blockIdx.x % (kHeads / kCombineHeads)) * kCombineHeads + threadIdx.x % 16;
  const int part = threadIdx.x / 16;   // chunks part * 4 .. part * 4 + 3
  const int b = m / T, t = m % T;
  const int s0 = slot_base[b], s1 = slot_base[b + 1];
  if (s1 - s0 == 1) return;   // one split held the whole sequence: it wrote o_lat itself
  float lmax = -INFINITY;
  for (int s = s0; s < s1; ++s) lmax = fmaxf(lmax, part_lse[((size_t)s * T + t) * kHeads + head]);
  float acc[4][8];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[j][e] = 0.f;
  float wsum = 0.f;
  for (int s = s0; s < s1; ++s) {
    const size_t st = (size_t)s * T + t;
    const float w = exp2f(part_lse[st * kHeads + head] - lmax);
    wsum += w;
    if (w == 0.f) continue;   // an empty split (no visible token) contributes nothing
    float x[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j) ld_cg_v8(part_o + part_off(st, head, (part * 4 + j) * 8), x[j]);
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[j][e] = fmaf(w, x[j][e], acc[j][e]);
  }
  // the 16 heads' rows (16 KB of o_lat, contiguous) staged in shared memory,
  // then stored 16 bytes per thread in address order
  __shared__ uint4 stage[kCombineHeads * kLat / 8];
  const float inv = 1.f / wsum;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[j][e] * inv, acc[j][e + 1] * inv);
      o[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    stage[(threadIdx.x % 16) * (kLat / 8) + part * 4 + j] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(o_lat + ((size_t)m * kHeads + head - threadIdx.x % 16) * kLat);
#pragma unroll
  for (int j = 0; j < 4; ++j) dst[threadIdx.x + 256 * j] = stage[threadIdx.x + 256 * j];
}

// K splits so that one wave fills the SMs, within the scratch budget.
// Each split streams at least min_chunks (and at least nt / 8) 64-column
// chunks of its weight rows, so that its fp32 partial (nt x 128 x 4 bytes)
// stays small next to the weights it summarises and the last CTA's
// reduction stays short.
int choose_k_splits(const mla_ctx* ctx, int m_tiles, int n_tiles, int nt, int k_chunks,
                    size_t partial_cap, int min_chunks = 4) {
  min_chunks = std::max(min_chunks, nt / 8);
  const int target = ctx->num_sms * wgemm_ctas_per_sm(nt);
  int s = target / std::max(1, m_tiles * n_tiles);
  s = std::max(1, std::min(s, k_chunks / min_chunks));
  while (s > 1 && (size_t)m_tiles * n_tiles * s * nt * 128 * sizeof(float) > partial_cap) --s;
  return s;
}

// Token tile for a GEMM with m_tiles weight tiles: the smallest power of two
// covering M (16..256), halved while fewer than 32 output tiles would exist,
// so that GEMMs with few weight rows still spread over the SMs.
int pick_token_tile(int M, int m_tiles) {
  int nt = wgemm_token_tile(M);
  while (nt > 16 && (long long)m_tiles * ((M + nt - 1) / nt) < 32) nt >>= 1;
  return nt;
}

struct GemmShape {
  int nt, n_tiles, splits;
};

GemmShape gemm_shape(const mla_ctx* ctx, int M, int m_tiles, int k_chunks, int min_chunks,
                     size_t partial_cap, bool rowmajor = false) {
  GemmShape g;
  g.nt = pick_token_tile(M, m_tiles);
  if (rowmajor) {
    // Row-major outputs run 128-token tiles in the short-K configuration
    // (three stages, two CTAs per SM): K of at most eight chunks takes it
    // at any width, longer K keeps 256-token tiles and their deep ring
    if (k_chunks <= 8 && g.nt == 256) g.nt = 128;
    if (k_chunks > 8 && g.nt == 128) g.nt = 256;
  }
  g.n_tiles = (M + g.nt - 1) / g.nt;
  g.splits = rowmajor && g.nt == 128
                 ? 1
                 : choose_k_splits(ctx, m_tiles, g.n_tiles, g.nt, k_chunks, partial_cap, min_chunks);
  return g;
}

struct Bf16Plans {
  GemmShape abs, uv, o;
  GemmShape dq, uq, qr;   // query path (d_cq > 0)
};

constexpr size_t kSplitCap = 64u << 20;   // bound on the split-K scratch of the largest-M cases

Bf16Plans decode_plans(const mla_ctx* ctx, int M) {
  const int D = ctx->cfg.d_model, dcq = ctx->cfg.d_cq;
  Bf16Plans p;
  p.abs = gemm_shape(ctx, M, kHeads * (kLat / 128), kNope / 64, 4, 0);
  p.abs.splits = 1;   // two K chunks only: never split
  p.uv = gemm_shape(ctx, M, kHeads, kLat / 64, 4, kSplitCap, true);
  p.o = gemm_shape(ctx, M, D / 128, kHeads * kDv / 64, 4, kSplitCap, true);
  if (dcq > 0) {
    p.dq = gemm_shape(ctx, M, dcq / 128, D / 64, 4, kSplitCap, true);
    p.uq = gemm_shape(ctx, M, kHeads, dcq / 64, 4, kSplitCap, true);
    p.qr = gemm_shape(ctx, M, kHeads * kRope / 128, D / 64, 4, kSplitCap, true);
  }
  return p;
}

size_t partial_bytes(const GemmShape& g, int m_tiles) {
  return (size_t)m_tiles * g.n_tiles * g.splits * g.nt * 128 * sizeof(float);
}

WgArgs base_args(const mla_ctx* ctx) {
  WgArgs a{};
  a.status = ctx->status;
  a.counters = ctx->counters;
  a.rope_cs = ctx->rope_cs;
  a.max_position = ctx->cfg.max_position;
  a.tiles_per_head = 1;
  a.valid_rows_last = 128;
  a.splits = 1;
  return a;
}

bool check(cudaError_t e) {
  if (e != cudaSuccess) return false;
  return true;
}

}  // namespace

size_t bf16_wg_partial_bytes(const mla_ctx* ctx, int M) {
  const Bf16Plans p = decode_plans(ctx, M);
  size_t b = std::max(partial_bytes(p.uv, kHeads), partial_bytes(p.o, ctx->cfg.d_model / 128));
  if (ctx->cfg.d_cq > 0) {
    b = std::max(b, partial_bytes(p.dq, ctx->cfg.d_cq / 128));
    b = std::max(b, partial_bytes(p.uq, kHeads));
    b = std::max(b, partial_bytes(p.qr, kHeads * kRope / 128));
  }
  return b;
}

bool bf16_setup(mla_ctx* ctx) {
  const int D = ctx->cfg.d_model;
  const mla_weights& w = ctx->w;
  bool ok = make_tmap_bf16_2d(&ctx->tm_wdkv, w.w_dkv, kLat, D, D, 64, 128, true) &&
            make_tmap_bf16_2d(&ctx->tm_wkr, w.w_kr, kRope, D, D, 64, 128, true) &&
            make_tmap_bf16_2d(&ctx->tm_wuk, w.w_uk, kHeads * kNope, kLat, kLat, 64, 64, true) &&
            make_tmap_bf16_2d(&ctx->tm_wuk_rows, w.w_uk, kHeads * kNope, kLat, kLat, 64, 128, true) &&
            make_tmap_bf16_2d(&ctx->tm_wuv, w.w_uv, kHeads * kDv, kLat, kLat, 64, 128, true) &&
            make_tmap_bf16_2d(&ctx->tm_wo, w.w_o, D, kHeads * kDv, kHeads * kDv, 64, 128, true);
  if (ok && ctx->cfg.d_cq > 0) {
    const int dcq = ctx->cfg.d_cq;
    ok = make_tmap_bf16_2d(&ctx->tm_wdq, w.w_dq, dcq, D, D, 64, 128, true) &&
         make_tmap_bf16_2d(&ctx->tm_wuq, w.w_uq, kHeads * kNope, dcq, dcq, 64, 128, true) &&
         make_tmap_bf16_2d(&ctx->tm_wqr, w.w_qr, kHeads * kRope, D, D, 64, 128, true);
  }
  if (!ok) return false;
  if (!sv_setup(ctx)) return false;
  if (kv_fp8(ctx) &&
      cudaMalloc(&ctx->stage, (size_t)kStageRows * kRow * sizeof(__nv_bfloat16)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (cudaMalloc(&ctx->append_partials, kAppendPartialBytes) != cudaSuccess ||
      cudaMalloc(&ctx->counters, kCounters * sizeof(int)) != cudaSuccess ||
      cudaMemset(ctx->counters, 0, kCounters * sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

void bf16_teardown(mla_ctx* ctx) {
  if (ctx->stage) cudaFree(ctx->stage);
  ctx->stage = nullptr;
  if (ctx->append_partials) cudaFree(ctx->append_partials);
  if (ctx->counters) cudaFree(ctx->counters);
  ctx->append_partials = nullptr;
  ctx->counters = nullptr;
}

// GEMM plan of the compress + RoPE + paged append step.
static bool append_plan(mla_ctx* ctx, const __nv_bfloat16* h, int B, int T, const int32_t* pos,
                        const int32_t* bt, int max_pages, __nv_bfloat16* cache, int num_pages,
                        WgPlan& p) {
  const int M = B * T, D = ctx->cfg.d_model;
  p = WgPlan{};
  const GemmShape g = gemm_shape(ctx, M, 5, D / 64, 8, kAppendPartialBytes);
  p.nt = g.nt;
  p.n_tiles = g.n_tiles;
  if (p.n_tiles > 65535) return false;
  p.m_tiles = 5;   // 4 tiles of W^DKV rows, 1 tile of W^KR rows
  p.tmA = ctx->tm_wdkv;
  p.tmA2 = ctx->tm_wkr;
  if (!make_tmap_bf16_2d(&p.tmB, h, M, D, D, 64, p.nt, false)) {
    cudaGetLastError();
    return false;
  }
  WgArgs& a = p.args;
  a = base_args(ctx);
  a.n_tokens = M;
  a.k_chunks = D / 64;
  a.splits = g.splits;
  a.tiles_per_head = 5;
  a.a_tiles_main = 4;
  a.valid_rows_last = kRope;
  a.cache = cache;
  a.pos = pos;
  a.bt = bt;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.T = T;
  a.append_rope_tile = 4;
  a.partials = ctx->append_partials;
  return true;
}

// Arguments of the CUDA-core projection kernel for M <= 2 tokens: the append
// of h (if given) and the absorbed query of q (if given).
static SmallProjArgs small_proj_args(const mla_ctx* ctx, int M, int T, const __nv_bfloat16* h,
                                     const WgArgs* app, const __nv_bfloat16* q, void* qimg) {
  SmallProjArgs sp{};
  sp.M = M;
  sp.T = T;
  sp.D = ctx->cfg.d_model;
  sp.h = h;
  sp.w_dkv = static_cast<const __nv_bfloat16*>(ctx->w.w_dkv);
  sp.w_kr = static_cast<const __nv_bfloat16*>(ctx->w.w_kr);
  if (h && app) {
    sp.pos = app->pos;
    sp.bt = app->bt;
    sp.max_pages = app->max_pages;
    sp.num_pages = app->num_pages;
    sp.stage_rows = app->stage_rows;
    sp.cache = app->cache;
  }
  sp.q = q;
  sp.w_uk = static_cast<const __nv_bfloat16*>(ctx->w.w_uk);
  sp.qimg = static_cast<__nv_bfloat16*>(qimg);
  sp.rope_cs = ctx->rope_cs;
  sp.max_position = ctx->cfg.max_position;
  sp.status = ctx->status;
  return sp;
}

// The append of a plan's M rows: the CUDA-core projection kernel for one or
// two tokens, else the weight-streaming GEMM.
static bool launch_append(mla_ctx* ctx, const __nv_bfloat16* h, int M, const WgPlan& p,
                          cudaStream_t st) {
  prof_mark(ctx, st, "compress_append");
  ctx->launches += 1;
  if (M <= kGemvMaxTokens) {
    SmallProjArgs sp = small_proj_args(ctx, M, p.args.T, h, &p.args, nullptr, nullptr);
    if (proj_small_supported(sp, ctx->num_sms)) return check(proj_small_launch(sp, ctx->num_sms, st));
  }
  return check(wgemm_launch(p, WG_APPEND, false, st, true));
}

bool bf16_compress_append(mla_ctx* ctx, const __nv_bfloat16* h, int B, int T,
                          const int32_t* pos, const int32_t* bt, int max_pages,
                          __nv_bfloat16* cache, int num_pages, cudaStream_t st) {
  if (kv_fp8(ctx)) {
    // bf16 rows of up to kStageRows tokens at a time into the staging
    // buffer, then quantised into the pool
    const int M = B * T, D = ctx->cfg.d_model;
    for (int m0 = 0; m0 < M; m0 += kStageRows) {
      const int mc = std::min(kStageRows, M - m0);
      WgPlan p;
      if (!append_plan(ctx, h + (size_t)m0 * D, 1, mc, pos + m0, bt, max_pages, ctx->stage,
                       num_pages, p))
        return false;
      p.args.stage_rows = 1;
      if (!launch_append(ctx, h + (size_t)m0 * D, mc, p, st)) return false;
      if (!f8_prepare(ctx, ctx->stage, mc, m0, pos, bt, T, max_pages,
                      reinterpret_cast<uint8_t*>(cache), num_pages, nullptr, 0, nullptr, st)) {
        cudaGetLastError();
        return false;
      }
    }
    return true;
  }
  WgPlan p;
  if (!append_plan(ctx, h, B, T, pos, bt, max_pages, cache, num_pages, p)) return false;
  return launch_append(ctx, h, B * T, p, st);
}

static bool decode_impl(mla_ctx* ctx, const __nv_bfloat16* q, const __nv_bfloat16* cache,
                        int num_pages, const int32_t* bt, int max_pages, const int32_t* seq_lens,
                        int B, int T, __nv_bfloat16* out, char* ws, const WsLayout& L,
                        cudaStream_t st, const WgPlan* append, const __nv_bfloat16* append_h);

bool bf16_decode(mla_ctx* ctx, const __nv_bfloat16* q, const __nv_bfloat16* cache,
                 int num_pages, const int32_t* bt, int max_pages, const int32_t* seq_lens,
                 int B, int T, __nv_bfloat16* out, char* ws, const WsLayout& L,
                 cudaStream_t st, const WgPlan* append) {
  return decode_impl(ctx, q, cache, num_pages, bt, max_pages, seq_lens, B, T, out, ws, L, st,
                     append, nullptr);
}

static bool decode_impl(mla_ctx* ctx, const __nv_bfloat16* q, const __nv_bfloat16* cache,
                        int num_pages, const int32_t* bt, int max_pages, const int32_t* seq_lens,
                        int B, int T, __nv_bfloat16* out, char* ws, const WsLayout& L,
                        cudaStream_t st, const WgPlan* append, const __nv_bfloat16* append_h) {
  const int M = B * T, D = ctx->cfg.d_model;
  const Bf16Plans bp = decode_plans(ctx, M);
  if (bp.abs.n_tiles > 65535 || bp.uv.n_tiles > 65535 || bp.o.n_tiles > 65535) return false;
  __nv_bfloat16* qimg = reinterpret_cast<__nv_bfloat16*>(ws + L.qfull);
  __nv_bfloat16* olat = reinterpret_cast<__nv_bfloat16*>(ws + L.o_lat);
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(ws + L.o);
  float* part = reinterpret_cast<float*>(ws + L.wg_part);

  // ---- absorbed query: W^UK_i^T q^C_i (+ rotated q^R) -> query image
  SmallProjArgs sp = small_proj_args(ctx, M, T, append ? append_h : nullptr,
                                     append ? &append->args : nullptr, q, qimg);
  sp.plan = PlanArgs{seq_lens, B, T, kPage, max_pages, ctx->cfg.max_position, L.G,
                     reinterpret_cast<int*>(ws + L.lens), reinterpret_cast<int*>(ws + L.page_prefix),
                     reinterpret_cast<int*>(ws + L.first_split),
                     reinterpret_cast<int*>(ws + L.slot_base), reinterpret_cast<int*>(ws + L.meta),
                     ctx->status};
  sp.do_plan = 1;
  if (append && append_h == nullptr) return false;   // an append plan comes with its h
  const bool small = M <= kGemvMaxTokens && proj_small_supported(sp, ctx->num_sms);
  if (small) {
    // one or two tokens: matrix-vector products on CUDA cores
    prof_mark(ctx, st, append ? "append_absorb" : "absorb_q");
    ctx->launches += 1;
    if (!check(proj_small_launch(sp, ctx->num_sms, st))) return false;
  } else {
    WgPlan p{};
    p.nt = bp.abs.nt;
    p.n_tiles = bp.abs.n_tiles;
    p.m_tiles = kHeads * (kLat / 128);
    p.tmA = ctx->tm_wuk;
    p.tmA2 = ctx->tm_wuk;
    if (!make_tmap_bf16_2d(&p.tmB, q, M, kHeads * (kNope + kRope), kHeads * (kNope + kRope), 64,
                           p.nt, false)) {
      cudaGetLastError();
      return false;
    }
    WgArgs& a = p.args;
    a = base_args(ctx);
    a.n_tokens = M;
    a.k_chunks = kNope / 64;
    a.tiles_per_head = kLat / 128;
    a.a_head_rows = kNope;
    a.b_head_cols = kNope + kRope;
    a.qimg = qimg;
    a.q = q;
    a.T = T;
    a.do_plan = 1;
    a.plan = PlanArgs{seq_lens, B, T, kPage, max_pages, ctx->cfg.max_position, L.G,
                      reinterpret_cast<int*>(ws + L.lens),
                      reinterpret_cast<int*>(ws + L.page_prefix),
                      reinterpret_cast<int*>(ws + L.first_split),
                      reinterpret_cast<int*>(ws + L.slot_base), reinterpret_cast<int*>(ws + L.meta),
                      ctx->status};
    if (append && (append->nt == 16 || append->nt == 32) && M > kGemvMaxTokens) {
      // the append and the absorbed query share no data: one launch
      prof_mark(ctx, st, "append_absorb");
      ctx->launches += 1;
      if (!check(wgemm_launch_dual(*append, p, st, true))) return false;
    } else {
      // (one or two tokens: the append as mla_compress_append runs it)
      if (append && !launch_append(ctx, append_h, M, *append, st)) return false;
      prof_mark(ctx, st, "absorb_q");
      ctx->launches += 1;
      if (!check(wgemm_launch(p, WG_QIMG, true, st, true))) return false;
    }
  }
  // ---- split-KV attention over the latent cache
  if (kv_fp8(ctx)) {
    // the appended rows (staged in bf16) into the FP8 pool, the query images
    // into FP8 images, then the attention on E4M3 operands
    uint8_t* q8 = reinterpret_cast<uint8_t*>(ws + L.q8);
    uint8_t* cache8 = reinterpret_cast<uint8_t*>(const_cast<__nv_bfloat16*>(cache));
    if (!f8_prepare(ctx, ctx->stage, append ? M : 0, 0, append ? append->args.pos : nullptr, bt,
                    T, max_pages, cache8, num_pages, qimg, M, q8, st) ||
        !f8_attend(ctx, q8, cache8, num_pages, bt, max_pages, B, T, ws, L, st)) {
      cudaGetLastError();
      return false;
    }
  } else if (!sv_attend(ctx, qimg, cache, num_pages, bt, max_pages, B, T, ws, L, st)) {
    return false;
  }
  // ---- one or two query tokens: the combine and W^UV in one weight-streaming
  // kernel (o_lat is merged in the CTAs that read W^UV)
  const float* part_o = reinterpret_cast<const float*>(ws + L.part_o);
  const float* part_lse = reinterpret_cast<const float*>(ws + L.part_lse);
  const int* slot_base = reinterpret_cast<const int*>(ws + L.slot_base);
  CombineValueArgs cv{static_cast<const __nv_bfloat16*>(ctx->w.w_uv), kHeads, M, T, L.n_slots,
                      part_o, part_lse, slot_base, olat, o, ctx->status};
  const bool fused_uv = combine_value_supported(cv, ctx->num_sms);
  if (fused_uv) {
    prof_mark(ctx, st, "combine_uv");
    ctx->launches += 1;
    if (!check(combine_value_launch(cv, ctx->num_sms, st))) return false;
  }
  // ---- log-sum-exp combine -> o_lat (bf16)
  if (!fused_uv) {
    prof_mark(ctx, st, "combine");
    ctx->launches += 1;
    // many splits per sequence: a CTA per (token, head); else a CTA per
    // (token, 16 heads)
    const bool per_head = L.n_slots >= 8 * B;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = per_head ? dim3(M * kHeads) : dim3(M * (kHeads / kCombineHeads));
    cfg.blockDim = per_head ? dim3(kCombineThreads) : dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e =
        per_head ? cudaLaunchKernelEx(&cfg, combine_heads_kernel, part_o, part_lse, slot_base, T,
                                      olat, ctx->status)
                 : cudaLaunchKernelEx(&cfg, combine_rows_kernel, part_o, part_lse, slot_base, T,
                                      olat);
    if (!check(e))
      return false;
  }
  // ---- value up-projection: o_i = W^UV_i o_lat_i
  if (!fused_uv) {
    WgPlan p{};
    p.nt = bp.uv.nt;
    p.n_tiles = bp.uv.n_tiles;
    p.m_tiles = kHeads;
    p.tmA = ctx->tm_wuv;
    p.tmA2 = ctx->tm_wuv;
    if (!make_tmap_bf16_2d(&p.tmB, olat, M, kHeads * kLat, kHeads * kLat, 64, p.nt, false)) {
      cudaGetLastError();
      return false;
    }
    WgArgs& a = p.args;
    a = base_args(ctx);
    a.n_tokens = M;
    a.k_chunks = kLat / 64;
    a.splits = bp.uv.splits;
    a.tiles_per_head = 1;
    a.a_head_rows = kDv;
    a.b_head_cols = kLat;
    a.out = o;
    a.ld_out = kHeads * kDv;
    a.out_head_cols = kDv;
    a.partials = part;
    prof_mark(ctx, st, "value_proj");
    ctx->launches += 1;
    if (!check(wgemm_launch(p, WG_ROWMAJOR, false, st, true))) return false;
  }
  // ---- output projection: u = W_O o
  GemvArgs go{static_cast<const __nv_bfloat16*>(ctx->w.w_o), D, kHeads * kDv, M, o,
              (long long)kHeads * kDv, D, 0, out, (long long)D};
  if (gemv_supported(go, ctx->num_sms)) {
    // one or two tokens: a matrix-vector product, bound by streaming W_O
    prof_mark(ctx, st, "out_proj");
    ctx->launches += 1;
    if (!check(gemv_launch(go, ctx->num_sms, st, true))) return false;
  } else {
    WgPlan p{};
    p.nt = bp.o.nt;
    p.n_tiles = bp.o.n_tiles;
    p.m_tiles = D / 128;
    p.tmA = ctx->tm_wo;
    p.tmA2 = ctx->tm_wo;
    if (!make_tmap_bf16_2d(&p.tmB, o, M, kHeads * kDv, kHeads * kDv, 64, p.nt, false)) {
      cudaGetLastError();
      return false;
    }
    WgArgs& a = p.args;
    a = base_args(ctx);
    a.n_tokens = M;
    a.k_chunks = kHeads * kDv / 64;
    a.splits = bp.o.splits;
    a.tiles_per_head = D / 128;
    a.out = out;
    a.ld_out = D;
    a.out_head_cols = 0;
    a.partials = part;
    prof_mark(ctx, st, "out_proj");
    ctx->launches += 1;
    if (!check(wgemm_launch(p, WG_ROWMAJOR, false, st, true))) return false;
  }
  return true;
}

// Query path: c^Q = W^DQ h, q^R = W^QR h (row r of W^QR is feature r % 64 of
// head r / 64), q^C = W^UQ c^Q, written as mla_decode's q [M, heads, 192].
bool bf16_query(mla_ctx* ctx, const __nv_bfloat16* h, int M, char* ws, const WsLayout& L,
                cudaStream_t st) {
  const int D = ctx->cfg.d_model, dcq = ctx->cfg.d_cq;
  const Bf16Plans bp = decode_plans(ctx, M);
  if (bp.dq.n_tiles > 65535 || bp.uq.n_tiles > 65535 || bp.qr.n_tiles > 65535) return false;
  __nv_bfloat16* cq = reinterpret_cast<__nv_bfloat16*>(ws + L.c_q);
  __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(ws + L.q_in);
  float* part = reinterpret_cast<float*>(ws + L.wg_part);
  constexpr int kQRow = kHeads * (kNope + kRope);
  auto rowmajor = [&](const GemmShape& g, int m_tiles, const CUtensorMap& wmap, const void* x,
                      int x_cols, int k_chunks, int tiles_per_head, int a_head_rows,
                      __nv_bfloat16* out, int ld_out, int out_head_cols, int rows_per_head,
                      const char* name) {
    WgPlan p{};
    p.nt = g.nt;
    p.n_tiles = g.n_tiles;
    p.m_tiles = m_tiles;
    p.tmA = wmap;
    p.tmA2 = wmap;
    if (!make_tmap_bf16_2d(&p.tmB, x, M, x_cols, x_cols, 64, p.nt, false)) {
      cudaGetLastError();
      return false;
    }
    WgArgs& a = p.args;
    a = base_args(ctx);
    a.n_tokens = M;
    a.k_chunks = k_chunks;
    a.splits = g.splits;
    a.tiles_per_head = tiles_per_head;
    a.a_head_rows = a_head_rows;
    a.b_head_cols = 0;
    a.out = out;
    a.ld_out = ld_out;
    a.out_head_cols = out_head_cols;
    a.out_rows_per_head = rows_per_head;
    a.partials = part;
    prof_mark(ctx, st, name);
    ctx->launches += 1;
    return check(wgemm_launch(p, WG_ROWMAJOR, false, st, true));
  };
  if (M <= kGemvMaxTokens) {
    // one or two tokens: matrix-vector products, bound by streaming the weights
    auto gemv = [&](const void* W, int R, int K, const __nv_bfloat16* x, __nv_bfloat16* out,
                    long long ldo, int rph, long long hs, const char* name) {
      GemvArgs g{static_cast<const __nv_bfloat16*>(W), R, K, M, x, (long long)K, R, 0, out,
                 ldo, rph, hs};
      if (!gemv_supported(g, ctx->num_sms)) return false;
      prof_mark(ctx, st, name);
      ctx->launches += 1;
      return check(gemv_launch(g, ctx->num_sms, st, true));
    };
    const GemvArgs probe_dq{nullptr, dcq, D, M, nullptr, D, dcq, 0, nullptr, dcq, 0, 0};
    const GemvArgs probe_uq{nullptr, kHeads * kNope, dcq, M, nullptr, dcq, kHeads * kNope, 0,
                            nullptr, kQRow, kNope, kNope + kRope};
    const GemvArgs probe_qr{nullptr, kHeads * kRope, D, M, nullptr, D, kHeads * kRope, 0,
                            nullptr, kQRow, kRope, kNope + kRope};
    if (gemv_supported(probe_dq, ctx->num_sms) && gemv_supported(probe_uq, ctx->num_sms) &&
        gemv_supported(probe_qr, ctx->num_sms)) {
      return gemv(ctx->w.w_dq, dcq, D, h, cq, dcq, 0, 0, "query_down") &&
             gemv(ctx->w.w_qr, kHeads * kRope, D, h, q + kNope, kQRow, kRope, kNope + kRope,
                  "query_rope") &&
             gemv(ctx->w.w_uq, kHeads * kNope, dcq, cq, q, kQRow, kNope, kNope + kRope,
                  "query_up");
    }
  }
  // c^Q [M, d_cq]
  if (!rowmajor(bp.dq, dcq / 128, ctx->tm_wdq, h, D, D / 64, dcq / 128, 0, cq, dcq, 0, 0,
                "query_down"))
    return false;
  // q^R (un-rotated) -> q[:, head, 128..191]
  if (!rowmajor(bp.qr, kHeads * kRope / 128, ctx->tm_wqr, h, D, D / 64, kHeads * kRope / 128, 0,
                q + kNope, kQRow, kNope + kRope, kRope, "query_rope"))
    return false;
  // q^C -> q[:, head, 0..127]
  return rowmajor(bp.uq, kHeads, ctx->tm_wuq, cq, dcq, dcq / 64, 1, kNope, q, kQRow,
                  kNope + kRope, 0, "query_up");
}

// out[t, f] = sum_k W[f, k] x[t, k] for the m_tiles * 128 rows of the weight
// map and k_chunks * 64 columns of x ([M, x_cols] row-major), out row-major
// with leading dimension ld_out.
bool bf16_rowmajor_gemm(mla_ctx* ctx, const CUtensorMap& wmap, int m_tiles, int k_chunks,
                        const __nv_bfloat16* x, int M, int x_cols, __nv_bfloat16* out,
                        int ld_out, float* part, cudaStream_t st, const char* name) {
  const GemmShape g = gemm_shape(ctx, M, m_tiles, k_chunks, 4, kSplitCap, true);
  if (g.n_tiles > 65535 || (g.splits > 1 && (long long)m_tiles * g.n_tiles > kCounters))
    return false;
  WgPlan p{};
  p.nt = g.nt;
  p.n_tiles = g.n_tiles;
  p.m_tiles = m_tiles;
  p.tmA = wmap;
  p.tmA2 = wmap;
  if (!make_tmap_bf16_2d(&p.tmB, x, M, x_cols, x_cols, 64, p.nt, false)) {
    cudaGetLastError();
    return false;
  }
  WgArgs& a = p.args;
  a = base_args(ctx);
  a.n_tokens = M;
  a.k_chunks = k_chunks;
  a.splits = g.splits;
  a.tiles_per_head = m_tiles;
  a.out = out;
  a.ld_out = ld_out;
  a.out_head_cols = 0;
  a.partials = part;
  prof_mark(ctx, st, name);
  ctx->launches += 1;
  return check(wgemm_launch(p, WG_ROWMAJOR, false, st, true));
}

size_t prefill_partial_bytes(const mla_ctx* ctx, int R, int M) {
  const int D = ctx->cfg.d_model;
  const GemmShape kv = gemm_shape(ctx, R, kHeads, kLat / 64, 4, kSplitCap, true);
  const GemmShape o = gemm_shape(ctx, M, D / 128, kHeads * kDv / 64, 4, kSplitCap, true);
  return std::max(partial_bytes(kv, kHeads), partial_bytes(o, D / 128));
}

bool bf16_append_decode(mla_ctx* ctx, const __nv_bfloat16* h, const int32_t* pos,
                        const __nv_bfloat16* q, __nv_bfloat16* cache, int num_pages,
                        const int32_t* bt, int max_pages, const int32_t* seq_lens, int B, int T,
                        __nv_bfloat16* out, char* ws, const WsLayout& L, cudaStream_t st) {
  if (kv_fp8(ctx) && B * T > kStageRows) {
    // more rows than one staging pass: append first, then decode
    return bf16_compress_append(ctx, h, B, T, pos, bt, max_pages, cache, num_pages, st) &&
           bf16_decode(ctx, q, cache, num_pages, bt, max_pages, seq_lens, B, T, out, ws, L, st);
  }
  WgPlan p;
  if (!append_plan(ctx, h, B, T, pos, bt, max_pages, kv_fp8(ctx) ? ctx->stage : cache, num_pages,
                   p))
    return false;
  p.args.stage_rows = kv_fp8(ctx) ? 1 : 0;
  return decode_impl(ctx, q, cache, num_pages, bt, max_pages, seq_lens, B, T, out, ws, L, st, &p,
                     h);
}

}  // namespace mla
