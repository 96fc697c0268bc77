// C ABI: argument validation, context, RoPE table and dispatch.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "mla_internal.h"

namespace {

struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { cudaGetLastError(); prev = -1; }
    ok = cudaSetDevice(dev) == cudaSuccess;
    if (!ok) cudaGetLastError();
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

mla_status validate_config(const mla_config* c) {
  if (c->d_model < 1 || c->n_heads < 1 || c->d_nope < 1 || c->d_v < 1 || c->d_latent < 1 ||
      c->d_rope < 2 || c->page_size < 1 || c->max_position < 1)
    return MLA_ERR_INVALID_ARG;
  if (c->d_rope % 2 != 0) return MLA_ERR_INVALID_ARG;
  if (!(c->softmax_scale > 0.f) || !std::isfinite(c->softmax_scale)) return MLA_ERR_INVALID_ARG;
  if (!(c->rope_base > 1.f) || !std::isfinite(c->rope_base)) return MLA_ERR_INVALID_ARG;
  if (c->max_position > (1 << 26)) return MLA_ERR_UNSUPPORTED;
  if (c->d_cq < 0) return MLA_ERR_INVALID_ARG;
  if (c->d_cq > (c->dtype == MLA_BF16 ? 16384 : 4096)) return MLA_ERR_UNSUPPORTED;
  if (c->dtype == MLA_BF16 && c->d_cq % 128 != 0) return MLA_ERR_UNSUPPORTED;
  if (c->dtype == MLA_BF16) {
    if (c->n_heads != 128 || c->d_nope != 128 || c->d_v != 128 || c->d_latent != 512 ||
        c->d_rope != 64 || c->page_size != 64 || c->d_model % 128 != 0 || c->d_model > 16384)
      return MLA_ERR_UNSUPPORTED;
  } else if (c->dtype == MLA_FP32) {
    if (c->n_heads > 128 || c->d_latent > 512 || c->d_latent + c->d_rope > 576 ||
        c->d_nope > 512 || c->d_v > 512 || c->d_latent % 2 != 0)
      return MLA_ERR_UNSUPPORTED;
  } else {
    return MLA_ERR_INVALID_ARG;
  }
  if (c->kv_dtype != MLA_KV_NATIVE && c->kv_dtype != MLA_KV_FP8) return MLA_ERR_INVALID_ARG;
  if (c->kv_dtype == MLA_KV_FP8 && c->dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

mla_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

namespace mla {
void prof_mark(mla_ctx* ctx, cudaStream_t st, const char* name) {
  if (!ctx->prof || ctx->n_marks >= 64) return;
  // inside stream capture the mark must become an event-record node of the graph
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) cudaGetLastError();
  const cudaError_t e = cs == cudaStreamCaptureStatusActive
                            ? cudaEventRecordWithFlags(ctx->marks[ctx->n_marks], st,
                                                       cudaEventRecordExternal)
                            : cudaEventRecord(ctx->marks[ctx->n_marks], st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  ctx->mark_names[ctx->n_marks++] = name;
}
}  // namespace mla

extern "C" {

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_DEVICE_INDEX: return "MLA_ERR_DEVICE_INDEX";
  }
  return "MLA_ERR_UNKNOWN";
}

mla_status mla_create(const mla_config* cfg, const mla_weights* w, int device, mla_ctx** out) {
  if (!cfg || !w || !out) return MLA_ERR_INVALID_ARG;
  *out = nullptr;
  mla_status s = validate_config(cfg);
  if (s != MLA_OK) return s;
  if (!w->w_dkv || !w->w_kr || !w->w_uk || !w->w_uv || !w->w_o) return MLA_ERR_INVALID_ARG;
  const size_t align = cfg->dtype == MLA_BF16 ? 16 : 4;
  if (!aligned(w->w_dkv, align) || !aligned(w->w_kr, align) || !aligned(w->w_uk, align) ||
      !aligned(w->w_uv, align) || !aligned(w->w_o, align))
    return MLA_ERR_INVALID_ARG;
  if (cfg->d_cq > 0 && (!w->w_dq || !w->w_uq || !w->w_qr || !aligned(w->w_dq, align) ||
                        !aligned(w->w_uq, align) || !aligned(w->w_qr, align)))
    return MLA_ERR_INVALID_ARG;
  if (device < 0) return MLA_ERR_INVALID_ARG;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess) { cudaGetLastError(); return MLA_ERR_CUDA; }
  if (device >= ndev) return MLA_ERR_INVALID_ARG;
  DeviceGuard g(device);
  if (!g.ok) return MLA_ERR_CUDA;
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (major != 10 || minor != 3) return MLA_ERR_UNSUPPORTED;   // built for sm_103a only

  mla_ctx* ctx = new (std::nothrow) mla_ctx();
  if (!ctx) return MLA_ERR_CUDA;
  ctx->cfg = *cfg;
  ctx->w = *w;
  ctx->device = device;
  ctx->num_sms = sms;

  // RoPE table: angle pos * base^(-2j/d_R), computed in float64.
  const int half = cfg->d_rope / 2;
  std::vector<float2> tab((size_t)cfg->max_position * half);
  for (int j = 0; j < half; ++j) {
    const double theta = std::pow((double)cfg->rope_base, -2.0 * j / cfg->d_rope);
    for (int p = 0; p < cfg->max_position; ++p) {
      const double a = (double)p * theta;
      tab[(size_t)p * half + j] = make_float2((float)std::cos(a), (float)std::sin(a));
    }
  }
  if (cudaMalloc(&ctx->rope_cs, tab.size() * sizeof(float2)) != cudaSuccess ||
      cudaMemcpy(ctx->rope_cs, tab.data(), tab.size() * sizeof(float2),
                 cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMalloc(&ctx->status, MLA_ST_WORDS * sizeof(int)) != cudaSuccess ||
      cudaMemset(ctx->status, 0, MLA_ST_WORDS * sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    if (ctx->rope_cs) cudaFree(ctx->rope_cs);
    if (ctx->status) cudaFree(ctx->status);
    delete ctx;
    return MLA_ERR_CUDA;
  }
  if (cfg->dtype == MLA_BF16 && !mla::bf16_setup(ctx)) {
    mla::bf16_teardown(ctx);
    cudaFree(ctx->rope_cs);
    cudaFree(ctx->status);
    delete ctx;
    return MLA_ERR_CUDA;
  }
  *out = ctx;
  return MLA_OK;
}

mla_status mla_destroy(mla_ctx* ctx) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  cudaDeviceSynchronize();
  mla_profile_enable(ctx, 0);
  mla::bf16_teardown(ctx);
  cudaFree(ctx->rope_cs);
  cudaFree(ctx->status);
  delete ctx;
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

mla_status mla_compress_append(mla_ctx* ctx, const void* h, int batch, int T,
                               const int32_t* positions, const int32_t* block_table,
                               int max_pages, void* cache, int num_pages, void* stream) {
  if (!ctx || !h || !positions || !block_table || !cache) return MLA_ERR_INVALID_ARG;
  if (batch < 1 || T < 1 || max_pages < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if ((long long)batch * T > (1LL << 30)) return MLA_ERR_INVALID_ARG;
  const size_t a = ctx->cfg.dtype == MLA_BF16 ? 16 : 4;
  if (!aligned(h, a) || !aligned(cache, a) || !aligned(positions, 4) || !aligned(block_table, 4))
    return MLA_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return MLA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bool launched = true;
  if (ctx->cfg.dtype == MLA_BF16) {
    launched = mla::bf16_compress_append(ctx, static_cast<const __nv_bfloat16*>(h), batch, T, positions,
                              block_table, max_pages, static_cast<__nv_bfloat16*>(cache),
                              num_pages, st);
  } else {
    mla::f32_compress_append(ctx, static_cast<const float*>(h), batch, T, positions,
                             block_table, max_pages, static_cast<float*>(cache), num_pages, st);
  }
  mla::prof_mark(ctx, st, nullptr);
  if (!launched) { cudaGetLastError(); return MLA_ERR_CUDA; }
  return launch_status();
}

size_t mla_decode_workspace_size(const mla_ctx* ctx, int batch, int T, int max_pages) {
  if (!ctx || batch < 1 || T < 1 || max_pages < 1) return 0;
  return mla::workspace_layout(ctx, batch, T, max_pages).total;
}

mla_status mla_decode_workspace_offsets(const mla_ctx* ctx, int batch, int T, int max_pages,
                                        size_t* o_lat_offset, size_t* o_offset) {
  if (!ctx || batch < 1 || T < 1 || max_pages < 1 || !o_lat_offset || !o_offset)
    return MLA_ERR_INVALID_ARG;
  const mla::WsLayout L = mla::workspace_layout(ctx, batch, T, max_pages);
  *o_lat_offset = L.o_lat;
  *o_offset = L.o;
  return MLA_OK;
}

mla_status mla_decode(mla_ctx* ctx, const void* q, const void* cache, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                      int batch, int T, void* out, void* workspace, size_t workspace_bytes,
                      void* stream) {
  if (!ctx || !q || !cache || !block_table || !seq_lens || !out || !workspace)
    return MLA_ERR_INVALID_ARG;
  if (batch < 1 || T < 1 || max_pages < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (T > 8 || (long long)batch * max_pages > (1LL << 30)) return MLA_ERR_INVALID_ARG;
  const size_t a = ctx->cfg.dtype == MLA_BF16 ? 16 : 4;
  if (!aligned(q, a) || !aligned(cache, a) || !aligned(out, a) || !aligned(workspace, 256) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return MLA_ERR_INVALID_ARG;
  const mla::WsLayout L = mla::workspace_layout(ctx, batch, T, max_pages);
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE;
  DeviceGuard g(ctx->device);
  if (!g.ok) return MLA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  bool launched = true;
  if (ctx->cfg.dtype == MLA_BF16) {
    launched = mla::bf16_decode(ctx, static_cast<const __nv_bfloat16*>(q),
                                static_cast<const __nv_bfloat16*>(cache), num_pages, block_table,
                                max_pages, seq_lens, batch, T, static_cast<__nv_bfloat16*>(out),
                                ws, L, st);
  } else {
    mla::prof_mark(ctx, st, "plan");
    mla::launch_plan(ctx, L, ws, seq_lens, batch, T, max_pages, st);
    ctx->launches += 1;
    mla::f32_decode(ctx, static_cast<const float*>(q), static_cast<const float*>(cache),
                    num_pages, block_table, max_pages, batch, T, static_cast<float*>(out), ws,
                    L, st);
  }
  mla::prof_mark(ctx, st, nullptr);
  if (!launched) { cudaGetLastError(); return MLA_ERR_CUDA; }
  return launch_status();
}

mla_status mla_append_decode(mla_ctx* ctx, const void* h, const int32_t* positions,
                             const void* q, void* cache, int num_pages,
                             const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                             int batch, int T, void* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!ctx || !h || !positions || !q || !cache || !block_table || !seq_lens || !out ||
      !workspace)
    return MLA_ERR_INVALID_ARG;
  if (batch < 1 || T < 1 || max_pages < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (T > 8 || (long long)batch * max_pages > (1LL << 30)) return MLA_ERR_INVALID_ARG;
  const size_t a = ctx->cfg.dtype == MLA_BF16 ? 16 : 4;
  if (!aligned(h, a) || !aligned(q, a) || !aligned(cache, a) || !aligned(out, a) ||
      !aligned(workspace, 256) || !aligned(positions, 4) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4))
    return MLA_ERR_INVALID_ARG;
  const mla::WsLayout L = mla::workspace_layout(ctx, batch, T, max_pages);
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE;
  DeviceGuard g(ctx->device);
  if (!g.ok) return MLA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  bool launched = true;
  if (ctx->cfg.dtype == MLA_BF16) {
    launched = mla::bf16_append_decode(
        ctx, static_cast<const __nv_bfloat16*>(h), positions, static_cast<const __nv_bfloat16*>(q),
        static_cast<__nv_bfloat16*>(cache), num_pages, block_table, max_pages, seq_lens, batch, T,
        static_cast<__nv_bfloat16*>(out), ws, L, st);
  } else {
    mla::f32_compress_append(ctx, static_cast<const float*>(h), batch, T, positions, block_table,
                             max_pages, static_cast<float*>(cache), num_pages, st);
    mla::prof_mark(ctx, st, "plan");
    mla::launch_plan(ctx, L, ws, seq_lens, batch, T, max_pages, st);
    ctx->launches += 1;
    mla::f32_decode(ctx, static_cast<const float*>(q), static_cast<const float*>(cache),
                    num_pages, block_table, max_pages, batch, T, static_cast<float*>(out), ws,
                    L, st);
  }
  mla::prof_mark(ctx, st, nullptr);
  if (!launched) { cudaGetLastError(); return MLA_ERR_CUDA; }
  return launch_status();
}

mla_status mla_layer_step(mla_ctx* ctx, const void* h, const int32_t* positions, void* cache,
                          int num_pages, const int32_t* block_table, int max_pages,
                          const int32_t* seq_lens, int batch, int T, void* out, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (!ctx || !h || !positions || !cache || !block_table || !seq_lens || !out || !workspace)
    return MLA_ERR_INVALID_ARG;
  if (ctx->cfg.d_cq <= 0) return MLA_ERR_UNSUPPORTED;
  if (batch < 1 || T < 1 || max_pages < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (T > 8 || (long long)batch * max_pages > (1LL << 30)) return MLA_ERR_INVALID_ARG;
  const size_t a = ctx->cfg.dtype == MLA_BF16 ? 16 : 4;
  if (!aligned(h, a) || !aligned(cache, a) || !aligned(out, a) || !aligned(workspace, 256) ||
      !aligned(positions, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return MLA_ERR_INVALID_ARG;
  const mla::WsLayout L = mla::workspace_layout(ctx, batch, T, max_pages);
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE;
  DeviceGuard g(ctx->device);
  if (!g.ok) return MLA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int M = batch * T;
  bool launched = true;
  if (ctx->cfg.dtype == MLA_BF16) {
    const __nv_bfloat16* hb = static_cast<const __nv_bfloat16*>(h);
    launched = mla::bf16_query(ctx, hb, M, ws, L, st) &&
               mla::bf16_append_decode(
                   ctx, hb, positions, reinterpret_cast<const __nv_bfloat16*>(ws + L.q_in),
                   static_cast<__nv_bfloat16*>(cache), num_pages, block_table, max_pages, seq_lens,
                   batch, T, static_cast<__nv_bfloat16*>(out), ws, L, st);
  } else {
    const float* hf = static_cast<const float*>(h);
    mla::f32_query(ctx, hf, M, ws, L, st);
    mla::f32_compress_append(ctx, hf, batch, T, positions, block_table, max_pages,
                             static_cast<float*>(cache), num_pages, st);
    mla::prof_mark(ctx, st, "plan");
    mla::launch_plan(ctx, L, ws, seq_lens, batch, T, max_pages, st);
    ctx->launches += 1;
    mla::f32_decode(ctx, reinterpret_cast<const float*>(ws + L.q_in),
                    static_cast<const float*>(cache), num_pages, block_table, max_pages, batch, T,
                    static_cast<float*>(out), ws, L, st);
  }
  mla::prof_mark(ctx, st, nullptr);
  if (!launched) { cudaGetLastError(); return MLA_ERR_CUDA; }
  return launch_status();
}

// The explicit form holds the up-projected keys and values of every cached
// row (32 KB per row): at most this many rows per call.
constexpr long long kExplicitRows = 1LL << 18;

static bool explicit_fits(const mla_ctx* ctx, int batch, int max_pages) {
  return ctx->cfg.dtype == MLA_BF16 && ctx->cfg.kv_dtype == MLA_KV_NATIVE &&
         (long long)batch * max_pages * ctx->cfg.page_size <= kExplicitRows;
}

size_t mla_prefill_workspace_size(const mla_ctx* ctx, int batch, int T, int max_pages) {
  if (!ctx || batch < 1 || T < 1 || max_pages < 1) return 0;
  size_t n = mla::workspace_layout(ctx, batch, T, max_pages).total;
  if (explicit_fits(ctx, batch, max_pages))
    n = std::max(n, mla::prefill_layout(ctx, batch, T, max_pages).total);
  return n;
}

// Estimated time of the two forms for `batch` sequences of T new tokens
// each against up to S keys, from per-unit costs of this library's kernels
// measured on B300 at DeepSeek-V2 widths (ns).  Explicit: 65 per cached key
// (gather, K^C and V up-projections), 16 per query token (rotated queries),
// 0.08 per visible (query, key) pair (2·128·320 FLOP).  Absorbed: 190 per
// query token (absorbed query, combine, W^UV) and 0.24 per pair
// (2·128·1088 FLOP).  The append and W_O are common to both.
static bool explicit_is_cheaper(int batch, int T, long long S) {
  const double B = batch, t = T, s = (double)S;
  const double pairs = B * t * (s - 0.5 * (t - 1.0));
  const double expl = 65.0 * B * s + 16.0 * B * t + 0.08 * pairs;
  const double absd = 190.0 * B * t + 0.24 * pairs;
  return expl < absd;
}

static int prefill_form(const mla_ctx* ctx, int batch, int T, int max_pages) {
  return explicit_fits(ctx, batch, max_pages) &&
                 explicit_is_cheaper(batch, T, (long long)max_pages * ctx->cfg.page_size)
             ? MLA_FORM_EXPLICIT
             : MLA_FORM_ABSORBED;
}

int mla_prefill_form(const mla_ctx* ctx, int batch, int T, int max_pages) {
  if (!ctx || batch < 1 || T < 1 || max_pages < 1) return -1;
  return prefill_form(ctx, batch, T, max_pages);
}

mla_status mla_prefill(mla_ctx* ctx, const void* h, const int32_t* positions, const void* q,
                       void* cache, int num_pages, const int32_t* block_table, int max_pages,
                       const int32_t* seq_lens, int batch, int T, int form, void* out,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!ctx || !h || !positions || !q || !cache || !block_table || !seq_lens || !out ||
      !workspace)
    return MLA_ERR_INVALID_ARG;
  if (batch < 1 || T < 1 || T > 4096 || max_pages < 1 || num_pages < 1) return MLA_ERR_INVALID_ARG;
  if ((long long)batch * max_pages > (1LL << 30) || (long long)batch * T > 32768)
    return MLA_ERR_INVALID_ARG;
  if (form < MLA_FORM_AUTO || form > MLA_FORM_ABSORBED) return MLA_ERR_INVALID_ARG;
  const bool bf = ctx->cfg.dtype == MLA_BF16;
  if ((!bf || ctx->cfg.kv_dtype != MLA_KV_NATIVE) && form == MLA_FORM_EXPLICIT)
    return MLA_ERR_UNSUPPORTED;
  if (form == MLA_FORM_EXPLICIT && !explicit_fits(ctx, batch, max_pages))
    return MLA_ERR_INVALID_ARG;
  const size_t a = bf ? 16 : 4;
  if (!aligned(h, a) || !aligned(q, a) || !aligned(cache, a) || !aligned(out, a) ||
      !aligned(workspace, 256) || !aligned(positions, 4) || !aligned(block_table, 4) ||
      !aligned(seq_lens, 4))
    return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < mla_prefill_workspace_size(ctx, batch, T, max_pages))
    return MLA_ERR_WORKSPACE;
  const bool expl = form == MLA_FORM_EXPLICIT ||
                    (form == MLA_FORM_AUTO &&
                     prefill_form(ctx, batch, T, max_pages) == MLA_FORM_EXPLICIT);
  DeviceGuard g(ctx->device);
  if (!g.ok) return MLA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  bool launched = true;
  if (expl) {
    const mla::PrefillLayout L = mla::prefill_layout(ctx, batch, T, max_pages);
    launched = mla::bf16_compress_append(ctx, static_cast<const __nv_bfloat16*>(h), batch, T,
                                         positions, block_table, max_pages,
                                         static_cast<__nv_bfloat16*>(cache), num_pages, st) &&
               mla::bf16_prefill_explicit(ctx, static_cast<const __nv_bfloat16*>(q),
                                          static_cast<const __nv_bfloat16*>(cache), num_pages,
                                          block_table, max_pages, seq_lens, batch, T,
                                          static_cast<__nv_bfloat16*>(out), ws, L, st);
  } else {
    const mla::WsLayout L = mla::workspace_layout(ctx, batch, T, max_pages);
    if (bf) {
      launched = mla::bf16_append_decode(
          ctx, static_cast<const __nv_bfloat16*>(h), positions,
          static_cast<const __nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(cache), num_pages,
          block_table, max_pages, seq_lens, batch, T, static_cast<__nv_bfloat16*>(out), ws, L, st);
    } else {
      mla::f32_compress_append(ctx, static_cast<const float*>(h), batch, T, positions, block_table,
                               max_pages, static_cast<float*>(cache), num_pages, st);
      mla::prof_mark(ctx, st, "plan");
      mla::launch_plan(ctx, L, ws, seq_lens, batch, T, max_pages, st);
      ctx->launches += 1;
      mla::f32_decode(ctx, static_cast<const float*>(q), static_cast<const float*>(cache),
                      num_pages, block_table, max_pages, batch, T, static_cast<float*>(out), ws,
                      L, st);
    }
  }
  mla::prof_mark(ctx, st, nullptr);
  if (!launched) { cudaGetLastError(); return MLA_ERR_CUDA; }
  return launch_status();
}

mla_status mla_check_status(mla_ctx* ctx, void* stream) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  int words[MLA_ST_WORDS] = {0, 0, 0, 0};
  if (cudaMemcpy(words, ctx->status, sizeof(words), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(ctx->status, 0, sizeof(words)) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return static_cast<mla_status>(words[MLA_ST_CODE]);
}

int64_t mla_launch_count(const mla_ctx* ctx) { return ctx ? ctx->launches : -1; }

mla_status mla_profile_enable(mla_ctx* ctx, int enable) {
  if (!ctx) return MLA_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return MLA_ERR_CUDA;
  if (enable && ctx->prof) {
    ctx->n_marks = 0;
  } else if (enable && !ctx->prof) {
    for (int i = 0; i < 64; ++i) {
      if (cudaEventCreate(&ctx->marks[i]) != cudaSuccess) {
        cudaGetLastError();
        for (int j = 0; j < i; ++j) cudaEventDestroy(ctx->marks[j]);
        return MLA_ERR_CUDA;
      }
    }
    ctx->prof = true;
    ctx->n_marks = 0;
  } else if (!enable && ctx->prof) {
    for (int i = 0; i < 64; ++i) cudaEventDestroy(ctx->marks[i]);
    ctx->prof = false;
    ctx->n_marks = 0;
  }
  return MLA_OK;
}

int mla_profile_read(mla_ctx* ctx, float* ms, const char** names, int max_kernels) {
  if (!ctx || !ms || !names || max_kernels < 0 || !ctx->prof) return -1;
  DeviceGuard g(ctx->device);
  if (!g.ok) return -1;
  int n = 0;
  if (ctx->n_marks > 0 && cudaEventSynchronize(ctx->marks[ctx->n_marks - 1]) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  for (int i = 0; i + 1 < ctx->n_marks && n < max_kernels; ++i) {
    if (!ctx->mark_names[i]) continue;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, ctx->marks[i], ctx->marks[i + 1]) != cudaSuccess) {
      cudaGetLastError();
      t = -1.f;
    }
    ms[n] = t;
    names[n] = ctx->mark_names[i];
    ++n;
  }
  return n;
}

mla_status mla_selftest_bounded_wait(mla_ctx* ctx, int spin_limit, void* stream) {
  if (!ctx || spin_limit < 1) return MLA_ERR_INVALID_ARG;
  DeviceGuard g(ctx->device);
  if (!g.ok) return MLA_ERR_CUDA;
  mla::launch_selftest_wait(ctx, spin_limit, static_cast<cudaStream_t>(stream));
  ctx->launches += 1;
  return launch_status();
}

}  // extern "C"
