// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>

#include "mla.h"

// Status word layout on the device: [code, detail, count, spare].
enum { MLA_ST_CODE = 0, MLA_ST_DETAIL = 1, MLA_ST_COUNT = 2, MLA_ST_WORDS = 4 };

struct mla_ctx {
  mla_config cfg;
  mla_weights w;
  int device;
  int num_sms;
  float2* rope_cs;     // device [max_position, d_rope/2] of (cos, sin)
  int* status;         // device [MLA_ST_WORDS]
  int64_t launches;
  // bf16 path: TMA maps of the weights, split-K scratch of the append
  CUtensorMap tm_wdkv, tm_wkr, tm_wuk, tm_wuv, tm_wo;
  CUtensorMap tm_wuk_rows;              // W^UK with 128-row boxes (K^C = W^UK c)
  CUtensorMap tm_wdq, tm_wuq, tm_wqr;   // query path (d_cq > 0)
  float* append_partials = nullptr;   // kAppendPartialBytes
  // FP8 cache: bf16 rows [kStageRows, 576] of an append before quantisation
  __nv_bfloat16* stage = nullptr;
  int* counters = nullptr;            // kCounters, zero between launches
  // attention clusters that fit on the device at once: [0] two-CTA clusters
  // (odd T), [1] four-CTA clusters (even T)
  int sv_clusters[2] = {0, 0};
  // per-kernel timing (mla_profile_enable)
  bool prof = false;
  int n_marks = 0;
  cudaEvent_t marks[64];
  const char* mark_names[64];
};

namespace mla {

constexpr size_t kAppendPartialBytes = 8u << 20;
constexpr int kStageRows = 4096;        // tokens per FP8 append pass
constexpr int kF8Row = 656;             // bytes of an FP8 cache row
constexpr int kQ8Bytes = 82432;         // FP8 query image of one token
constexpr int kCounters = 65536;

// Byte layout of the decode workspace (all offsets 256-byte aligned).
struct WsLayout {
  int G;           // KV splits of the global page list
  int n_slots;     // partial-result slots (G + batch bounds the segment count)
  size_t lens, page_prefix, first_split, slot_base;   // int32 arrays
  size_t meta;     // int32 [4]: splits in use G_eff = min(G, pages), total pages
  size_t qfull;    // [batch*T, n_heads, R] query rows in the dtype (image layout for bf16)
  size_t part_o;   // fp32 [n_slots, T, n_heads, d_latent]
  size_t part_lse; // fp32 [n_slots, T, n_heads] (log2 domain)
  size_t o_lat;    // dtype [batch*T, n_heads, d_latent]
  size_t o;        // dtype [batch*T, n_heads*d_v]
  size_t wg_part;  // fp32 split-K partials of the projections
  size_t c_q;      // query path (d_cq > 0): dtype [batch*T, d_cq]
  size_t q_in;     // query path: dtype [batch*T, n_heads, d_nope + d_rope]
  size_t q8;       // FP8 cache: [batch*T] FP8 query images of kQ8Bytes
  size_t total;
};

// Record a timing mark on `st` when profiling is on: `name` is the kernel
// enqueued next, nullptr closes the previous one.
void prof_mark(mla_ctx* ctx, cudaStream_t st, const char* name);

WsLayout workspace_layout(const mla_ctx* ctx, int B, int T, int max_pages);

// Splits the global page list across G workers; see plan.cu.
void launch_plan(const mla_ctx* ctx, const WsLayout& L, char* ws, const int32_t* seq_lens,
                 int B, int T, int max_pages, cudaStream_t st);

// fp32 kernels (any small widths).
void f32_compress_append(mla_ctx* ctx, const float* h, int B, int T, const int32_t* pos,
                         const int32_t* bt, int max_pages, float* cache, int num_pages,
                         cudaStream_t st);
void f32_decode(mla_ctx* ctx, const float* q, const float* cache, int num_pages,
                const int32_t* bt, int max_pages, int B, int T, float* out, char* ws,
                const WsLayout& L, cudaStream_t st);

// bf16 kernels (DeepSeek-V2 head widths).
bool bf16_compress_append(mla_ctx* ctx, const __nv_bfloat16* h, int B, int T,
                          const int32_t* pos, const int32_t* bt, int max_pages,
                          __nv_bfloat16* cache, int num_pages, cudaStream_t st);
struct WgPlan;
// `append` (optional): the append step's GEMM plan, run in the same launch
// as the absorbed query (the two share no data).
bool bf16_decode(mla_ctx* ctx, const __nv_bfloat16* q, const __nv_bfloat16* cache,
                 int num_pages, const int32_t* bt, int max_pages, const int32_t* seq_lens,
                 int B, int T, __nv_bfloat16* out, char* ws, const WsLayout& L,
                 cudaStream_t st, const WgPlan* append = nullptr);
// Append the B*T new rows, then decode them (mla_append_decode).
bool bf16_append_decode(mla_ctx* ctx, const __nv_bfloat16* h, const int32_t* pos,
                        const __nv_bfloat16* q, __nv_bfloat16* cache, int num_pages,
                        const int32_t* bt, int max_pages, const int32_t* seq_lens, int B, int T,
                        __nv_bfloat16* out, char* ws, const WsLayout& L, cudaStream_t st);

// Prefill in the explicit form (prefill.cu): byte layout of its workspace.
struct PrefillLayout {
  int Smax;        // rows per sequence in the gathered buffers (max_pages * page)
  size_t rows;     // bf16 [B*Smax, 576] the cached rows of every sequence, zero padded
  size_t k;        // bf16 [B*Smax, n_heads*d_nope] K^C = W^UK c
  size_t v;        // bf16 [B*Smax, n_heads*d_v] V = W^UV c
  size_t q_rot;    // bf16 [B*T, n_heads, d_nope + d_rope] queries with q^R rotated
  size_t o;        // bf16 [B*T, n_heads*d_v]
  size_t wg_part;  // fp32 split-K partials
  size_t total;
};
PrefillLayout prefill_layout(const mla_ctx* ctx, int B, int T, int max_pages);
size_t prefill_partial_bytes(const mla_ctx* ctx, int R, int M);
bool bf16_prefill_explicit(mla_ctx* ctx, const __nv_bfloat16* q, const __nv_bfloat16* cache,
                           int num_pages, const int32_t* bt, int max_pages,
                           const int32_t* seq_lens, int B, int T, __nv_bfloat16* out, char* ws,
                           const PrefillLayout& L, cudaStream_t st);
bool bf16_rowmajor_gemm(mla_ctx* ctx, const CUtensorMap& wmap, int m_tiles, int k_chunks,
                        const __nv_bfloat16* x, int M, int x_cols, __nv_bfloat16* out,
                        int ld_out, float* part, cudaStream_t st, const char* name);

// Query path of mla_layer_step: q = [W^UQ W^DQ h ; W^QR h] per head into
// the workspace's q_in (layout of mla_decode's q).
bool bf16_query(mla_ctx* ctx, const __nv_bfloat16* h, int M, char* ws, const WsLayout& L,
                cudaStream_t st);
void f32_query(mla_ctx* ctx, const float* h, int M, char* ws, const WsLayout& L,
               cudaStream_t st);

// bf16 path helpers
bool bf16_setup(mla_ctx* ctx);                 // weight maps + scratch, at create
void bf16_teardown(mla_ctx* ctx);
size_t bf16_wg_partial_bytes(const mla_ctx* ctx, int M);
// Split-KV attention over the latent cache (attend_sv.cu): one cluster per
// (KV split, query token) for odd T, per (KV split, token pair) for even T.
bool sv_attend(mla_ctx* ctx, const __nv_bfloat16* qimg, const __nv_bfloat16* cache,
               int num_pages, const int32_t* bt, int max_pages, int B, int T, char* ws,
               const WsLayout& L, cudaStream_t st);
// Fills ctx->sv_clusters (at context creation).
bool sv_setup(mla_ctx* ctx);
// FP8 cache (attend_f8.cu).  f8_prepare quantises `rows` staged bf16 rows
// (tokens m0.. of the batch; none when rows == 0) into the pool and the M_q
// bf16 query images into FP8 query images, in one launch.
bool f8_prepare(mla_ctx* ctx, const __nv_bfloat16* stage, int rows, int m0, const int32_t* pos,
                const int32_t* bt, int T, int max_pages, uint8_t* cache8, int num_pages,
                const __nv_bfloat16* qimg, int M_q, uint8_t* q8img, cudaStream_t st);
// Split-KV attention over the FP8 pool: two CTAs (latent halves) per
// (KV split, query token).
bool f8_attend(mla_ctx* ctx, const uint8_t* q8img, const uint8_t* cache8, int num_pages,
               const int32_t* bt, int max_pages, int B, int T, char* ws, const WsLayout& L,
               cudaStream_t st);
inline bool kv_fp8(const mla_ctx* ctx) { return ctx->cfg.kv_dtype == MLA_KV_FP8; }

void launch_selftest_wait(const mla_ctx* ctx, int spin_limit, cudaStream_t st);

}  // namespace mla
