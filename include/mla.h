/*
 * mla.h -- C ABI of a single-GPU Multi-head Latent Attention (MLA) decode
 * library for NVIDIA B300 (sm_103a).
 *
 * What the library computes is the DeepSeek-V2 form of MLA as stated on the
 * page "DeepSeek-V2：在“大力出奇迹”的AI军备竞赛中，四两拨千斤" (liang.world),
 * 第二章 "侠客甲——MLA" §1-§3, and restated on "DeepSeek 系列模型技术深度解读"
 * (tuntang.top), section "Multi-head Latent Attention (MLA)":
 *
 *   per token:  c^KV = W^DKV h,  k^R = RoPE_pos(W^KR h)          (cached)
 *   per query:  q_i = [q^C_i ; RoPE_pos(q^R_i)],
 *               k_{p,i} = [W^UK_i c_p ; k^R_p],  v_{p,i} = W^UV_i c_p,
 *               o_i = softmax_p(q_i . k_{p,i} * scale) . v_{.,i},
 *               u = W_O [o_1; ...; o_{n_h}].
 *
 * Only the 576-wide row [c^KV ; k^R] is cached per token (bf16: 1152 bytes).
 * Decode never forms K or V: W^UK is folded into the query and W^UV is
 * applied to the attention output (the absorption paragraph of §2).
 *
 * Conventions for every call:
 *  - Pointers marked "device" are CUDA device pointers on the context's
 *    device; the caller owns them and keeps them alive until the work that
 *    uses them has finished on the stream.  The context borrows the weight
 *    pointers from mla_create until mla_destroy.
 *  - All matrices are row-major.  Matrices act on column vectors ("W h"):
 *      w_dkv [d_latent, d_model]          w_kr [d_rope, d_model]
 *      w_uk  [n_heads*d_nope, d_latent]   w_uv [n_heads*d_v, d_latent]
 *      w_o   [d_model, n_heads*d_v]
 *    Head i owns rows i*d_nope.. of w_uk and i*d_v.. of w_uv.
 *  - Element type of every float buffer is the context dtype (bf16 or
 *    fp32).  Index buffers are int32.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work and never synchronise, except mla_check_status.
 *  - Argument errors are returned before anything is enqueued.  Errors found
 *    on the device (a page id or length out of range, a bounded wait that
 *    gave up) set a status word on the device; the offending access is
 *    skipped and mla_check_status reports the error.  No call traps,
 *    asserts or exits.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer  */
  MLA_ERR_UNSUPPORTED = 2,   /* widths or device this build does not serve */
  MLA_ERR_CUDA = 3,          /* a CUDA runtime call failed                 */
  MLA_ERR_WORKSPACE = 4,     /* workspace smaller than mla_decode_workspace_size */
  MLA_ERR_TIMEOUT = 5,       /* a device-side bounded wait gave up         */
  MLA_ERR_DEVICE_INDEX = 6   /* device saw a page id / length out of range */
} mla_status;

typedef enum { MLA_BF16 = 0, MLA_FP32 = 1 } mla_dtype;

/* Model widths.  bf16 contexts run the tensor-core kernels and need the
 * DeepSeek-V2 head widths: n_heads 128, d_nope 128, d_v 128, d_latent 512,
 * d_rope 64, page_size 64, and d_model a multiple of 128 (<= 16384).
 * fp32 contexts run plain fp32 kernels for small widths: n_heads <= 128,
 * d_latent <= 512, d_latent + d_rope <= 576, d_rope even, d_nope, d_v
 * <= 512, any page_size >= 1.  softmax_scale is applied to q.k; the pages
 * give none (1/sqrt(d_nope + d_rope) is the usual choice).  rope_base is
 * the RoPE frequency base; positions must stay below max_position. */
typedef struct {
  int d_model;
  int n_heads;
  int d_nope;
  int d_v;
  int d_latent;
  int d_rope;
  int page_size;
  int max_position;
  float softmax_scale;
  float rope_base;
  mla_dtype dtype;
  /* Width d_c' of the query latent c^Q = W^DQ h, for mla_layer_step; 0 when
   * the context decodes from given queries only.  The pages give no value.
   * bf16 contexts need a multiple of 128 (<= 16384); fp32 any width
   * <= 4096. */
  int d_cq;
  /* Storage of the latent cache rows: MLA_KV_NATIVE (the context dtype,
   * (d_latent + d_rope) elements per row) or MLA_KV_FP8 (bf16 contexts at
   * DeepSeek-V2 widths only).  An FP8 row is 656 bytes:
   *   bytes   0..511  the 512 latent values c^KV as E4M3 codes (OCP OFP8
   *                   E4M3: bias 7, 3 mantissa bits, largest value 448),
   *   bytes 512..639  the 64 RoPE-key values k^R as bf16, divided by s,
   *   bytes 640..643  s (fp32), bytes 644..655 zero,
   * standing for [s * E4M3(code_i) ; s * stored_j].  s = amax / 448 with
   * amax = max |c_i| of the row as produced in bf16 (s = 1 for a zero
   * row), code_i = E4M3(c_i * (448 / amax)) rounded to nearest-even with
   * saturation, each quotient and product rounded to fp32.  The pages name
   * FP8 for the attention GEMMs of the forward pass (tuntang.top
   * "DeepSeek 系列模型技术深度解读", "FP8 混合精度训练") but give no scaling
   * scheme for a cache; this per-row one lets the score contraction run on
   * the E4M3 codes with a single accumulator. */
  int kv_dtype;
} mla_config;

enum { MLA_KV_NATIVE = 0, MLA_KV_FP8 = 1 };
#define MLA_FP8_ROW_BYTES 656

/* Device pointers to the projection matrices (layouts above).  The last
 * three (query path, mla_layer_step) are read only when d_cq > 0:
 *      w_dq [d_cq, d_model]   w_uq [n_heads*d_nope, d_cq]
 *      w_qr [n_heads*d_rope, d_model]
 * head i owning rows i*d_nope.. of w_uq and i*d_rope.. of w_qr. */
typedef struct {
  const void* w_dkv;
  const void* w_kr;
  const void* w_uk;
  const void* w_uv;
  const void* w_o;
  const void* w_dq;
  const void* w_uq;
  const void* w_qr;
} mla_weights;

typedef struct mla_ctx mla_ctx;

/* Create a context on CUDA device `device`: validates the widths, builds
 * the RoPE cos/sin table (float64 on the host, stored as fp32 on the
 * device, [max_position, d_rope/2]) and allocates the device status word.
 * The weights are borrowed, not copied.  On success *out owns those two
 * allocations until mla_destroy. */
mla_status mla_create(const mla_config* cfg, const mla_weights* weights,
                      int device, mla_ctx** out);

/* Free what mla_create allocated.  Synchronises the device first. */
mla_status mla_destroy(mla_ctx* ctx);

/* Compress + RoPE + paged append (liang.world ch.2 §2, §3; the RoPE key is
 * cached with the latent, www.pptc.cn/news/140720 §3.4).
 *   h           device, [batch*T, d_model]; row b*T+t is token t of
 *               sequence b.
 *   positions   device int32 [batch*T]: position of each token (0-based,
 *               < max_position).
 *   block_table device int32 [batch, max_pages]: physical page of each
 *               logical page of each sequence.
 *   cache       device, [num_pages*page_size, d_latent+d_rope], the pool
 *               (rows of MLA_FP8_ROW_BYTES bytes with MLA_KV_FP8).
 * Writes row [W^DKV h ; RoPE_pos(W^KR h)] (fp32 accumulation, rounded once
 * to the context dtype; with MLA_KV_FP8 rounded to bf16, then quantised as
 * the kv_dtype comment states) to pool row
 *   block_table[b][pos / page_size] * page_size + pos % page_size.
 * Rows of other tokens are untouched.  A page id outside [0, num_pages) or
 * a position out of range skips that token and sets MLA_ERR_DEVICE_INDEX.
 * Any batch*T >= 1 is accepted (prefill chunks included). */
mla_status mla_compress_append(mla_ctx* ctx, const void* h, int batch, int T,
                               const int32_t* positions,
                               const int32_t* block_table, int max_pages,
                               void* cache, int num_pages, void* stream);

/* Bytes of scratch memory mla_decode needs for this batch shape. */
size_t mla_decode_workspace_size(const mla_ctx* ctx, int batch, int T,
                                 int max_pages);

/* Absorbed decode of the last T tokens of each sequence (liang.world ch.2
 * §1-§3; absorption of W^UK into the query and of W^UV after attention).
 *   q          device, [batch, T, n_heads, d_nope + d_rope]: q^C then the
 *              un-rotated q^R of each head.
 *   cache      device pool as written by mla_compress_append (the T query
 *              tokens must already be appended).
 *   seq_lens   device int32 [batch]: cached tokens per sequence, the query
 *              tokens included.  Query t of sequence b sits at position
 *              seq_lens[b] - T + t and attends to positions 0..itself.
 *   out        device, [batch, T, d_model]: u = W_O [o_1 ... o_{n_h}].
 *   workspace  device scratch of at least mla_decode_workspace_size bytes,
 *              256-byte aligned; its contents need not be initialised.
 * 1 <= T <= 8 (longer chunks go through mla_prefill): other T, a null or
 * misaligned pointer return MLA_ERR_INVALID_ARG before anything is enqueued.
 * A length outside [T, max_pages*page_size] or a bad page id sets
 * MLA_ERR_DEVICE_INDEX on the device; the bad part is skipped. */
mla_status mla_decode(mla_ctx* ctx, const void* q, const void* cache,
                      int num_pages, const int32_t* block_table, int max_pages,
                      const int32_t* seq_lens, int batch, int T, void* out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* One decode step: mla_compress_append of the batch*T new tokens followed by
 * mla_decode of the same tokens, with the arguments, layouts, ownership and
 * error behaviour of those two calls (normally positions[b*T+t] =
 * seq_lens[b] - T + t).  Results are those of the two calls bit for bit;
 * the library may overlap the append with the absorbed-query step, which
 * does not read the cache. */
mla_status mla_append_decode(mla_ctx* ctx, const void* h, const int32_t* positions,
                             const void* q, void* cache, int num_pages,
                             const int32_t* block_table, int max_pages,
                             const int32_t* seq_lens, int batch, int T, void* out,
                             void* workspace, size_t workspace_bytes, void* stream);

/* One decode step of the attention layer from the hidden states alone:
 * the query path, then mla_append_decode.  The query of new token t of
 * sequence b comes from its hidden state h_t (the row appended to the
 * cache) as the pages give it (liang.world ch.2 §2, last paragraph: the
 * query's own low-rank compression c^Q; tuntang.top, "RoPE 的兼容性处理":
 * q_t = [W^UQ c_t^Q ; W^QR h_t . RoPE(t)]):
 *   c^Q = W^DQ h,  q^C_i = (W^UQ c^Q)_i,  q^R_i = (W^QR h)_i rotated at the
 *   token's position,
 * then q_i = [q^C_i ; q^R_i] is decoded as by mla_decode.  W^UK is folded
 * into the query after W^UQ (the same absorption as mla_decode).
 * Arguments, layouts, ownership and errors are those of mla_append_decode
 * without `q`; the context needs d_cq > 0 (else MLA_ERR_UNSUPPORTED), and
 * the workspace (mla_decode_workspace_size) then also holds c^Q and q. */
mla_status mla_layer_step(mla_ctx* ctx, const void* h, const int32_t* positions,
                          void* cache, int num_pages, const int32_t* block_table,
                          int max_pages, const int32_t* seq_lens, int batch,
                          int T, void* out, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Prefill: the new tokens come in chunks of T per sequence (T up to 4096),
 * appended and attended to with the causal mask inside the chunk: the
 * results are those of mla_append_decode of the same T tokens.  The pages
 * warn that the absorbed form is not always the fastest
 * (www.pptc.cn/news/140720 §6 问题三): recovering K and V pays off when many
 * queries share them.  `form` chooses how the attention is computed:
 *   MLA_FORM_ABSORBED  the decode path (W^UK folded into the queries, every
 *                      query scoring the 576-wide rows directly);
 *   MLA_FORM_EXPLICIT  K^C_i = W^UK_i c and V_i = W^UV_i c for every cached
 *                      row, then per-head causal attention over
 *                      [K^C_i ; k^R] (192 features) and V_i (bf16 only);
 *   MLA_FORM_AUTO      the form mla_prefill_form names for this shape.
 * Arguments as for mla_append_decode (q: [batch, T, n_heads, 192]) with
 * T <= 4096 and batch·T <= 32768; the workspace must hold
 * mla_prefill_workspace_size bytes (MLA_ERR_WORKSPACE otherwise).  The
 * explicit form's buffers: the gathered rows, K^C and V of every row of
 * the batch (batch·max_pages·page_size rows of 1152 + 2·32768 bytes), the
 * rotated queries and the per-head outputs.  MLA_ERR_UNSUPPORTED for
 * MLA_FORM_EXPLICIT on an fp32 context or an FP8 cache (the explicit form
 * reads bf16 rows), MLA_ERR_INVALID_ARG for it past
 * the row bound.  Device-side index errors are reported as for
 * mla_append_decode. */
enum { MLA_FORM_AUTO = 0, MLA_FORM_EXPLICIT = 1, MLA_FORM_ABSORBED = 2 };

size_t mla_prefill_workspace_size(const mla_ctx* ctx, int batch, int T,
                                  int max_pages);

/* The form MLA_FORM_AUTO takes for this shape (MLA_FORM_EXPLICIT or
 * MLA_FORM_ABSORBED; -1 for invalid arguments): the one with the smaller
 * estimated time, from per-unit costs of the two forms' kernels measured on
 * B300 at DeepSeek-V2 widths.  The explicit form pays per cached key (the
 * K^C and V up-projections, 2·2·512·16384 FLOP) and less per (query, key)
 * pair (2·n_h·320 FLOP against 2·n_h·1088); the absorbed form pays per query
 * token (absorbed query, combine, W^UV).  With S = max_pages·page_size keys
 * per sequence: the explicit form for prompts on an empty cache from a few
 * dozen tokens up, the absorbed form for decode and for short chunks after
 * a long prefix (below about 380 tokens after 12288).  fp32 contexts, FP8
 * caches, and calls whose batch·max_pages·page_size exceeds
 * 2^18 rows, always get MLA_FORM_ABSORBED. */
int mla_prefill_form(const mla_ctx* ctx, int batch, int T, int max_pages);

mla_status mla_prefill(mla_ctx* ctx, const void* h, const int32_t* positions,
                       const void* q, void* cache, int num_pages,
                       const int32_t* block_table, int max_pages,
                       const int32_t* seq_lens, int batch, int T, int form,
                       void* out, void* workspace, size_t workspace_bytes,
                       void* stream);

/* One decode step through a stack of n_layers attention layers, each with
 * its own context (weights, d_cq > 0) and its own cache pool; the pools
 * share one page layout (block_table, num_pages).  The pages count the cache
 * over all l layers of the model (liang.world ch.2 §2: (d_c + d_h^R) x l
 * elements per token).  Layer j runs mla_layer_step on h_j (its new rows go
 * into caches[j], its queries come from h_j) and then
 *   h_{j+1} = h_j + u_j
 * (fp32 addition, rounded to the context dtype): the residual connection of
 * a transformer block around the attention output; the FFN sublayer and any
 * normalisation are outside this library.
 *   h          device, [batch*T, d_model], in/out: h_0 on entry, h_L on
 *              return (overwritten layer by layer).
 *   caches     host array of n_layers device pool pointers.
 *   u_scratch  device, [batch*T, d_model]: holds u of the last layer.
 *   workspace  as for mla_layer_step, shared by the layers (one at a time).
 * Other arguments as for mla_layer_step.  All contexts must share dtype,
 * d_model and device; a bad argument of any layer is reported before
 * anything is enqueued. */
mla_status mla_multi_layer_step(mla_ctx* const* ctxs, int n_layers, void* h,
                                const int32_t* positions, void* const* caches,
                                int num_pages, const int32_t* block_table,
                                int max_pages, const int32_t* seq_lens,
                                int batch, int T, void* u_scratch,
                                void* workspace, size_t workspace_bytes,
                                void* stream);

/* Decode without a workspace argument, for callers that cannot allocate
 * device memory when they decode (a fixed memory budget reserved up front,
 * an allocator that is not reachable from the issuing thread, a plugin that
 * is only handed its input and output buffers).  The pages have no
 * counterpart to this call: it is a packaging of mla_decode.
 *
 * Same arguments, layouts and results as mla_decode, minus the workspace:
 * the scratch is a 32 MiB array that the library reserves statically on
 * every GPU where its device code is loaded (held until the process exits).
 * The call itself allocates nothing.  Shapes whose
 * mla_decode_workspace_size exceeds 32 MiB return MLA_ERR_WORKSPACE before
 * anything is enqueued.  The first call on a device looks up the array's
 * device address (once per device) and keeps it for the life of the
 * process; make that first call before any stream capture.  A
 * cudaDeviceReset of that device invalidates the kept address: do not call
 * this entry point on a device after resetting it.  All calls share the one array, so calls that overlap on the GPU
 * (other streams, threads or contexts) race and give wrong results; nothing
 * in it needs to be cleared between calls. */
mla_status mla_decode_static_workspace(mla_ctx* ctx, const void* q,
                                       const void* cache, int num_pages,
                                       const int32_t* block_table,
                                       int max_pages, const int32_t* seq_lens,
                                       int batch, int T, void* out,
                                       void* stream);

/* Offsets (bytes from the workspace start) of two intermediates that
 * mla_decode leaves in the workspace, for diagnostics: the latent attention
 * output o_lat [batch*T, n_heads, d_latent] (sum_p a_p c_p) and the value
 * output o [batch*T, n_heads*d_v], both in the context dtype. */
mla_status mla_decode_workspace_offsets(const mla_ctx* ctx, int batch, int T,
                                        int max_pages, size_t* o_lat_offset,
                                        size_t* o_offset);

/* Synchronise `stream`, then read and clear the device status word.
 * Returns MLA_OK, MLA_ERR_TIMEOUT, MLA_ERR_DEVICE_INDEX or MLA_ERR_CUDA. */
mla_status mla_check_status(mla_ctx* ctx, void* stream);

/* Number of kernels this context has enqueued since creation. */
int64_t mla_launch_count(const mla_ctx* ctx);

/* Diagnostic: enqueue one kernel whose single bounded wait on an mbarrier
 * that nothing arrives on gives up after about `spin_limit` polls and
 * records MLA_ERR_TIMEOUT in the status word (the path every in-kernel wait
 * of this library takes when it gives up). */
mla_status mla_selftest_bounded_wait(mla_ctx* ctx, int spin_limit, void* stream);

/* Per-kernel timing for benchmarks.  mla_profile_enable(ctx, 1) starts a
 * fresh recording: from then on every call records a CUDA event on its
 * stream before each kernel it enqueues and one after the last (at most 64
 * events; later kernels are not recorded).  Calls captured into a CUDA
 * graph record event nodes, so each replay re-times the same kernels.
 * mla_profile_read waits for the last recorded event and writes, for at
 * most `max_kernels` recorded kernels, the kernel's name (a static string)
 * and its duration in milliseconds; it returns the number written or -1.
 * The events mark kernel boundaries, which keeps a kernel from overlapping
 * its predecessor: time whole steps with profiling off. */
mla_status mla_profile_enable(mla_ctx* ctx, int enable);
int mla_profile_read(mla_ctx* ctx, float* ms, const char** names, int max_kernels);

/* Static string naming a status code. */
const char* mla_status_string(mla_status s);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
