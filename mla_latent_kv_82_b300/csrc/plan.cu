// Split-KV work plan and workspace layout.
//
// Long caches are split across SMs (flash-decoding style) and merged with a
// log-sum-exp combine.  The plan is built on the device from seq_lens so the
// host never waits for it:
//   * pages(b)      = ceil(len_b / page_size), len_b validated and clamped;
//   * prefix[b]     = pages of sequences 0..b-1  (prefix[B] = P, all pages);
//   * G_eff = min(G, max(1, P / kMinPagesPerSplit)) splits are used (none is
//     empty, and short caches are not cut so thin that merging the partial
//     results costs more than the attention itself); split c < G_eff
//     owns global pages [floor(cP/G_eff), floor((c+1)P/G_eff));
//   * first_split[b] = split holding page prefix[b]; the splits touching
//     sequence b are first_split[b] .. split(prefix[b+1]-1);
//   * slot_base[b]   = partial-result slots of sequences 0..b-1; split c's
//     piece of sequence b lands in slot slot_base[b] + c - first_split[b].
// Every split does the same number of pages (+-1), whatever the length mix.
#include "plan_device.cuh"

namespace mla {

namespace {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t* __restrict__ seq_lens, int B, int T, int page, int max_pages,
            int max_position, int G_max, int* lens, int* prefix, int* first_split,
            int* slot_base, int* meta, int* status) {
  __shared__ int tmp[33];
  // seq_lens may have been written by the kernel before us
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  PlanArgs pa{seq_lens, B, T, page, max_pages, max_position, G_max, lens, prefix, first_split,
              slot_base, meta, status};
  build_plan<kPlanThreads>(threadIdx.x, [] { __syncthreads(); }, tmp, pa);
}

__global__ void selftest_wait_kernel(int spin_limit, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) mbar_init(&bar, 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing ever arrives on `bar`: the bounded wait must give up.
    const bool done = mbar_wait(&bar, 0, status, 424242, spin_limit, 200000000ull);
    (void)done;
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_inval(&bar);
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

// KV splits: enough to fill the SMs with the attention kernel's CTAs, never
// more than there are pages.
static int choose_splits(const mla_ctx* ctx, int B, int T, int max_pages) {
  const long long pages_bound = (long long)B * max_pages;
  int G;
  if (kv_fp8(ctx)) {
    // two CTAs (latent halves) per (split, query token), one per SM
    G = ctx->num_sms / (2 * T);
  } else if (ctx->cfg.dtype == MLA_BF16) {
    // one cluster of two CTAs per (split, query token) for odd T, of four
    // per (split, token pair) for even T, one CTA per SM, all resident at once
    G = ctx->num_sms / (2 * T);
    const int fit = T % 2 ? ctx->sv_clusters[0] / T : ctx->sv_clusters[1] / (T / 2);
    if (fit >= 1 && fit < G) G = fit;
  } else {
    const int groups = (ctx->cfg.n_heads + 7) / 8;
    G = (2 * ctx->num_sms + T * groups - 1) / (T * groups);
  }
  if (G < 1) G = 1;
  if (G > pages_bound) G = (int)pages_bound;
  return G;
}

WsLayout workspace_layout(const mla_ctx* ctx, int B, int T, int max_pages) {
  const mla_config& c = ctx->cfg;
  const size_t es = c.dtype == MLA_BF16 ? 2 : 4;
  const size_t M = (size_t)B * T;
  const size_t R = (size_t)c.d_latent + c.d_rope;
  WsLayout L{};
  L.G = choose_splits(ctx, B, T, max_pages);
  L.n_slots = L.G + B;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align256(off + bytes); return o; };
  L.lens = take(sizeof(int) * B);
  L.page_prefix = take(sizeof(int) * (B + 1));
  L.first_split = take(sizeof(int) * B);
  L.slot_base = take(sizeof(int) * (B + 1));
  L.meta = take(sizeof(int) * 4);
  L.qfull = take(es * M * c.n_heads * R);
  L.part_o = take(sizeof(float) * L.n_slots * T * c.n_heads * c.d_latent);
  L.part_lse = take(sizeof(float) * L.n_slots * T * c.n_heads);
  L.o_lat = take(es * M * c.n_heads * c.d_latent);
  L.o = take(es * M * c.n_heads * c.d_v);
  L.wg_part = take(c.dtype == MLA_BF16 ? bf16_wg_partial_bytes(ctx, (int)M) : 0);
  if (c.d_cq > 0) {
    L.c_q = take(es * M * c.d_cq);
    L.q_in = take(es * M * c.n_heads * (c.d_nope + c.d_rope));
  }
  if (kv_fp8(ctx)) L.q8 = take((size_t)kQ8Bytes * M);
  L.total = off;
  return L;
}

void launch_plan(const mla_ctx* ctx, const WsLayout& L, char* ws, const int32_t* seq_lens,
                 int B, int T, int max_pages, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, plan_kernel, seq_lens, B, T, ctx->cfg.page_size, max_pages,
                     ctx->cfg.max_position, L.G, reinterpret_cast<int*>(ws + L.lens),
                     reinterpret_cast<int*>(ws + L.page_prefix),
                     reinterpret_cast<int*>(ws + L.first_split),
                     reinterpret_cast<int*>(ws + L.slot_base), reinterpret_cast<int*>(ws + L.meta),
                     ctx->status);
}

void launch_selftest_wait(const mla_ctx* ctx, int spin_limit, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(spin_limit, ctx->status);
}

}  // namespace mla
