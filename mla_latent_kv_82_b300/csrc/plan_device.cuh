// Split-KV work plan built on the device by a group of threads.
//
// Long caches are split across SMs (flash-decoding style) and merged with a
// log-sum-exp combine.  The plan is built on the device from seq_lens so the
// host never waits for it:
//   * len_b validated (T <= len_b <= min(max_pages*page, max_position)) and
//     clamped; pages(b) = ceil(len_b / page);
//   * prefix[b]     = pages of sequences 0..b-1  (prefix[B] = P, all pages);
//   * G_eff = min(G, max(1, P / kMinPagesPerSplit)) splits are used (none is
//     empty, and short caches are not cut so thin that merging the partial
//     results costs more than the attention itself); split c < G_eff owns
//     global pages [floor(cP/G_eff), floor((c+1)P/G_eff));
//   * first_split[b] = split holding page prefix[b]; the splits touching
//     sequence b are first_split[b] .. split(prefix[b+1]-1);
//   * slot_base[b]   = partial-result slots of sequences 0..b-1; split c's
//     piece of sequence b lands in slot slot_base[b] + c - first_split[b].
// Every split does the same number of pages (+-1), whatever the length mix.
#pragma once

#include "device_util.cuh"

namespace mla {

constexpr int kMinPagesPerSplit = 2;

struct PlanArgs {
  const int32_t* seq_lens;
  int B, T, page, max_pages, max_position, G_max;
  int* lens;
  int* prefix;
  int* first_split;
  int* slot_base;
  int* meta;
  int* status;
};

// The validated length of sequence b (the clamp the plan applies).
__device__ __forceinline__ int plan_len(const int32_t* seq_lens, int b, int T, int page,
                                        int max_pages, int max_position) {
  int len = seq_lens[b];
  const int cap = min(max_pages * page, max_position);
  return len < T ? T : (len > cap ? cap : len);
}

__device__ __forceinline__ long long split_of_page(long long g, long long P, int G) {
  return ((g + 1) * G - 1) / P;
}

// Exclusive scan of one int per thread over NTHREADS threads (tid 0..N-1);
// `sync` synchronises exactly those threads; tmp holds 33 ints.
template <int NTHREADS, class Sync>
__device__ int group_exclusive_scan(int tid, int v, int* out, int* tmp, Sync sync) {
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = NTHREADS / 32;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  sync();
  if (warp == 0) {
    int s = lane < kWarps ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    tmp[lane] = s;  // inclusive warp totals
  }
  sync();
  const int total = tmp[kWarps - 1];
  *out = x - v + (warp > 0 ? tmp[warp - 1] : 0);
  sync();
  return total;
}

// Builds lens, prefix, first_split, slot_base and meta = {G_eff, P}.
template <int NTHREADS, class Sync>
__device__ void build_plan(int tid, Sync sync, int* tmp, const PlanArgs& a) {
  int carry = 0;
  // pass 1: validated lengths and the page prefix
  for (int base = 0; base < a.B; base += NTHREADS) {
    const int b = base + tid;
    int pages = 0;
    if (b < a.B) {
      const int raw = a.seq_lens[b];
      const int len = plan_len(a.seq_lens, b, a.T, a.page, a.max_pages, a.max_position);
      if (len != raw) report(a.status, MLA_ERR_DEVICE_INDEX, 1000000 + b);
      a.lens[b] = len;
      pages = (len + a.page - 1) / a.page;
    }
    int ex;
    const int tot = group_exclusive_scan<NTHREADS>(tid, pages, &ex, tmp, sync);
    if (b < a.B) a.prefix[b] = carry + ex;
    carry += tot;
  }
  const long long P = carry;
  long long g_want = P / kMinPagesPerSplit;
  if (g_want < 1) g_want = 1;
  const int G = g_want < a.G_max ? (int)g_want : a.G_max;
  if (tid == 0) {
    a.prefix[a.B] = carry;
    a.meta[0] = G;
    a.meta[1] = carry;
  }
  __threadfence_block();
  sync();
  // pass 2: splits per sequence and their slot bases
  carry = 0;
  for (int base = 0; base < a.B; base += NTHREADS) {
    const int b = base + tid;
    int ns = 0;
    if (b < a.B) {
      const long long c0 = split_of_page(a.prefix[b], P, G);
      const long long c1 = split_of_page(a.prefix[b + 1] - 1, P, G);
      a.first_split[b] = (int)c0;
      ns = (int)(c1 - c0 + 1);
    }
    int ex;
    const int tot = group_exclusive_scan<NTHREADS>(tid, ns, &ex, tmp, sync);
    if (b < a.B) a.slot_base[b] = carry + ex;
    carry += tot;
  }
  if (tid == 0) a.slot_base[a.B] = carry;
}

}  // namespace mla
