// Pieces shared by the attention kernels (attend_sv.cu, the split-KV
// latent attention, and prefill.cu, the per-head causal attention):
// segment iteration over a split's pages, pool-row lookup, stale-row
// zeroing, the softmax arithmetic on a 128-token score row, warp-uniform
// bounded waits and ring positions.
#pragma once

#include "layouts.cuh"
#include "tc_util.cuh"
#include "mla_internal.h"

namespace mla {
namespace att {

constexpr int kTile = 128;                                 // tokens per tile (2 pages)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 256;                            // S buffers at 256 and 384
constexpr float kRescale = 8.0f;                           // log2 units

struct AttArgs {
  const int* lens;
  const int* prefix;
  const int* first_split;
  const int* slot_base;
  const int* meta;
  const int32_t* bt;
  const uint8_t* qimg;
  const __nv_bfloat16* cache;
  float* part_o;
  float* part_lse;
  __nv_bfloat16* o_lat;   // final latent output of sequences held by one split
  int* status;
  int B, T, max_pages, num_pages;
  float scale_log2;
};


// Iterates the (sequence, page range) segments of split c, in order.
struct SegIter {
  const AttArgs* a;
  int c, t;
  long long g0, g1;
  int b;
  __device__ void init(const AttArgs* args, int c_, int t_) {
    a = args;
    c = c_;
    t = t_;
    const int G = a->meta[0];
    if (c >= G) { g0 = g1 = 0; b = a->B; return; }
    split_range(c, a->prefix[a->B], G, &g0, &g1);
    b = seq_of_page(a->prefix, a->B, g0);
  }
  // Next segment: sequence, first token, end token (exclusive, visible), slot.
  __device__ bool next(int* sb, int* p0, int* p1, int* slot) {
    if (b >= a->B || a->prefix[b] >= g1) return false;
    const long long pb = a->prefix[b];
    const long long lo = g0 > pb ? g0 : pb;
    const long long hi = g1 < a->prefix[b + 1] ? g1 : a->prefix[b + 1];
    const int vis = a->lens[b] - a->T + t + 1;
    *sb = b;
    *p0 = (int)(lo - pb) * kPage;
    *p1 = min((int)(hi - pb) * kPage, vis);
    *slot = a->slot_base[b] + (c - a->first_split[b]);
    ++b;
    return true;
  }
};

__device__ __forceinline__ int ntiles_of(int p0, int p1) {
  return p1 > p0 ? (p1 - p0 + kTile - 1) / kTile : 0;
}

// value slabs (32 tokens) of tile i that hold at least one visible token
__device__ __forceinline__ int nslabs_of(int tile_start, int p1) {
  const int v = p1 - tile_start;
  return v >= kTile ? 4 : (v + 31) / 32;
}

// Block-table entries of a tile's two pages.  The producer loads them one
// tile ahead of use and validates them only when used, so the global-load
// latency stays off its per-stage issue path.
struct TilePages {
  int pg0 = 0, pg1 = 0;
  bool two = false;   // the tile's second page starts before the visible end
  __device__ __forceinline__ void load(const AttArgs& a, int sb, int ts, int p1) {
    const int32_t* row = a.bt + (size_t)sb * a.max_pages + ts / kPage;
    pg0 = row[0];
    two = ts + kPage < p1;
    pg1 = two ? row[1] : 0;
  }
  // Pool row of page k (0 or 1); a missing second page gives oob_row (the
  // TMA fills it with zeros); a bad id is reported and replaced by page 0.
  __device__ __forceinline__ int row(const AttArgs& a, int k, int sb, int oob_row) const {
    if (k == 1 && !two) return oob_row;
    int pg = k ? pg1 : pg0;
    if (pg < 0 || pg >= a.num_pages) {
      report(a.status, MLA_ERR_DEVICE_INDEX, 4000000 + sb);
      pg = 0;
    }
    return pg * kPage;
  }
};

// Rows vis..31 of a value slab hold stale pool data past the visible end:
// zero them so that 0 * (Inf or NaN) cannot reach the accumulator.  The slab
// is NB SW128 blocks of 32 rows x 128 B (64 features each); the 32 lanes of
// a warp share the 16-byte chunks, and each makes its writes visible to the
// tensor cores.
template <int NB>
__device__ __forceinline__ void zero_stale_rows(uint8_t* slab, int vis, int lane) {
  for (int e = vis * NB * 8 + lane; e < 32 * NB * 8; e += 32) {
    const int r = e / (NB * 8), f = (e >> 3) % NB, ch = e & 7;
    *reinterpret_cast<uint4*>(slab + f * 4096 + (r >> 3) * 1024 + (r & 7) * 128 + ch * 16) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  tc::fence_async_smem();
}

// Row maximum of the raw scores of tokens 0..valid-1 (lo: 0..63, hi: 64..127).
template <bool kMask>
__device__ __forceinline__ float row_max(const uint32_t (&lo)[64], const uint32_t (&hi)[64],
                                         int valid) {
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    if (!kMask || j < valid) m0 = fmaxf(m0, __uint_as_float(lo[j]));
    if (!kMask || 64 + j < valid) m1 = fmaxf(m1, __uint_as_float(hi[j]));
  }
  return fmaxf(m0, m1);
}

// p = 2^(s * scale_log2 - m) for tokens below `valid` (0 beyond), rounded to
// bf16 and packed two per word: pk[j] holds tokens 2j (low) and 2j+1 (high).
// Returns the sum of the fp32 values.
template <bool kMask>
__device__ __forceinline__ float exp_pack(const uint32_t (&lo)[64], const uint32_t (&hi)[64],
                                          int valid, float scale_log2, float m,
                                          uint32_t (&pk)[64]) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const int t0 = 2 * j, t1 = 2 * j + 1;
    const float x0 = __uint_as_float(t0 < 64 ? lo[t0] : hi[t0 - 64]);
    const float x1 = __uint_as_float(t1 < 64 ? lo[t1] : hi[t1 - 64]);
    const float e0 = (!kMask || t0 < valid) ? tc::ex2_approx(fmaf(x0, scale_log2, -m)) : 0.f;
    const float e1 = (!kMask || t1 < valid) ? tc::ex2_approx(fmaf(x1, scale_log2, -m)) : 0.f;
    s0 += e0;
    s1 += e1;
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(e0, e1);
    pk[j] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  return s0 + s1;
}

// Bounded wait by a whole warp; the outcome is made warp-uniform.  The
// common case (phase already complete) costs one probe and one vote.
// kCluster: the barrier also receives arrivals from the other CTA of a pair.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* status, int where) {
  if (kCluster) return __all_sync(0xffffffffu, mbar_wait_cluster(bar, parity, status, where));
  if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status, where));
}

// One thread's bounded wait, local or cluster-fed barrier.
template <bool kCluster>
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, int* status, int where) {
  return kCluster ? mbar_wait_cluster(bar, parity, status, where)
                  : mbar_wait(bar, parity, status, where);
}

// Position in a stage ring of R slots: slot, phase bit of this pass over the
// ring, and the number of stages passed so far.
template <int R>
struct RingPos {
  int s = 0, n = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next() {
    ++n;
    if (++s == R) {
      s = 0;
      ph ^= 1u;
    }
  }
};

}  // namespace att
}  // namespace mla
