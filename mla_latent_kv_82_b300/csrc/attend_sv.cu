// Split-KV flash-decoding over the bf16 latent cache, with the score and the
// value halves of attention on different CTAs of a cluster.
//
// Absorbed MLA attention (page "DeepSeek-V2：在“大力出奇迹”的AI军备竞赛中，
// 四两拨千斤", liang.world, 第二章 §2 absorption and §3 decoupled RoPE): with
// the query image Q = [W^UK_i^T q^C_i ; RoPE(q^R_i)] (128 heads x 576) and the
// cached rows C = [c^KV ; k^R] (tokens x 576),
//     s = Q C^T * scale,  a = softmax(s),  o_lat = a C[:, :512].
// Heads are the M side of both MMAs, 128 cache tokens the N side of the
// score MMA.  The output O (128 heads x 512 fp32) fills a whole tensor memory
// (512 columns), so one CTA cannot hold O and S together.  Here each cache
// tile's S is computed once, by a score CTA, and its bf16 P is sent over
// distributed shared memory to a value CTA that owns the whole O:
//
//   score CTA   TMEM: q~ (the 512 latent features of Q, bf16 packed two per
//               column, 256 columns) and two S buffers (2 x 128 columns);
//               shared memory: the RoPE block of Q (16 KB), a staging
//               buffer for P and an 11-stage ring of score blocks [tokens x
//               64 features].  S = q~ C_lat^T (A from TMEM) + RoPE(q^R)
//               k^R^T (A from shared memory); softmax from registers; P
//               (bf16) and the row statistics staged in local shared memory
//               and pushed by one bulk copy into the value CTA's landing
//               buffer (its bytes complete the landing barrier there).
//   value CTA   TMEM: O (512 columns); shared memory: two landing buffers
//               (P [128 heads x 128 tokens] + rescale factor + running row
//               sum) and a 9-stage ring of value slabs [32 tokens x 256
//               columns]; O += P V (A = P from shared memory); lazy rescale
//               of O by the correction warps; O / l at the end of a segment.
//
// Odd T: a cluster of two CTAs (rank 0 score, rank 1 value) per (KV split,
// query token).  Even T: query tokens 2j and 2j+1 see the same cache tiles,
// so a cluster of four runs them together: ranks 0-1 are a cta_group::2 pair
// computing S for both tokens with M = 256 MMAs (each CTA loads one of the
// tile's two pages), ranks 2-3 a pair accumulating both tokens' O with M =
// 256 MMAs (each CTA loads half of the value columns).
//
// Warps (224 threads): 0 TMA producer; 1 MMA issuer (pair leader) and TMEM
// allocation; 2-5 softmax (score) or correction and epilogue (value), thread
// = head; 6 relay in the odd value CTA of a pair (zeroes the stale rows of a
// value slab reaching past the visible end before its bytes count on the
// leader's barrier).  Every wait is bounded; a failure sets the abort flag
// of every CTA of the cluster, and each CTA drains its own copies and MMAs
// before the cluster ends.
#include "attend_common.cuh"
#include "tmap.h"
#include "launch_util.h"

namespace mla {
namespace {

using namespace att;

constexpr uint32_t kStage = 16384;
constexpr int kVRing = 9;                                   // value ring stages
// landing buffer: P [2 token blocks][128 heads][128 B] (SW128, K-major),
// then the rescale factor f[128] and the running row sum l[128]
constexpr uint32_t kLandP = 32768;
constexpr uint32_t kLandBytes = kLandP + 512 + 512;         // 33792
constexpr uint32_t kOffQr = 0;                              // score: RoPE block of Q
constexpr uint32_t kOffStage = 16384;                       // score: P staging buffers
constexpr uint32_t kOffLand = 0;                            // value: landing buffers
constexpr uint32_t kOffVRing = 2 * kLandBytes;              // 67584

// The score side's shared memory holds one staging buffer for P and an
// 11-stage ring for a single query token (9 stages per tile), two staging
// buffers and an 8-stage ring for a token pair (5 stages per tile).  With one
// buffer a tile's P waits for the previous tile's copy to land; measured,
// that wait bounds the pair kernel, while the single-token kernel is bound
// by its score-block loads and gains from the deeper ring.
template <bool kPair> struct SvLayout {
  static constexpr int kStaging = kPair ? 2 : 1;
  static constexpr int kSRing = kPair ? 8 : 11;
  static constexpr uint32_t kOffSRing = kOffStage + kStaging * kLandBytes;
  static constexpr uint32_t kOffBar = kOffSRing + kSRing * kStage;   // same in every CTA
  static constexpr uint32_t kSmem = kOffBar + 512 + 1024;
  static_assert(kOffVRing + kVRing * kStage <= kOffBar, "value ring overlaps the barriers");
  static_assert(kOffSRing % 1024 == 0, "SW128 operands need 1 KB alignment");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};
static_assert(kOffVRing % 1024 == 0 && kLandBytes % 1024 == 0, "SW128 operands need 1 KB alignment");

// Barrier slots (8 bytes each) at kOffBar, at the same offset in every CTA of
// a cluster so that multicast commits and remote arrivals can name them.
enum : int {
  kBFull = 0,      // [16] ring stage filled (pair: both CTAs' bytes on the leader's)
  kBEmpty = 16,    // [16] ring stage consumed by the MMAs
  kBSFull = 32,    // [2] score: S of tiles of that parity done
  kBSFree = 34,    // [2] score: S of that parity read by the softmax warps
  kBPvd = 36,      // [2] PV of tiles of that parity done (value: O may be read /
                   //     rescaled; score: that landing buffer may be rewritten)
  kBLand = 38,     // [2] value: P of that parity landed (bulk copy from the score CTA)
  kBOok = 40,      // [2] value: O corrected for that tile (pair leader: 8 warps)
  kBQReady = 42,   // score: q~ stored in TMEM and the RoPE block landed
  kBQr = 43,       // score: RoPE block of Q landed (local copy)
  kBQEmpty = 44,   // score: S MMAs of the segment done (q~ and RoPE block free)
  kBDrained = 46,  // this CTA's MMAs all complete
  kBZb = 47,       // odd value CTA: partial value slab landed locally
  kBZDone = 48,    // odd value CTA: relay finished a partial slab
  kBStgFree = 49,  // score: the staged P of the last tile has landed (value CTA)
  kBSlot = 50      // TMEM base address (u32) and abort flag (u32)
};

constexpr uint32_t kColQ = 0;     // score: q~ (256 columns)
constexpr uint32_t kColS = 256;   // score: S buffers at 256 and 384

template <bool kPair>
__device__ __forceinline__ bool cwait(uint64_t* bar, uint32_t parity, int* status, int where) {
  return warp_wait<kPair>(bar, parity, status, where);
}

// The four K steps (4 x 16 features) of one 64-feature score block: A from
// TMEM at aq (8 columns per step), B the block's descriptor (32 bytes per
// step); the first step accumulates if acc0.
template <bool kPair>
__device__ __forceinline__ void score_mma4(uint32_t d, uint32_t aq, uint64_t b, uint32_t idesc,
                                           uint32_t acc0) {
  if (kPair) {
    tc::mma2_ts(d, aq, b, idesc, acc0);
    tc::mma2_ts(d, aq + 8, b + 2, idesc, 1u);
    tc::mma2_ts(d, aq + 16, b + 4, idesc, 1u);
    tc::mma2_ts(d, aq + 24, b + 6, idesc, 1u);
  } else {
    tc::mma_ts(d, aq, b, idesc, acc0);
    tc::mma_ts(d, aq + 8, b + 2, idesc, 1u);
    tc::mma_ts(d, aq + 16, b + 4, idesc, 1u);
    tc::mma_ts(d, aq + 24, b + 6, idesc, 1u);
  }
}

// The same for the RoPE block with A (the rotated q^R) in shared memory.
template <bool kPair>
__device__ __forceinline__ void score_mma4_ss(uint32_t d, uint64_t a, uint64_t b,
                                              uint32_t idesc) {
  if (kPair) {
    tc::mma2_ss(d, a, b, idesc, 1u);
    tc::mma2_ss(d, a + 2, b + 2, idesc, 1u);
    tc::mma2_ss(d, a + 4, b + 4, idesc, 1u);
    tc::mma2_ss(d, a + 6, b + 6, idesc, 1u);
  } else {
    tc::mma_ss(d, a, b, idesc, 1u);
    tc::mma_ss(d, a + 2, b + 2, idesc, 1u);
    tc::mma_ss(d, a + 4, b + 4, idesc, 1u);
    tc::mma_ss(d, a + 6, b + 6, idesc, 1u);
  }
}

template <bool kPair>
__global__ void __launch_bounds__(224, 1)
attend_sv_kernel(const __grid_constant__ CUtensorMap tmS,    // pool, box {64, 64}
                 const __grid_constant__ CUtensorMap tmS2,   // pool blocks, box {64, 64, 2}
                 const __grid_constant__ CUtensorMap tmV,    // pool blocks, box {64, 32, kPair ? 2 : 4}
                 const AttArgs a) {
  using Lay = SvLayout<kPair>;
  constexpr int kSRing = Lay::kSRing;
  constexpr uint32_t kOffSRing = Lay::kOffSRing;
  constexpr uint32_t kOffBar = Lay::kOffBar;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + kBSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* sm_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);   // softmax warps

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = tc::cluster_rank();
  constexpr uint32_t kCluster = kPair ? 4 : 2;
  const bool score = kPair ? rank < 2 : rank == 0;
  const bool leader = kPair ? (rank & 1u) == 0 : true;      // issues its pair's MMAs
  const uint32_t lead_rank = kPair ? (rank & ~1u) : rank;
  const uint32_t pair_mask = kPair ? (3u << (rank & 2u)) : (1u << rank);
  int c, t;
  if (kPair) {
    c = blockIdx.y;
    t = 2 * blockIdx.z + (int)(rank & 1u);
  } else {
    c = blockIdx.x >> 1;
    t = blockIdx.y;
  }
  const int t_iter = kPair ? (t | 1) : t;   // a pair iterates the odd token's range

  tc::grid_dep_launch();
  tc::grid_dep_wait();   // plan, query image and cache come from earlier kernels
  if (c >= a.meta[0]) return;   // every CTA of the cluster has the same split

  if (threadIdx.x == 0) {
    const uint32_t pw = kPair ? 8 : 4;   // warps arriving on a pair leader's barrier
    for (int i = 0; i < 16; ++i) {
      mbar_init(&bar[kBFull + i], 1);
      mbar_init(&bar[kBEmpty + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[kBSFull + i], 1);
      mbar_init(&bar[kBSFree + i], pw);
      mbar_init(&bar[kBPvd + i], 1);
      mbar_init(&bar[kBLand + i], 1);
      mbar_init(&bar[kBOok + i], pw);
    }
    mbar_init(&bar[kBQReady], pw);
    mbar_init(&bar[kBQr], 1);
    mbar_init(&bar[kBQEmpty], 1);
    mbar_init(&bar[kBDrained], 1);
    mbar_init(&bar[kBZb], 1);
    mbar_init(&bar[kBZDone], 1);
    mbar_init(&bar[kBStgFree], 1);
    *abort_flag = 0;
    *sm_fail = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    if (kPair) {
      tc::tmem_alloc2(smem_u32(tmem_slot), kTmemCols);
      tc::tmem_relinquish2();
    } else {
      tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tc::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmS);
    tc::prefetch_tmap(&tmS2);
    tc::prefetch_tmap(&tmV);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();   // every CTA's barriers and TMEM ready
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // cluster address of barrier slot i in CTA r
  const uint32_t bar_local = smem_u32(bar);
  auto cbar = [&](int i, uint32_t r) { return tc::mapa_shared(bar_local + 8u * i, r); };
  auto set_abort = [&] {
    *abort_flag = 1;
    for (uint32_t r = 0; r < kCluster; ++r)
      if (r != rank) tc::st_cluster_u32(tc::mapa_shared(smem_u32((const void*)abort_flag), r), 1u);
  };
  auto aborted = [&] { return __any_sync(0xffffffffu, *abort_flag != 0); };
  const int oob_row = a.num_pages * kPage + kPage;   // TMA zero-fills rows out of range
  int issued = 0;     // producer: ring stages issued
  int qr_issued = 0;  // producer: RoPE blocks issued

  if (score && warp == 0) {
    // ------------------------------------------------------ score producer
    // Per segment: the RoPE block of this CTA's query image (after the
    // previous segment's score MMAs), then the score blocks of every tile:
    // single CTA, 9 stages of [128 tokens x 64 features] (one box per
    // page); pair, 5 stages of this CTA's page, two blocks per stage (the
    // last one block), whose bytes count on the leader's barrier.
    const bool el = tc::elect_one();
    RingPos<kSRing> rp;
    SegIter it;
    it.init(&a, c, t_iter);
    int sb, p0, p1, slot, k = 0;
    bool ok = true;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      if (k > 0 && !cwait<kPair>(&bar[kBQEmpty], (k - 1) & 1, a.status, 71)) { ok = false; break; }
      if (aborted()) { ok = false; break; }
      ++qr_issued;
      if (el) {
        tc::mbar_arrive_expect_tx(smem_u32(&bar[kBQr]), 16384);
        tc::bulk_load(smem_u32(smem + kOffQr),
                      a.qimg + ((size_t)sb * a.T + t) * kQImgBytes + 8 * 16384, 16384,
                      smem_u32(&bar[kBQr]));
      }
      TilePages cur;
      cur.load(a, sb, p0, p1);
      constexpr int kNst = kPair ? 5 : 9;
      for (int i = 0; ok && i < n; ++i) {
        TilePages nxt;
        if (i + 1 < n) nxt.load(a, sb, p0 + (i + 1) * kTile, p1);   // used next tile
        int y0 = 0, y1 = 0;
        if (kPair) {
          y0 = cur.row(a, (int)(rank & 1u), sb, oob_row);
        } else {
          y0 = cur.row(a, 0, sb, oob_row);
          y1 = cur.row(a, 1, sb, oob_row);
        }
        for (int j = 0; j < kNst; ++j, rp.next()) {
          const int s = rp.s;
          if (rp.n >= kSRing &&
              !cwait<kPair>(&bar[kBEmpty + s], rp.ph ^ 1u, a.status, 72)) {
            ok = false;
            break;
          }
          if (aborted()) { ok = false; break; }
          issued = rp.n + 1;
          if (el) {
            const uint32_t dst = smem_u32(smem + kOffSRing + s * kStage);
            const uint32_t fb = smem_u32(&bar[kBFull + s]);
            if (!kPair) {
              tc::mbar_arrive_expect_tx(fb, kStage);
              tc::tma_load_2d(dst, &tmS, j * 64, y0, fb);
              tc::tma_load_2d(dst + 8192, &tmS, j * 64, y1, fb);
            } else {
              const int cnt = j == 4 ? 1 : 2;
              const uint32_t lb = cbar(kBFull + s, lead_rank);
              if (leader) tc::mbar_arrive_expect_tx(fb, 2u * cnt * 8192u);
              if (cnt == 2) {
                if (leader) tc::tma_load_3d(dst, &tmS2, 0, y0, 2 * j, fb);
                else tc::tma_load_3d_pair(dst, &tmS2, 0, y0, 2 * j, lb);
              } else {
                if (leader) tc::tma_load_2d(dst, &tmS, 8 * 64, y0, fb);
                else tc::tma_load_2d_pair(dst, &tmS, 8 * 64, y0, lb);
              }
            }
          }
        }
        cur = nxt;
      }
      ++k;
    }
    if (!ok) set_abort();
  } else if (score && warp == 1 && leader) {
    // ------------------------------------------------------ score MMA issuer
    // S(g) (128 or 256 rows x 128 tokens) into S buffer g & 1, once the
    // softmax warps have read S(g-2) out of it.  Feature blocks 0-7: A = q~
    // from TMEM (8 columns per K step of 16); block 8: A = the RoPE block of
    // Q from shared memory.
    const bool el = tc::elect_one();
    constexpr uint32_t idS = tc::idesc_bf16(kPair ? 256 : 128, kTile, false, false);
    const uint64_t dQr = tc::sdesc(smem_u32(smem + kOffQr), 16, 1024);
    const uint64_t dR = tc::sdesc(smem_u32(smem + kOffSRing), 16, 1024);
    constexpr int kNst = kPair ? 5 : 9;
    RingPos<kSRing> rp;
    int g = 0, k = 0;
    bool ok = true;
    SegIter it;
    it.init(&a, c, t_iter);
    int sb, p0, p1, slot;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      if (!cwait<kPair>(&bar[kBQReady], k & 1, a.status, 73)) { ok = false; break; }
      tc::fence_after_sync();
      for (int i = 0; ok && i < n; ++i) {
        const int gs = g + i;
        if (gs >= 2 &&
            !cwait<kPair>(&bar[kBSFree + (gs & 1)], ((gs - 2) >> 1) & 1, a.status, 74)) {
          ok = false;
          break;
        }
        if (aborted()) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t dcol = tmem + kColS + (gs & 1) * kTile;
        for (int j = 0; j < kNst; ++j, rp.next()) {
          const int s = rp.s;
          if (!cwait<kPair>(&bar[kBFull + s], rp.ph, a.status, 75)) { ok = false; break; }
          tc::fence_after_sync();
          if (el) {
            // Each stage's MMAs are issued as straight-line code: a branch
            // between two tcgen05.mma instructions was measured to slow their
            // issue from 64 to about 95 cycles each (M = 128, N = 128).
            const uint64_t dRs = dR + ((s * kStage) >> 4);
            if (j < kNst - 1) {
              // latent blocks: A = q~ from TMEM, 8 columns per K step of 16
              const int b0 = kPair ? 2 * j : j;
              const uint32_t aq = tmem + kColQ + b0 * 32;
              score_mma4<kPair>(dcol, aq, dRs, idS, j > 0 ? 1u : 0u);
              if (kPair) score_mma4<kPair>(dcol, aq + 32, dRs + (8192 >> 4), idS, 1u);
            } else {
              // RoPE block: A from shared memory
              score_mma4_ss<kPair>(dcol, dQr, dRs, idS);
            }
            if (kPair) tc::mma2_commit_mc(smem_u32(&bar[kBEmpty + s]), (uint16_t)pair_mask);
            else tc::mma_commit(smem_u32(&bar[kBEmpty + s]));
          }
        }
        if (!ok) break;
        if (el) {
          if (kPair) {
            tc::mma2_commit_mc(smem_u32(&bar[kBSFull + (gs & 1)]), (uint16_t)pair_mask);
            if (i == n - 1) tc::mma2_commit_mc(smem_u32(&bar[kBQEmpty]), (uint16_t)pair_mask);
          } else {
            tc::mma_commit(smem_u32(&bar[kBSFull + (gs & 1)]));
            if (i == n - 1) tc::mma_commit(smem_u32(&bar[kBQEmpty]));
          }
        }
      }
      g += n;
      ++k;
    }
    if (!ok) set_abort();
    if (el) {
      if (kPair) tc::mma2_commit_mc(smem_u32(&bar[kBDrained]), (uint16_t)pair_mask);
      else tc::mma_commit(smem_u32(&bar[kBDrained]));
    }
  } else if (score && warp >= 2 && warp < 6) {
    // ------------------------------------------------------ softmax warps
    // Thread = head.  Per segment: q~ of this CTA's token into TMEM (after
    // the previous segment's score MMAs), then per tile: S row into
    // registers, S buffer released, row maximum, P = 2^(s * scale - m) in
    // the log2 domain with a lazy rescale (m moves only when the maximum
    // grows by more than 2^kRescale, so P <= 256), P as bf16 into the value
    // CTA's landing buffer with the rescale factor f and the running sum l.
    // The four warps meet at a named barrier twice per tile (the staging
    // buffer is shared), so every decision to stop is taken by all of them
    // together: a warp whose wait fails raises sm_fail and goes on to the
    // next barrier; right after it every thread reads sm_fail and all stop.
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const uint32_t vrank = rank + (kPair ? 2u : 1u);   // the value CTA of this token
    const uint32_t land0 = tc::mapa_shared(smem_u32(smem + kOffLand), vrank);
    const uint32_t prow_off = (uint32_t)((row >> 3) * 1024 + (row & 7) * 128);
    SegIter it;
    it.init(&a, c, t_iter);
    int sb, p0, p1, slot, g = 0, k = 0;
    bool ok = true, fail = false;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      const size_t prow = ((size_t)slot * a.T + t) * kHeads + row;
      if (n == 0) {
        a.part_lse[prow] = -INFINITY;   // an empty partial: weight 0 in the combine
        continue;
      }
      // ---- q~ of this segment's token: image blocks 0-7, row `row`
      if (!fail && k > 0) fail = !cwait<kPair>(&bar[kBQEmpty], (k - 1) & 1, a.status, 76);
      if (!fail) {
        tc::fence_after_sync();
        // chunk-major image: 32-byte chunk J of this head at J * 4096 +
        // row * 32, so the warp's 32 heads read 1 KB contiguous per load
        const uint8_t* img = a.qimg + ((size_t)sb * a.T + t) * kQImgBytes + row * 32;
        // two rounds of four feature blocks (four chunks each), 16 loads of
        // 32 bytes in flight per thread
#pragma unroll 1
        for (int f0 = 0; f0 < 8; f0 += 4) {
          uint32_t v[4][32];
#pragma unroll
          for (int fb = 0; fb < 4; ++fb)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              ld_nc_v8(img + ((f0 + fb) * 4 + j) * 4096, &v[fb][8 * j]);
#pragma unroll
          for (int fb = 0; fb < 4; ++fb) tc::tmem_st32(trow + kColQ + (f0 + fb) * 32, v[fb]);
        }
        tc::fence_before_sync();
        // the RoPE block lands in parallel; q~ and it are ready together
        fail = !warp_wait<false>(&bar[kBQr], k & 1, a.status, 77);
        __syncwarp();
        if (!fail && lane == 0) {
          if (kPair) tc::mbar_arrive_cluster_relaxed(cbar(kBQReady, lead_rank));
          else tc::mbar_arrive(smem_u32(&bar[kBQReady]));
        }
      }
      ++k;
      // ---- tiles
      const int p1_own = min(p1, a.lens[sb] - a.T + t + 1);   // this token's causal end
      float m_used = -INFINITY, l = 0.f;
      for (int i = 0; i < n; ++i, ++g) {
        if (!fail) fail = !cwait<kPair>(&bar[kBSFull + (g & 1)], (g >> 1) & 1, a.status, 78);
        uint32_t pk[64];
        float f = 1.f;
        if (!fail) {
          tc::fence_after_sync();
          uint32_t lo[64], hi[64];
          const uint32_t scol = trow + kColS + (g & 1) * kTile;
          tc::tmem_ld64(scol, lo);
          tc::tmem_ld64(scol + 64, hi);
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            if (kPair) tc::mbar_arrive_cluster_relaxed(cbar(kBSFree + (g & 1), lead_rank));
            else tc::mbar_arrive(smem_u32(&bar[kBSFree + (g & 1)]));
          }
          const int valid = max(0, min(kTile, p1_own - (p0 + i * kTile)));
          const float mx = (valid == kTile ? row_max<false>(lo, hi, valid)
                                           : row_max<true>(lo, hi, valid)) * a.scale_log2;
          if (i == 0) {
            m_used = mx;
          } else if (mx > m_used + kRescale) {
            f = exp2f(m_used - mx);
            m_used = mx;
            l *= f;
          }
          const float psum = valid == kTile
                                 ? exp_pack<false>(lo, hi, valid, a.scale_log2, m_used, pk)
                                 : exp_pack<true>(lo, hi, valid, a.scale_log2, m_used, pk);
          l += psum;
          // landing buffer g & 1 is free once PV(g - 2) has read it, and so
          // is staging buffer g & 1 of a pair (its copy landed before that);
          // the single staging buffer once the copy of P(g - 1) has landed
          if (warp == 2) {
            bool w = true;
            if (!kPair && g >= 1)
              w = bar_wait<true>(&bar[kBStgFree], (g - 1) & 1, a.status, 80);
            if (w && g >= 2)
              w = bar_wait<true>(&bar[kBPvd + (g & 1)], ((g - 2) >> 1) & 1, a.status, 79);
            fail = !__all_sync(0xffffffffu, w);
          }
        }
        if (fail) *sm_fail = 1;
        if (warp == 2 && lane == 0 && *abort_flag) *sm_fail = 1;
        tc::named_sync(1, 128);
        if (*sm_fail) { ok = false; break; }   // the same value for every thread
        uint8_t* stg = smem + kOffStage + (kPair ? (g & 1) * kLandBytes : 0u);
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const uint32_t off = (uint32_t)((ch >> 3) * 16384) + prow_off +
                               (uint32_t)(((ch & 7) ^ (row & 7)) << 4);
          *reinterpret_cast<uint4*>(stg + off) =
              make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        }
        reinterpret_cast<float*>(stg + kLandP)[row] = f;
        reinterpret_cast<float*>(stg + kLandP + 512)[row] = l;
        tc::fence_async_smem();   // the staged P is read by the bulk copy (async proxy)
        tc::named_sync(1, 128);
        if (warp == 2 && lane == 0) {
          const uint32_t lb = cbar(kBLand + (g & 1), vrank);
          tc::mbar_arrive_expect_tx_cluster(lb, kLandBytes);
          tc::bulk_s2c(land0 + (g & 1) * kLandBytes, smem_u32(stg), kLandBytes, lb);
        }
      }
      if (!ok) break;
      a.part_lse[prow] = l > 0.f ? m_used + log2f(l) : -INFINITY;
    }
    if (!ok || fail) set_abort();
  } else if (!score && warp == 0) {
    // ------------------------------------------------------ value producer
    // Value slabs of every tile in order: single CTA, [32 tokens x 256
    // columns] per stage, both halves of each slab; pair, [32 tokens x
    // (2 + 2) blocks of 64 columns] per stage (this CTA's half of both
    // 256-column groups), whose bytes count on the leader's barrier, except
    // a slab reaching past the visible end in the odd CTA, which lands on a
    // local barrier for the relay warp.
    const bool el = tc::elect_one();
    RingPos<kVRing> rp;
    SegIter it;
    it.init(&a, c, t_iter);
    int sb, p0, p1, slot, nz = 0;
    bool ok = true;
    const int r = (int)(rank & 1u);
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      TilePages cur;
      cur.load(a, sb, p0, p1);
      for (int i = 0; ok && i < n; ++i) {
        TilePages nxt;
        if (i + 1 < n) nxt.load(a, sb, p0 + (i + 1) * kTile, p1);
        const int ts = p0 + i * kTile;
        const int nv = nslabs_of(ts, p1);
        constexpr int kH = kPair ? 1 : 2;
        for (int v = 0; ok && v < nv; ++v) {
          const int y = cur.row(a, v >> 1, sb, oob_row) + (v & 1) * 32;
          const bool partial = p1 - (ts + 32 * v) < 32;
          for (int h = 0; h < kH; ++h, rp.next()) {
            const int s = rp.s;
            if (rp.n >= kVRing &&
                !cwait<kPair>(&bar[kBEmpty + s], rp.ph ^ 1u, a.status, 81)) {
              ok = false;
              break;
            }
            // the relay must be done with the previous partial slab before
            // another lands on the same local barrier
            if (kPair && !leader && partial && nz > 0 &&
                !warp_wait<false>(&bar[kBZDone], (nz - 1) & 1, a.status, 82)) {
              ok = false;
              break;
            }
            if (aborted()) { ok = false; break; }
            issued = rp.n + 1;
            const uint32_t dst = smem_u32(smem + kOffVRing + s * kStage);
            const uint32_t fb = smem_u32(&bar[kBFull + s]);
            if (el) {
              if (!kPair) {
                tc::mbar_arrive_expect_tx(fb, kStage);
                tc::tma_load_3d(dst, &tmV, 0, y, h * 4, fb);
              } else if (leader) {
                tc::mbar_arrive_expect_tx(fb, 2 * kStage);
                tc::tma_load_3d(dst, &tmV, 0, y, 2 * r, fb);
                tc::tma_load_3d(dst + 8192, &tmV, 0, y, 4 + 2 * r, fb);
              } else if (partial) {
                const uint32_t zb = smem_u32(&bar[kBZb]);
                tc::mbar_arrive_expect_tx(zb, kStage);
                tc::tma_load_3d(dst, &tmV, 0, y, 2 * r, zb);
                tc::tma_load_3d(dst + 8192, &tmV, 0, y, 4 + 2 * r, zb);
              } else {
                const uint32_t lb = cbar(kBFull + s, lead_rank);
                tc::tma_load_3d_pair(dst, &tmV, 0, y, 2 * r, lb);
                tc::tma_load_3d_pair(dst + 8192, &tmV, 0, y, 4 + 2 * r, lb);
              }
            }
            if (kPair && !leader && partial) ++nz;
          }
        }
        cur = nxt;
      }
    }
    if (!ok) set_abort();
  } else if (!score && warp == 1 && leader) {
    // ------------------------------------------------------ value MMA issuer
    // For tile g, once the correction warps released it (P(g) landed and O
    // rescaled if needed): O[:, h*256..] += P(g)[:, slab tokens] V_h(slab),
    // K = 16 tokens per MMA.  Stale rows of a slab past the visible end are
    // zeroed first (this CTA's; the odd CTA's relay zeroes its own).
    const bool el = tc::elect_one();
    constexpr uint32_t idO = tc::idesc_bf16(kPair ? 256 : 128, 256, false, true);
    const uint64_t dP = tc::sdesc(smem_u32(smem + kOffLand), 16, 1024);
    const uint64_t dV = tc::sdesc(smem_u32(smem + kOffVRing), 4096, 1024);
    const uint16_t pvd_mask = (uint16_t)((1u << kCluster) - 1u);   // every CTA
    RingPos<kVRing> rp;
    int g = 0, k = 0;
    bool ok = true;
    SegIter it;
    it.init(&a, c, t_iter);
    int sb, p0, p1, slot;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      for (int i = 0; ok && i < n; ++i) {
        const int gv = g + i;
        // the correction warps release a segment's first tile only after
        // reading out the previous segment's O, so O may be overwritten
        if (!cwait<kPair>(&bar[kBOok + (gv & 1)], (gv >> 1) & 1, a.status, 84)) { ok = false; break; }
        if (aborted()) { ok = false; break; }
        tc::fence_after_sync();
        const int ts = p0 + i * kTile;
        const int nv = nslabs_of(ts, p1);
        const uint64_t dPg = dP + (((gv & 1) * kLandBytes) >> 4);
        constexpr int kH = kPair ? 1 : 2;
        for (int v = 0; ok && v < nv; ++v) {
          for (int h = 0; h < kH; ++h, rp.next()) {
            const int s = rp.s;
            if (!cwait<kPair>(&bar[kBFull + s], rp.ph, a.status, 85)) { ok = false; break; }
            tc::fence_after_sync();
            const int vis = p1 - (ts + 32 * v);
            if (vis < 32) {
              zero_stale_rows<4>(smem + kOffVRing + s * kStage, vis, lane);
              __syncwarp();
            }
            if (el) {
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                const int tok = 32 * v + 16 * kk;   // first token of the K step
                const uint64_t ap = dPg + ((((tok >> 6) * 16384) + (tok & 63) * 2) >> 4);
                const uint32_t acc = (i > 0 || v > 0 || kk > 0) ? 1u : 0u;
                if (!kPair) {
                  tc::mma_ss(tmem + h * 256, ap, dV + ((s * kStage + kk * 2048) >> 4), idO, acc);
                } else {
#pragma unroll
                  for (int cc = 0; cc < 2; ++cc)
                    tc::mma2_ss(tmem + cc * 256, ap,
                                dV + ((s * kStage + cc * 8192 + kk * 2048) >> 4), idO, acc);
                }
              }
              if (kPair) tc::mma2_commit_mc(smem_u32(&bar[kBEmpty + s]), (uint16_t)pair_mask);
              else tc::mma_commit(smem_u32(&bar[kBEmpty + s]));
            }
          }
        }
        if (!ok) break;
        if (el) {
          if (kPair) tc::mma2_commit_mc(smem_u32(&bar[kBPvd + (gv & 1)]), pvd_mask);
          else tc::mma_commit_mc(smem_u32(&bar[kBPvd + (gv & 1)]), pvd_mask);
        }
      }
      g += n;
      ++k;
    }
    if (!ok) set_abort();
    if (el) {
      if (kPair) tc::mma2_commit_mc(smem_u32(&bar[kBDrained]), (uint16_t)pair_mask);
      else tc::mma_commit(smem_u32(&bar[kBDrained]));
    }
  } else if (!score && warp >= 2 && warp < 6) {
    // ------------------------------------------------------ correction / epilogue
    // Thread = head of this CTA's token.  Per tile: wait for P(g), read f
    // and l; if some row of the warp rescales, wait for PV(g-1) and scale O
    // rows by f; release the tile to the MMA issuer.  At the end of a
    // segment: O / l as the segment's fp32 partial.
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const float* landf = reinterpret_cast<const float*>(smem + kOffLand + kLandP);
    const uint32_t srank = rank - (kPair ? 2u : 1u);   // the score CTA of this token
    SegIter it;
    it.init(&a, c, t_iter);
    int sb, p0, p1, slot, g = 0;
    bool ok = true;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      const size_t st_idx = (size_t)slot * a.T + t;   // (slot, token) of the split result
      float* dst = a.part_o + part_off(st_idx, row, 0);   // chunk j at + j * 128
      if (n == 0) {
        const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        for (int j = 0; j < kLat / 8; ++j) st_v8(dst + (size_t)j * 128, z);
        continue;
      }
      float l = 0.f;
      for (int i = 0; i < n; ++i, ++g) {
        if (!bar_wait<true>(&bar[kBLand + (g & 1)], (g >> 1) & 1, a.status, 86)) ok = false;
        if (__any_sync(0xffffffffu, !ok || *abort_flag)) { ok = false; break; }
        // the copy of P(g) has landed: the single staging buffer is free
        if (!kPair && warp == 2 && lane == 0)
          tc::mbar_arrive_cluster_relaxed(cbar(kBStgFree, srank));
        const float* lf = reinterpret_cast<const float*>(
            reinterpret_cast<const uint8_t*>(landf) + (g & 1) * kLandBytes);
        const float f = lf[row];
        l = lf[128 + row];
        if (__any_sync(0xffffffffu, f != 1.f)) {
          // O holds PV(0..g-1); i > 0 here (the first tile never rescales)
          if (!bar_wait<true>(&bar[kBPvd + ((g - 1) & 1)], ((g - 1) >> 1) & 1, a.status, 87))
            ok = false;
          if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
          tc::fence_after_sync();
          for (int c0 = 0; c0 < kLat; c0 += 16) {
            float v[16];
            tc::tmem_ld16(trow + c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] *= f;
            tc::tmem_st16(trow + c0, v);
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          if (kPair) tc::mbar_arrive_cluster_relaxed(cbar(kBOok + (g & 1), lead_rank));
          else tc::mbar_arrive(smem_u32(&bar[kBOok + (g & 1)]));
        }
      }
      if (!ok) break;
      // PV of the segment's last tile done implies every earlier one is
      if (!bar_wait<true>(&bar[kBPvd + ((g - 1) & 1)], ((g - 1) >> 1) & 1, a.status, 88)) ok = false;
      if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
      tc::fence_after_sync();
      // l = 0 only when this token sees none of the segment's tokens
      const float inv = l > 0.f ? 1.f / l : 0.f;
      if (a.slot_base[sb + 1] - a.slot_base[sb] == 1) {
        // the sequence lies in this split alone: O / l is its latent output
        // (bf16, as the combine would write it); the combine skips it
        __nv_bfloat16* od = a.o_lat + (((size_t)sb * a.T + t) * kHeads + row) * kLat;
        for (int c0 = 0; c0 < kLat; c0 += 64) {
          uint32_t v[64];
          tc::tmem_ld64(trow + c0, v);
#pragma unroll
          for (int j = 0; j < 64; j += 16) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[j + 2 * e]) * inv,
                                                              __uint_as_float(v[j + 2 * e + 1]) * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            st_v8(od + c0 + j, w);
          }
        }
      } else {
        for (int c0 = 0; c0 < kLat; c0 += 64) {
          uint32_t v[64];
          tc::tmem_ld64(trow + c0, v);
#pragma unroll
          for (int j = 0; j < 64; j += 8) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(__uint_as_float(v[j + e]) * inv);
            st_v8(dst + (size_t)((c0 + j) >> 3) * 128, w);
          }
        }
      }
      tc::fence_before_sync();
    }
    if (!ok) set_abort();
  } else if (kPair && !score && !leader && warp == 6) {
    // ------------------------------------------------------ relay (odd value CTA)
    // A value slab reaching past the visible end lands on the local zb
    // barrier; zero its stale rows, then count its bytes on the leader's
    // ring barrier.  The producer waits for zdone before the next such slab.
    const bool el = tc::elect_one();
    RingPos<kVRing> rp;
    SegIter it;
    it.init(&a, c, t_iter);
    int sb, p0, p1, slot, nz = 0;
    bool ok = true;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      for (int i = 0; ok && i < n; ++i) {
        const int ts = p0 + i * kTile;
        const int nv = nslabs_of(ts, p1);
        for (int v = 0; v < nv; ++v, rp.next()) {
          const int vis = p1 - (ts + 32 * v);
          if (vis >= 32) continue;
          if (!warp_wait<false>(&bar[kBZb], nz & 1, a.status, 89)) { ok = false; break; }
          if (aborted()) { ok = false; break; }
          zero_stale_rows<4>(smem + kOffVRing + rp.s * kStage, vis, lane);
          __syncwarp();
          if (el) {
            tc::fence_acq_rel_cluster();   // publish the zeros to the leader's MMA
            tc::mbar_complete_tx_cluster(cbar(kBFull + rp.s, lead_rank), kStage);
            tc::mbar_arrive(smem_u32(&bar[kBZDone]));
          }
          ++nz;
        }
      }
    }
    if (!ok) set_abort();
  }

  // ------------------------------------------------------------ teardown
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    // let this CTA's own copies land before its shared memory goes away; the
    // odd CTA of a pair counts its ring copies on the leader's barriers, so
    // it waits a fixed time far above a copy's latency instead
    if (!kPair || leader) {
      const int R = score ? kSRing : kVRing;
      for (int i = 0; i < R && i < issued; ++i) {
        const int u = issued - 1 - i;
        mbar_wait_cluster(&bar[kBFull + u % R], (u / R) & 1, a.status, 90, 100000000ull);
      }
    } else {
      const uint64_t t0 = global_ns();
      while (global_ns() - t0 < 200000ull) {
      }
    }
    if (qr_issued > 0) mbar_wait(&bar[kBQr], (qr_issued - 1) & 1, a.status, 91, 1 << 20, 100000000ull);
  }
  if (warp == 1) {
    // the pair leader's MMAs read this CTA's shared memory and write its TMEM
    mbar_wait_cluster(&bar[kBDrained], 0, a.status, 92, 100000000ull);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();   // no CTA leaves while another may still write into it
  tc::fence_after_sync();
  if (warp == 1) {
    if (kPair) tc::tmem_dealloc2(tmem, kTmemCols);
    else tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool kPair>
bool launch_sv(mla_ctx* ctx, const CUtensorMap& tmS, const CUtensorMap& tmS2,
               const CUtensorMap& tmV, const AttArgs& a, int G, int T, cudaStream_t st) {
  auto kern = attend_sv_kernel<kPair>;
  static std::atomic<uint64_t> attr_done{0};
  if (smem_attr_once(attr_done, kern, (int)SvLayout<kPair>::kSmem) != cudaSuccess) return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = kPair ? dim3(4, G, T / 2) : dim3(2 * G, T, 1);
  cfg.blockDim = dim3(224);
  cfg.dynamicSmemBytes = SvLayout<kPair>::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kPair ? 4 : 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  prof_mark(ctx, st, "attend");
  ctx->launches += 1;
  return cudaLaunchKernelEx(&cfg, kern, tmS, tmS2, tmV, a) == cudaSuccess;
}

}  // namespace

bool sv_attend(mla_ctx* ctx, const __nv_bfloat16* qimg, const __nv_bfloat16* cache,
               int num_pages, const int32_t* bt, int max_pages, int B, int T, char* ws,
               const WsLayout& L, cudaStream_t st) {
  const bool pair = T % 2 == 0;
  CUtensorMap tmS, tmS2, tmV;
  const uint64_t rows = (uint64_t)num_pages * kPage;
  if (!make_tmap_bf16_2d(&tmS, cache, rows, kRow, kRow, 64, 64, false) ||
      !make_tmap_pool_blocks(&tmS2, cache, rows, 64, 2) ||
      !make_tmap_pool_blocks(&tmV, cache, rows, 32, pair ? 2 : 4))
    return false;
  AttArgs a{};
  a.lens = reinterpret_cast<const int*>(ws + L.lens);
  a.prefix = reinterpret_cast<const int*>(ws + L.page_prefix);
  a.first_split = reinterpret_cast<const int*>(ws + L.first_split);
  a.slot_base = reinterpret_cast<const int*>(ws + L.slot_base);
  a.meta = reinterpret_cast<const int*>(ws + L.meta);
  a.bt = bt;
  a.qimg = reinterpret_cast<const uint8_t*>(qimg);
  a.cache = cache;
  a.part_o = reinterpret_cast<float*>(ws + L.part_o);
  a.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  a.o_lat = reinterpret_cast<__nv_bfloat16*>(ws + L.o_lat);
  a.status = ctx->status;
  a.B = B;
  a.T = T;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.scale_log2 = ctx->cfg.softmax_scale * 1.4426950408889634f;
  return pair ? launch_sv<true>(ctx, tmS, tmS2, tmV, a, L.G, T, st)
              : launch_sv<false>(ctx, tmS, tmS2, tmV, a, L.G, T, st);
}

}  // namespace mla

namespace mla {

// How many attention clusters of each kind the device runs at once (the
// split count never exceeds it, so every split starts in the first wave).
bool sv_setup(mla_ctx* ctx) {
  for (int pair = 0; pair < 2; ++pair) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = pair ? dim3(4, 1, 1) : dim3(2, 1, 1);
    cfg.blockDim = dim3(224);
    cfg.dynamicSmemBytes = pair ? SvLayout<true>::kSmem : SvLayout<false>::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = pair ? 4 : 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e;
    if (pair) {
      static std::atomic<uint64_t> done{0};
      e = smem_attr_once(done, attend_sv_kernel<true>, (int)SvLayout<true>::kSmem);
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, attend_sv_kernel<true>, &cfg);
    } else {
      static std::atomic<uint64_t> done{0};
      e = smem_attr_once(done, attend_sv_kernel<false>, (int)SvLayout<false>::kSmem);
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveClusters(&n, attend_sv_kernel<false>, &cfg);
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    ctx->sv_clusters[pair] = n;
  }
  return true;
}

}  // namespace mla
