// Split-KV flash-decoding for an even number of query tokens per sequence,
// on pairs of CTAs (tcgen05 cta_group::2).
//
// Absorbed MLA attention as in attend_tc.cu (page "DeepSeek-V2：在“大力出奇迹”
// 的AI军备竞赛中，四两拨千斤", liang.world, 第二章 §2 absorption and §3
// decoupled RoPE): s = Q C^T * scale, a = softmax(s), o_lat = a C[:, :512].
// Query tokens 2j and 2j+1 of a sequence attend over the same cache tiles
// (the causal limit differs by one token and is applied per row), so a
// cluster of two CTAs, one per token, for the same KV split and the same
// half of d_latent computes both with M = 256 MMAs: rows 0..127 are the heads
// of token 2j (even CTA), rows 128..255 the heads of token 2j+1 (odd CTA).
// Each CTA streams only its half of every tile:
//   score MMA  S (256 x 128 tokens): B = the tile's 128 cache rows, split by
//              N: the even CTA loads the tile's first page, the odd CTA the
//              second, 8 KB [64 tokens x 64 features] per block;
//   value MMA  O (256 x 256 cols) += P V: B = V[:, this half], split by N:
//              each CTA loads 128 of the half's 256 columns, 8 KB
//              [32 tokens x 128 columns] per slab.
// So a CTA moves 104 KB per 128-token tile (the unpaired kernel: 208 KB) in
// 7 ring stages of 16 KB (the unpaired kernel: 13), and one MMA instruction
// serves two query tokens: issuing stages, not the tensor cores, is what
// bounds these kernels.  The even CTA's threads
// issue every MMA; each CTA's softmax warps work on their own TMEM rows.
//
// Ring protocol (5 stages of 16 KB in each CTA): the even CTA's `ring`
// barrier of a stage expects both CTAs' bytes; the odd CTA's copies complete
// it directly (cta_group::2 form of the TMA load).  The one exception is a
// value slab reaching past the visible end: the odd CTA loads it against a
// local barrier, its relay warp zeroes the stale rows and then counts the
// bytes on the even CTA's barrier.  The relay also forwards the odd CTA's
// query image.  MMA commits reach the barrier at the same offset in both
// CTAs; the softmax warps of both CTAs arrive on the even CTA's p_full and
// o_free.
//
// Roles (256 threads): warp 0 producer (both CTAs), warp 1 score-MMA issuer
// (even CTA) and TMEM allocation (both), warps 2-5 softmax (both), warp 6
// value-MMA issuer (even CTA), warp 7 relay (odd CTA).  Every wait is
// bounded; a failure sets both CTAs' abort flags.
#include "attend_common.cuh"
#include "tmap.h"
#include "launch_util.h"

namespace mla {
namespace {

using namespace att;

constexpr int kPRing = 5;                                   // ring stages
constexpr uint32_t kPStage = 16384;                         // one ring stage
constexpr uint32_t kPHalf = 8192;                           // one block or slab
constexpr uint32_t kPOffRing = kQImgBytes;                  // 147456
constexpr uint32_t kPOffBar = kPOffRing + kPRing * kPStage; // 229376
constexpr uint32_t kPSmem = kPOffBar + 512 + 1024;
using PRing = RingPos<kPRing>;

// A stage holds two 8 KB units of this CTA's half: score blocks b, b+1 (or
// block 8 alone) or value slabs v, v+1 (or the last slab alone).  Ring step
// i of a segment (i = 0..n) holds the score stages {0,1} {2,3} of tile i,
// the value stages of tile i-1, then the score stages {4,5} {6,7} {8} of
// tile i (score stages only for i < n, value stages only for i >= 1), so
// PV(i-1) overlaps S(i).  Stage j of a step with (sc) score blocks and nv
// value slabs: returns the first block (>= 0) or -1 - first slab, and the
// number of units in *cnt.
__device__ __forceinline__ int step_stage(int j, bool sc, int nv, int* cnt) {
  const int nvs = (nv + 1) >> 1;
  const int head = sc ? 2 : 0;
  if (j < head) {
    *cnt = 2;
    return 2 * j;
  }
  if (j < head + nvs) {
    const int v = 2 * (j - head);
    *cnt = min(2, nv - v);
    return -1 - v;
  }
  const int b = 2 * (j - nvs);
  *cnt = b == 8 ? 1 : 2;
  return b;
}

__device__ __forceinline__ int step_stages(bool sc, int nv) { return (sc ? 5 : 0) + ((nv + 1) >> 1); }

__global__ void __launch_bounds__(256, 1)
attend_pair_kernel(const __grid_constant__ CUtensorMap tmS,
                   const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmS2,   // two score blocks
                   const __grid_constant__ CUtensorMap tmV2,   // two value slabs
                   const AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kPOffBar);
  uint64_t* ring = bar;            // [kPRing] see the ring protocol above
  uint64_t* empty = bar + 10;      // [kPRing] stage consumed by the MMAs
  uint64_t* s_full = bar + 20;     // [2] S of tiles of that parity done
  uint64_t* pv_done = bar + 22;    // [2] PV of tiles of that parity done
  uint64_t* p_full = bar + 24;     // [2] even CTA: P written (8 warps)
  uint64_t* q_full = bar + 26;     // even CTA: both query images; odd: its own
  uint64_t* q_empty = bar + 27;    // score MMAs of a segment done
  uint64_t* o_free = bar + 28;     // even CTA: O read out (8 warps)
  uint64_t* drained = bar + 29;    // both MMA issuers' last MMAs done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 30);
  uint64_t* zb = bar + 31;         // odd CTA: partial value slab loaded locally
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // grid (T, splits, 2): the CTA pair runs along x (tokens 2j, 2j+1), as
  // cta_group::2 pairs are formed along the cluster's x dimension
  const int t = blockIdx.x, c = blockIdx.y, half = blockIdx.z;
  const uint32_t rank = tc::cluster_rank();   // t & 1
  const bool even = rank == 0;

  tc::grid_dep_launch();
  tc::grid_dep_wait();   // plan, query image and cache come from earlier kernels
  if (c >= a.meta[0]) return;   // both CTAs of a pair have the same split

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPRing; ++i) {
      mbar_init(&ring[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&pv_done[i], 1);
      mbar_init(&p_full[i], 8);
    }
    mbar_init(q_full, even ? 2 : 1);
    mbar_init(q_empty, 1);
    mbar_init(o_free, 8);
    mbar_init(drained, 2);
    mbar_init(zb, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc2(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish2();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmS);
    tc::prefetch_tmap(&tmV);
    tc::prefetch_tmap(&tmS2);
    tc::prefetch_tmap(&tmV2);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();   // barriers and TMEM of both CTAs ready
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const uint32_t sQ = smem_u32(smem);
  const uint32_t sR = smem_u32(smem + kPOffRing);
  const int oob_row = a.num_pages * kPage + kPage;   // TMA zero-fills rows out of range
  // cluster address of a barrier of this block in the even CTA
  const uint32_t bar_even = tc::mapa_shared(smem_u32(bar), 0);
  auto even_bar = [&](uint64_t* b) {
    return bar_even + (uint32_t)(reinterpret_cast<uint8_t*>(b) - reinterpret_cast<uint8_t*>(bar));
  };
  auto set_abort = [&] {
    *abort_flag = 1;
    tc::st_cluster_u32(tc::mapa_shared(smem_u32((const void*)abort_flag), rank ^ 1u), 1u);
  };
  int issued = 0;     // producer: ring stages issued
  int q_issued = 0;   // producer: query images issued

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    // Warp-uniform loop, one elected lane issues.  Per segment: this CTA's
    // query image, then ring steps i = 0..n (see step_stage) with this CTA's
    // half of each stage.  The odd CTA's producer waits on its own `empty`
    // barriers (the MMA commits reach both CTAs) but signals the even CTA's.
    const bool leader = tc::elect_one();
    PRing rp;
    SegIter it;
    it.init(&a, c, t | 1);   // the pair iterates the odd token's range
    int sb, p0, p1, slot, k = 0;
    bool ok = true;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      if (k > 0 && !warp_wait<true>(q_empty, (k - 1) & 1, a.status, 41)) { ok = false; break; }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      ++q_issued;
      if (leader) {
        tc::mbar_arrive_expect_tx(smem_u32(q_full), kQImgBytes);
        const uint8_t* qsrc = a.qimg + ((size_t)sb * a.T + t) * kQImgBytes;
        for (int fb = 0; fb < 9; ++fb)
          tc::bulk_load(sQ + fb * 16384, qsrc + fb * 16384, 16384, smem_u32(q_full));
      }
      TilePages cur, prev;   // tile i (score blocks) and tile i-1 (value slabs)
      cur.load(a, sb, p0, p1);
      for (int i = 0; ok && i <= n; ++i) {
        const bool sc = i < n;
        const int tv = p0 + (i - 1) * kTile;   // tile whose value slabs follow
        const int nv = i >= 1 ? nslabs_of(tv, p1) : 0;
        TilePages nxt;
        if (i + 1 < n) nxt.load(a, sb, p0 + (i + 1) * kTile, p1);   // used next step
        // pool row of this CTA's page of tile i
        const int ys = sc ? cur.row(a, (int)rank, sb, oob_row) : 0;
        const int ns = step_stages(sc, nv);
        for (int j = 0; j < ns; ++j, rp.next()) {
          const int s = rp.s;
          if (rp.n >= kPRing && !warp_wait<true>(&empty[s], rp.ph ^ 1u, a.status, 42)) {
            ok = false;
            break;
          }
          if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
          int cnt;
          const int first = step_stage(j, sc, nv, &cnt);
          const uint32_t fb = smem_u32(&ring[s]);
          const uint32_t dst = sR + s * kPStage;
          // slab rows: slab v is page v / 2 of tile i-1, rows (v % 2) * 32..
          int y[2] = {0, 0};
          bool partial = false;   // the stage holds a slab past the visible end
          if (first < 0) {
            const int v = -1 - first;
            for (int u = 0; u < cnt; ++u)
              y[u] = prev.row(a, (v + u) >> 1, sb, oob_row) + ((v + u) & 1) * 32;
            partial = p1 - (tv + 32 * (v + cnt - 1)) < 32;
          }
          issued = rp.n + 1;
          if (leader) {
            const uint32_t bytes = cnt * kPHalf;
            if (even) tc::mbar_arrive_expect_tx(fb, 2 * bytes);   // both CTAs' halves
            if (!even && partial) tc::mbar_arrive_expect_tx(smem_u32(zb), bytes);
            const uint32_t eb = even_bar(&ring[s]);
            const uint32_t zbb = smem_u32(zb);
            const int vb = half * 4 + (int)rank * 2;   // this CTA's value column blocks
            if (cnt == 2 && first >= 0) {
              // both blocks in one copy ([2][64 rows][64])
              if (even) tc::tma_load_3d(dst, &tmS2, 0, ys, first, fb);
              else tc::tma_load_3d_pair(dst, &tmS2, 0, ys, first, eb);
            } else if (cnt == 2) {
              // both slabs (one page, 64 rows) in one copy ([2][2 blocks][32][64])
              const int slab = y[0] / 32;
              if (even) tc::tma_load_4d(dst, &tmV2, 0, 0, vb, slab, fb);
              else if (partial) tc::tma_load_4d(dst, &tmV2, 0, 0, vb, slab, zbb);
              else tc::tma_load_4d_pair(dst, &tmV2, 0, 0, vb, slab, eb);
            } else if (first >= 0) {
              if (even) tc::tma_load_2d(dst, &tmS, first * 64, ys, fb);
              else tc::tma_load_2d_pair(dst, &tmS, first * 64, ys, eb);
            } else {
#pragma unroll
              for (int f = 0; f < 2; ++f) {
                const uint32_t d = dst + f * 4096;
                const int x = (vb + f) * 64;
                if (even) tc::tma_load_2d(d, &tmV, x, y[0], fb);
                else if (partial) tc::tma_load_2d(d, &tmV, x, y[0], zbb);
                else tc::tma_load_2d_pair(d, &tmV, x, y[0], eb);
              }
            }
          }
        }
        prev = cur;
        cur = nxt;
      }
      ++k;
    }
    if (!ok) set_abort();
  } else if (warp == 1 && even) {
    // -------------------------------------------------------- score-MMA issuer
    // As in the unpaired kernel, with M = 256 and a stage made of both CTAs'
    // halves; steps over the value stages.
    const bool leader = tc::elect_one();
    constexpr uint32_t idS = tc::idesc_bf16(256, kTile, false, false);
    const uint64_t dQ = tc::sdesc(sQ, 16, 1024);
    const uint64_t dR = tc::sdesc(sR, 16, 1024);
    PRing rp;
    int g = 0, k = 0;
    bool ok = true;
    SegIter it;
    it.init(&a, c, t | 1);   // the pair iterates the odd token's range
    int sb, p0, p1, slot;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      if (!warp_wait<true>(q_full, k & 1, a.status, 45)) { ok = false; break; }
      for (int i = 0; ok && i <= n; ++i) {
        const int gs = g + i;
        const bool sc = i < n;
        const int nv = i >= 1 ? nslabs_of(p0 + (i - 1) * kTile, p1) : 0;
        if (sc) {
          // S(gs) reuses the TMEM columns of P(gs-2), and its slots last held
          // value slabs of tiles gs-2 (and gs-1 at a segment's first tile)
          if (gs >= 2 && !warp_wait<true>(&pv_done[gs & 1], ((gs - 2) >> 1) & 1, a.status, 46)) {
            ok = false;
            break;
          }
          if (i == 0 && gs >= 1 &&
              !warp_wait<true>(&pv_done[(gs - 1) & 1], ((gs - 1) >> 1) & 1, a.status, 55)) {
            ok = false;
            break;
          }
        }
        const uint32_t dcol = tmem + kColS + (gs & 1) * kTile;
        const int ns = step_stages(sc, nv);
        for (int j = 0; j < ns; ++j, rp.next()) {
          int cnt;
          const int b0 = step_stage(j, sc, nv, &cnt);
          if (b0 < 0) continue;   // value slabs: the value-MMA warp's
          const int s = rp.s;
          if (!warp_wait<true>(&ring[s], rp.ph, a.status, 47)) { ok = false; break; }
          tc::fence_after_sync();
          if (leader) {
            for (int u = 0; u < cnt; ++u) {
              const int b = b0 + u;
              const uint64_t dRs = dR + ((s * kPStage + u * kPHalf) >> 4);
              const uint64_t dQb = dQ + ((b * 16384) >> 4);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc::mma2_ss(dcol, dQb + kk * 2, dRs + kk * 2, idS, (b > 0 || kk > 0) ? 1u : 0u);
            }
            tc::mma2_commit_both(smem_u32(&empty[s]));
          }
        }
        if (!ok) break;
        if (sc && leader) {
          tc::mma2_commit_both(smem_u32(&s_full[gs & 1]));
          if (i == n - 1) tc::mma2_commit_both(smem_u32(q_empty));
        }
      }
      g += n;
      ++k;
    }
    if (!ok) set_abort();
    if (leader) tc::mma2_commit_both(smem_u32(drained));
  } else if (warp == 6 && even) {
    // -------------------------------------------------------- value-MMA issuer
    // Steps over the score stages; for tile x waits for P(x) of both CTAs,
    // then O += P(x) V(x).
    const bool leader = tc::elect_one();
    constexpr uint32_t idO = tc::idesc_bf16(256, 256, false, true);
    const uint64_t dV = tc::sdesc(sR, 4096, 1024);   // value slab: MN-major, 2 x 64 columns
    PRing rp;
    int g = 0, k = 0;
    bool ok = true;
    SegIter it;
    it.init(&a, c, t | 1);   // the pair iterates the odd token's range
    int sb, p0, p1, slot;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      for (int i = 0; ok && i <= n; ++i) {
        const int gv = g + i - 1;
        const int tv = p0 + (i - 1) * kTile;
        const bool sc = i < n;
        const int nv = i >= 1 ? nslabs_of(tv, p1) : 0;
        if (i >= 1) {
          if (i == 1 && k > 0 && !warp_wait<true>(o_free, (k - 1) & 1, a.status, 48)) { ok = false; break; }
          // P(gv) written means S(gv) is done, so every slot this step's
          // slabs reuse has been consumed in its previous lap
          if (!warp_wait<true>(&p_full[gv & 1], (gv >> 1) & 1, a.status, 49)) { ok = false; break; }
          if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
          tc::fence_after_sync();
        }
        const uint32_t pcol = tmem + kColS + (gv & 1) * kTile;
        const int ns = step_stages(sc, nv);
        for (int j = 0; j < ns; ++j, rp.next()) {
          int cnt;
          const int first = step_stage(j, sc, nv, &cnt);
          if (first >= 0) continue;   // score blocks: the score-MMA warp's
          const int v0 = -1 - first;
          const int s = rp.s;
          if (!warp_wait<true>(&ring[s], rp.ph, a.status, 51)) { ok = false; break; }
          tc::fence_after_sync();
          const int vis = p1 - (tv + 32 * (v0 + cnt - 1));   // last slab of the stage
          if (vis < 32) {
            zero_stale_rows<2>(smem + kPOffRing + s * kPStage + (cnt - 1) * kPHalf, vis, lane);
            __syncwarp();
          }
          if (leader) {
            for (int u = 0; u < cnt; ++u) {
              const int v = v0 + u;
#pragma unroll
              for (int kk = 0; kk < 2; ++kk)
                tc::mma2_ts(tmem, pcol + 16 * v + 8 * kk,
                            dV + ((s * kPStage + u * kPHalf + kk * 2048) >> 4), idO,
                            (i > 1 || v > 0 || kk > 0) ? 1u : 0u);
            }
            tc::mma2_commit_both(smem_u32(&empty[s]));
          }
        }
        if (!ok) break;
        if (i >= 1 && leader) tc::mma2_commit_both(smem_u32(&pv_done[gv & 1]));
      }
      g += n;
      ++k;
    }
    if (!ok) set_abort();
    if (leader) tc::mma2_commit_both(smem_u32(drained));
  } else if (warp == 7 && !even) {
    // -------------------------------------------------------------- relay
    // Forwards this CTA's query image, and finishes the value stages that
    // reach past the visible end: zero the stale rows, then count the bytes
    // on the even CTA's ring barrier.  Such a stage is a segment's last, so
    // two of them are at least a ring lap apart: zb never runs two phases
    // ahead of this warp.
    const bool leader = tc::elect_one();
    PRing rp;
    SegIter it;
    it.init(&a, c, t | 1);   // the pair iterates the odd token's range
    int sb, p0, p1, slot, k = 0, nz = 0;
    bool ok = true;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      if (!warp_wait<true>(q_full, k & 1, a.status, 43)) { ok = false; break; }
      if (leader) tc::mbar_arrive_cluster_relaxed(even_bar(q_full));
      for (int i = 0; ok && i <= n; ++i) {
        const bool sc = i < n;
        const int tv = p0 + (i - 1) * kTile;
        const int nv = i >= 1 ? nslabs_of(tv, p1) : 0;
        const int ns = step_stages(sc, nv);
        for (int j = 0; j < ns; ++j, rp.next()) {
          int cnt;
          const int first = step_stage(j, sc, nv, &cnt);
          if (first >= 0) continue;
          const int vis = p1 - (tv + 32 * (-1 - first + cnt - 1));
          if (vis >= 32) continue;
          if (!warp_wait<true>(zb, nz & 1, a.status, 44)) { ok = false; break; }
          if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
          zero_stale_rows<2>(smem + kPOffRing + rp.s * kPStage + (cnt - 1) * kPHalf, vis, lane);
          __syncwarp();
          if (leader) {
            tc::fence_acq_rel_cluster();   // publish the zeros to the even CTA
            tc::mbar_complete_tx_cluster(even_bar(&ring[rp.s]), cnt * kPHalf);
          }
          ++nz;
        }
      }
      ++k;
    }
    if (!ok) set_abort();
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ softmax warps
    // One arrival per warp on the even CTA's barriers, after every lane's
    // TMEM stores (P) or loads (O) have been waited for and fenced inside
    // softmax_role; nothing else needs publishing, so the arrive is relaxed.
    softmax_role<true>(
        a, tmem, warp, lane, c, t, t | 1, half, &s_full[0], &s_full[1], &pv_done[0], &pv_done[1],
        abort_flag,
        [&](int g) {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive_cluster_relaxed(even_bar(&p_full[g & 1]));
        },
        [&] {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive_cluster_relaxed(even_bar(o_free));
        });
    if (*abort_flag) set_abort();
  }

  // ------------------------------------------------------------ teardown
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    // let this CTA's own copies land before its shared memory goes away; the
    // odd CTA's ring copies complete the even CTA's barriers, so it waits a
    // fixed time far above a copy's latency instead
    if (even) {
      for (int i = 0; i < kPRing && i < issued; ++i) {
        const int u = issued - 1 - i;
        mbar_wait_cluster(&ring[u % kPRing], (u / kPRing) & 1, a.status, 52, 100000000ull);
      }
    } else {
      const uint64_t t0 = global_ns();
      while (global_ns() - t0 < 200000ull) {
      }
    }
    if (q_issued > 0) mbar_wait_cluster(q_full, (q_issued - 1) & 1, a.status, 53, 100000000ull);
  }
  if (warp == 1) {
    // the even CTA's MMAs read this CTA's shared memory and write its TMEM
    mbar_wait_cluster(drained, 0, a.status, 54, 100000000ull);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc2(tmem, kTmemCols);
}

}  // namespace

bool tc_attend_pair(mla_ctx* ctx, const __nv_bfloat16* qimg, const __nv_bfloat16* cache,
                    int num_pages, const int32_t* bt, int max_pages, int B, int T, char* ws,
                    const WsLayout& L, cudaStream_t st) {
  if (T % 2 != 0) return false;
  CUtensorMap tmS, tmV, tmS2, tmV2;
  const uint64_t rows = (uint64_t)num_pages * kPage;
  if (!make_tmap_bf16_2d(&tmS, cache, rows, kRow, kRow, 64, 64, false) ||
      !make_tmap_bf16_2d(&tmV, cache, rows, kRow, kRow, 64, 32, false) ||
      !make_tmap_pool_blocks(&tmS2, cache, rows, 64, 2) || !make_tmap_pool_slabs(&tmV2, cache, rows, 2))
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
  a.status = ctx->status;
  a.B = B;
  a.T = T;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.scale_log2 = ctx->cfg.softmax_scale * 1.4426950408889634f;
  static std::atomic<uint64_t> attr_done{0};
  if (smem_attr_once(attr_done, attend_pair_kernel, (int)kPSmem) != cudaSuccess) return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T, L.G, 2);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  prof_mark(ctx, st, "attend");
  ctx->launches += 1;
  return cudaLaunchKernelEx(&cfg, attend_pair_kernel, tmS, tmV, tmS2, tmV2, a) == cudaSuccess;
}

}  // namespace mla
