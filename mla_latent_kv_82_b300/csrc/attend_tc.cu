// Split-KV flash-decoding over the bf16 latent cache on tcgen05 tensor cores.
//
// Absorbed MLA attention (page "DeepSeek-V2：在“大力出奇迹”的AI军备竞赛中，
// 四两拨千斤", liang.world, 第二章 §2 absorption and §3 decoupled RoPE): with
// the query image Q = [W^UK_i^T q^C_i ; RoPE(q^R_i)] (128 heads x 576) and
// the cached rows C = [c^KV ; k^R] (tokens x 576),
//     s = Q C^T * scale,  a = softmax(s),  o_lat = a C[:, :512].
// The 128 heads are the M = 128 side of both MMAs, 128 cache tokens the N
// side of the score MMA (one tcgen05.mma takes about as long at N = 16 as at
// N = 128, so narrow token tiles waste the tensor core):
//     S (128 x 128 tokens)  = sum over 9 feature blocks Q_b . C_b^T  -> TMEM
//     O (128 x 256 cols)   += P (128 x 128, bf16) . C[:, half]       -> TMEM
// One CTA owns one KV split of one query token and one half (256 columns)
// of the latent output; both halves compute the same S, so their softmax
// statistics agree bit for bit.  TMEM: O half (256 columns) + two S buffers
// (2 x 128), so S of the next tile is computed while the softmax of this one
// runs; P (bf16) overwrites the S buffer it came from and feeds the value
// MMA straight from TMEM.  Shared memory: the query image stays resident
// (144 KB); the cache streams through a 5-deep ring of 16 KB stages, first
// as score blocks [128 tokens x 64 features] (one per feature block), then
// as value slabs [32 tokens x 256 features of this half].
//
// Roles (224 threads): warp 0 = TMA producer, warp 1 = score-MMA issuer and
// TMEM owner, warp 6 = value-MMA issuer (two issuing threads, so that the
// per-stage issue overhead of the two streams overlaps), warps 2-5 = softmax
// (thread = head): online softmax in the log2 domain with a lazy rescale (O
// and l are rescaled only when a row maximum grows by more than 2^8, so
// P <= 256), P packed two bf16 per TMEM column.  At the end of a segment the
// same warps write O / l and m + log2 l for the log-sum-exp combine.  Every
// wait is bounded; on a timeout the CTA records MLA_ERR_TIMEOUT, drains its
// own loads and frees TMEM.
#include "attend_common.cuh"
#include "tmap.h"
#include "launch_util.h"

namespace mla {
namespace {

constexpr int kRing = 5;                                   // ring stages
constexpr uint32_t kStage = 16384;                         // one ring stage
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffRing = kQImgBytes;                  // 147456
constexpr uint32_t kOffBar = kOffRing + kRing * kStage;    // 229376
constexpr uint32_t kSmem = kOffBar + 256 + 1024;

using namespace att;
using Ring = RingPos<kRing>;

__global__ void __launch_bounds__(224, 1)
attend_tc_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmV,
                 const AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bar;          // [kRing]
  uint64_t* empty = bar + 8;     // [kRing]
  uint64_t* s_full = bar + 16;   // [2] S buffer g&1 holds S(g)
  // P(g) written: two barriers by tile parity, so the softmax warps, which
  // may finish tile g+1 before the MMA thread waits for tile g, never move
  // one barrier two phases past its waiter
  uint64_t* const p_full = bar + 18;   // tile g: p_full + 6 * (g & 1)
  // PV(g) done, also by tile parity: a waiter for PV(g) has always seen
  // PV(g-2) complete (it precedes S(g) in the MMA pipe) and PV(g+2) cannot
  // start before that waiter's own P(g+2)
  uint64_t* const pv_done = bar + 19;  // tile g: pv_done + 6 * (g & 1)
  uint64_t* const drained = bar + 26;   // both MMA issuers' last MMAs done
  uint64_t* q_full = bar + 20;
  uint64_t* q_empty = bar + 21;
  uint64_t* o_free = bar + 22;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 23);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, t = blockIdx.y, half = blockIdx.z;

  tc::grid_dep_launch();
  tc::grid_dep_wait();   // plan, query image and cache come from earlier kernels
  if (c >= a.meta[0]) return;   // more CTAs than KV splits in use

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&s_full[i], 1);
    mbar_init(p_full, 128);
    mbar_init(p_full + 6, 128);
    mbar_init(pv_done, 1);
    mbar_init(pv_done + 6, 1);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(o_free, 128);
    mbar_init(drained, 2);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmS);
    tc::prefetch_tmap(&tmV);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint32_t sR = smem_u32(smem + kOffRing);
  const int oob_row = a.num_pages * kPage + kPage;   // TMA zero-fills rows out of range
  int issued = 0;     // producer: ring stages issued
  int q_issued = 0;   // producer: query images issued

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    // The whole warp runs the loop with identical (warp-uniform) values and
    // one elected lane issues the copies: a single divergent lane would keep
    // every operand in per-thread registers and pay a conversion per issue.
    // Per segment: the query image, then step i = 0..n loads the 9 score
    // blocks of tile i (i < n) followed by the value slabs of tile i-1
    // (i >= 1), the order in which the MMA warp consumes them.
    const bool leader = tc::elect_one();
    Ring rp;   // next stage to fill
    SegIter it;
    it.init(&a, c, t);
    int sb, p0, p1, slot, k = 0;
    bool ok = true;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      if (k > 0 && !warp_wait(q_empty, (k - 1) & 1, a.status, 21)) { ok = false; break; }
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
        const int nsc = i < n ? 9 : 0;
        const int tv = p0 + (i - 1) * kTile;   // tile whose value slabs follow
        const int nv = i >= 1 ? nslabs_of(tv, p1) : 0;
        TilePages nxt;
        if (i + 1 < n) nxt.load(a, sb, p0 + (i + 1) * kTile, p1);   // used next step
        int y0 = 0, y1 = 0;
        if (nsc) {
          y0 = cur.row(a, 0, sb, oob_row);
          y1 = cur.row(a, 1, sb, oob_row);
        }
        for (int j = 0; j < nsc + nv; ++j, rp.next()) {
          const int s = rp.s;
          // the stage's previous pass must have been consumed
          if (rp.n >= kRing && !warp_wait(&empty[s], rp.ph ^ 1u, a.status, 22)) {
            ok = false;
            break;
          }
          if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
          const uint32_t fb = smem_u32(&full[s]);
          const uint32_t dst = sR + s * kStage;
          int y = 0;
          if (j >= nsc) {
            const int v = j - nsc;   // slab: page v / 2 of tile i-1, rows (v % 2) * 32..
            y = prev.row(a, v >> 1, sb, oob_row) + (v & 1) * 32;
          }
          issued = rp.n + 1;
          if (leader) {
            tc::mbar_arrive_expect_tx(fb, kStage);
            if (j < nsc) {
              tc::tma_load_2d(dst, &tmS, j * 64, y0, fb);
              tc::tma_load_2d(dst + 8192, &tmS, j * 64, y1, fb);
            } else {
              // the slab's 4 column blocks of this half in one copy ([4][32][64])
              tc::tma_load_3d(dst, &tmV, 0, y, half * 4, fb);
            }
          }
        }
        prev = cur;
        cur = nxt;
      }
      ++k;
    }
    if (!ok) *abort_flag = 1;
  } else if (warp == 1) {
    // -------------------------------------------------------- score-MMA issuer
    // Warp-uniform loop, one elected lane issues (as for the producer).  It
    // consumes the score stages of the ring and steps over the value stages,
    // which the value-MMA warp consumes.  S(x) overwrites the TMEM columns
    // that held P(x-2), so it first waits for PV(x-2) to complete.
    const bool leader = tc::elect_one();
    constexpr uint32_t idS = tc::idesc_bf16(128, kTile, false, false);
    // descriptors at offset 0; a K step adds (byte offset / 16)
    const uint64_t dQ = tc::sdesc(sQ, 16, 1024);
    const uint64_t dR = tc::sdesc(sR, 16, 1024);
    Ring rp;   // next stage in ring order
    int g = 0, k = 0;
    bool ok = true;
    SegIter it;
    it.init(&a, c, t);
    int sb, p0, p1, slot;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      if (!warp_wait(q_full, k & 1, a.status, 24)) { ok = false; break; }
      for (int i = 0; ok && i <= n; ++i) {
        if (i < n) {
          const int gs = g + i;
          if (gs >= 2 &&
              !warp_wait(pv_done + 6 * (gs & 1), ((gs - 2) >> 1) & 1, a.status, 33)) {
            ok = false;
            break;
          }
          // A new segment's first score stages follow the previous segment's
          // last value stages, which this warp stepped over: PV of that tile
          // must be done, or a slot could still be a lap behind.
          if (i == 0 && k > 0 &&
              !warp_wait(pv_done + 6 * ((gs - 1) & 1), ((gs - 1) >> 1) & 1, a.status, 35)) {
            ok = false;
            break;
          }
          const uint32_t dcol = tmem + kColS + (gs & 1) * kTile;
          for (int b = 0; b < 9; ++b, rp.next()) {
            const int s = rp.s;
            if (!warp_wait(&full[s], rp.ph, a.status, 23)) { ok = false; break; }
            tc::fence_after_sync();
            const uint64_t dRs = dR + ((s * kStage) >> 4);
            const uint64_t dQb = dQ + ((b * 16384) >> 4);
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc::mma_ss(dcol, dQb + kk * 2, dRs + kk * 2, idS, (b > 0 || kk > 0) ? 1u : 0u);
              tc::mma_commit(smem_u32(&empty[s]));
            }
          }
          if (!ok) break;
          if (leader) {
            tc::mma_commit(smem_u32(&s_full[gs & 1]));
            if (i == n - 1) tc::mma_commit(smem_u32(q_empty));
          }
        }
        if (i >= 1) rp.skip(nslabs_of(p0 + (i - 1) * kTile, p1));   // value stages of tile i-1
      }
      g += n;
      ++k;
    }
    if (!ok) *abort_flag = 1;
    if (leader) tc::mma_commit(smem_u32(drained));
  } else if (warp == 6) {
    // -------------------------------------------------------- value-MMA issuer
    // Steps over the score stages; for tile x waits for P(x) from the
    // softmax warps, then O += P(x) V(x) from the value slabs.
    const bool leader = tc::elect_one();
    constexpr uint32_t idO = tc::idesc_bf16(128, 256, false, true);
    const uint64_t dV = tc::sdesc(sR, 4096, 1024);   // value slab: MN-major
    Ring rp;
    int g = 0, k = 0;
    bool ok = true;
    SegIter it;
    it.init(&a, c, t);
    int sb, p0, p1, slot;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      for (int i = 0; ok && i <= n; ++i) {
        if (i < n) rp.skip(9);   // score stages of tile i
        if (i >= 1) {
          const int gv = g + i - 1;
          const int tv = p0 + (i - 1) * kTile;
          if (i == 1 && k > 0 && !warp_wait(o_free, (k - 1) & 1, a.status, 25)) { ok = false; break; }
          if (!warp_wait(p_full + 6 * (gv & 1), (gv >> 1) & 1, a.status, 26)) { ok = false; break; }
          // The value stages of tile x sit behind the score stages of tile
          // x+1 in the ring.  This warp steps over those without waiting, so
          // before waiting on its own slots it makes sure S(x+1) is done (all
          // its stages filled): otherwise a slot's barrier could still be a
          // whole lap behind, which a parity wait cannot tell apart.
          if (i < n && !warp_wait(&s_full[(gv + 1) & 1], ((gv + 1) >> 1) & 1, a.status, 34)) {
            ok = false;
            break;
          }
          if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t pcol = tmem + kColS + (gv & 1) * kTile;
          const int ns = nslabs_of(tv, p1);
          for (int v = 0; v < ns; ++v, rp.next()) {
            const int s = rp.s;
            if (!warp_wait(&full[s], rp.ph, a.status, 23)) { ok = false; break; }
            tc::fence_after_sync();
            const int vis = p1 - (tv + 32 * v);
            if (vis < 32) {
              zero_stale_rows<4>(smem + kOffRing + s * kStage, vis, lane);
              __syncwarp();
            }
            if (leader) {
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                // P tokens 32v+16kk.. live in columns (32v+16kk)/2.. of the S buffer
                tc::mma_ts(tmem, pcol + 16 * v + 8 * kk, dV + ((s * kStage + kk * 2048) >> 4),
                           idO, (i > 1 || v > 0 || kk > 0) ? 1u : 0u);
              }
              tc::mma_commit(smem_u32(&empty[s]));
            }
          }
          if (!ok) break;
          if (leader) tc::mma_commit(smem_u32(pv_done + 6 * (gv & 1)));
        }
      }
      g += n;
      ++k;
    }
    if (!ok) *abort_flag = 1;
    if (leader) tc::mma_commit(smem_u32(drained));
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ softmax warps
    softmax_role<false>(a, tmem, warp, lane, c, t, t, half, &s_full[0], &s_full[1], pv_done,
                        pv_done + 6, abort_flag,
                        [&](int g) { tc::mbar_arrive(smem_u32(p_full + 6 * (g & 1))); },
                        [&] { tc::mbar_arrive(smem_u32(o_free)); });
  }

  // ------------------------------------------------------------ teardown
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    for (int i = 0; i < kRing && i < issued; ++i) {
      const int u = issued - 1 - i;
      mbar_wait(&full[u % kRing], (u / kRing) & 1, a.status, 30, 1 << 20, 100000000ull);
    }
    if (q_issued > 0) mbar_wait(q_full, (q_issued - 1) & 1, a.status, 31, 1 << 20, 100000000ull);
  }
  __syncthreads();
  if (warp == 1) {
    // TMEM is freed only once both issuing threads' MMAs have completed
    mbar_wait(drained, 0, a.status, 32, 1 << 20, 100000000ull);
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool tc_attend(mla_ctx* ctx, const __nv_bfloat16* qimg, const __nv_bfloat16* cache,
               int num_pages, const int32_t* bt, int max_pages, int B, int T, char* ws,
               const WsLayout& L, cudaStream_t st) {
  CUtensorMap tmS, tmV;
  const uint64_t rows = (uint64_t)num_pages * kPage;
  if (!make_tmap_bf16_2d(&tmS, cache, rows, kRow, kRow, 64, 64, false) ||
      !make_tmap_pool_blocks(&tmV, cache, rows, 32, 4))
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
  if (smem_attr_once(attr_done, attend_tc_kernel, (int)kSmem) != cudaSuccess) return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.G, T, 2);
  cfg.blockDim = dim3(224);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_mark(ctx, st, "attend");
  ctx->launches += 1;
  return cudaLaunchKernelEx(&cfg, attend_tc_kernel, tmS, tmV, a) == cudaSuccess;
}

}  // namespace mla
