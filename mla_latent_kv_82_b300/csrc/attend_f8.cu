// Decode attention over the FP8 latent cache, and the quantisation that
// fills it.
//
// FP8 cache row (656 bytes, the format stated with MLA_KV_FP8 in mla.h):
// 512 E4M3 codes of c^KV, 64 bf16 values of k^R / s, the row scale s (fp32)
// and zero padding; the row stands for [s * E4M3(code) ; s * stored].
//
// Scores: the absorbed form of page "DeepSeek-V2：在“大力出奇迹”的AI军备竞赛
// 中，四两拨千斤" (liang.world, 第二章 §2-§3) with the attention GEMM on FP8
// operands, as the forward pass of page "DeepSeek 系列模型技术深度解读"
// (tuntang.top, "FP8 混合精度训练") runs its attention GEMMs.  f8_prepare
// quantises each head's absorbed query q~ (512 values) to E4M3 with its own
// scale sq = amax / 448 and stores the rotated RoPE query divided by sq.
// With a row's codes c8 and its stored k^R / s one accumulator holds
//     D = q8 . c8 + (q^R / sq) . (k^R / s),      score = sq * s * D,
// the first term on tcgen05 kind::f8f6f4 (E4M3 x E4M3), the second on
// kind::f16 (bf16).
// Values: O += P' V with V = the rows' E4M3 codes widened to bf16 (exact)
// and P' = p * s in bf16, so that O = sum over keys of p * s * E4M3(code).
//
// One CTA per (KV split, query token, latent half of 256 columns); both
// halves compute the same S (E4M3 score MMAs take half the time of bf16
// ones), so their softmax statistics agree bit for bit.
// TMEM: this half's O at columns 0..255, two S buffers at 256 and 384; P'
// overwrites its S buffer and feeds the value MMA from TMEM.
// Shared memory: the FP8 query image (82432 B), a ring of four 16 KB stages
// (per tile: four latent blocks [128 keys][128 codes], then the RoPE block
// [128 keys][64 bf16]), two buffers of a tile's row scales, and this half's
// values of the tile widened to bf16 (64 KB).
// Roles (256 threads): warp 0 TMA producer; warp 1 score-MMA issuer and
// TMEM owner; warps 2-5 softmax and epilogue (thread = head); warps 6-7 load
// this half's codes of each tile straight from the pool into registers (a
// tile ahead), widen them into the value buffer once the previous PV has
// read it, and issue the tile's value MMAs.
// Every wait is bounded; on a timeout the CTA records MLA_ERR_TIMEOUT,
// drains its own copies and frees TMEM.
#include "attend_common.cuh"
#include "launch_util.h"
#include "tmap.h"

namespace mla {
namespace {

using namespace att;

constexpr int kF8Ring = 4;
constexpr uint32_t kF8Stage = 16384;
constexpr uint32_t kOffQ8 = 0;                                   // FP8 query image
constexpr uint32_t kQ8Rope = 65536;                              // its RoPE block
constexpr uint32_t kQ8Scale = 81920;                             // its head scales
constexpr uint32_t kOffRing8 = 83968;
constexpr uint32_t kSclBytes = kTile * 16;                       // [128 keys][16 B]
constexpr uint32_t kOffScl = kOffRing8 + kF8Ring * kF8Stage;     // 149504
constexpr uint32_t kOffV8 = kOffScl + 2 * kSclBytes;             // 153600
constexpr uint32_t kOffBar8 = kOffV8 + 4 * 16384;                // 219136
constexpr uint32_t kF8Smem = kOffBar8 + 256 + 1024;
constexpr int kF8Threads = 256;
static_assert(kOffRing8 % 1024 == 0 && kOffV8 % 1024 == 0, "swizzled operands");
static_assert(kQ8Scale + 4 * kHeads == (uint32_t)kQ8Bytes, "query image size");

// barriers (uint64 each)
enum : int {
  kF = 0,     // [4] ring stage loaded
  kE = 4,     // [4] ring stage consumed (MMA commit)
  kSF = 8,    // [2] S of tiles of that parity done
  kPF = 10,   // [2] P' written (4 softmax warps)
  kPD = 12,   // [2] PV of tiles of that parity done
  // 14, 15 unused
  kCF = 16,   // [2] row scales of the tile loaded
  kCE = 18,   // [2] row scales read (4 softmax warps)
  kQF = 20,   // query image loaded
  kQE = 21,   // query image consumed: last S commit + 4 softmax warps (scales read)
  kOF = 22,   // epilogue read O (4 softmax warps)
  kDR = 23,   // the last score MMAs and the last value MMAs done
  kSlot = 24  // tmem slot, abort flag, converter failure flag
};

// Two E4M3 codes at bits 0..7 and 16..23 -> bf16x2 of their values.  The
// code's exponent and mantissa bits land in the bf16 exponent and mantissa
// fields as they are, which gives value * 2^-120 (subnormal codes included),
// then one exact multiply by 2^120.
__device__ __forceinline__ uint32_t e4m3x2_bf16x2(uint32_t t) {
  const uint32_t h = ((t << 4) & 0x07F007F0u) | ((t << 8) & 0x80008000u);
  const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&h);
  const __nv_bfloat16 k = __ushort_as_bfloat16((unsigned short)0x7B80);   // 2^120
  const __nv_bfloat162 r = __hmul2(v, __nv_bfloat162(k, k));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// p = 2^(x * a - m) for keys below `valid` (0 beyond) with x = D * s; P' =
// p * s packed as bf16 two per word (keys 2j low, 2j+1 high); returns the
// sum of p.
template <bool kMask>
__device__ __forceinline__ float exp_pack_f8(const uint32_t (&lo)[64], const uint32_t (&hi)[64],
                                             int valid, float a, float m, const float* scl,
                                             uint32_t (&pk)[64]) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const int t0 = 2 * j, t1 = 2 * j + 1;
    const float x0 = __uint_as_float(t0 < 64 ? lo[t0] : hi[t0 - 64]);
    const float x1 = __uint_as_float(t1 < 64 ? lo[t1] : hi[t1 - 64]);
    const float e0 = (!kMask || t0 < valid) ? tc::ex2_approx(fmaf(x0, a, -m)) : 0.f;
    const float e1 = (!kMask || t1 < valid) ? tc::ex2_approx(fmaf(x1, a, -m)) : 0.f;
    s0 += e0;
    s1 += e1;
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(e0 * scl[t0 * 4], e1 * scl[t1 * 4]);
    pk[j] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  return s0 + s1;
}

__global__ void __launch_bounds__(kF8Threads, 1)
attend_f8_kernel(const __grid_constant__ CUtensorMap tmB,   // pool, box {128 B, 64 rows}, SW128
                 const __grid_constant__ CUtensorMap tmC,   // pool, box {16 B, 64 rows}
                 const AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + kSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* conv_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, t = blockIdx.y, half = blockIdx.z;
  const int vb0 = 2 * half;   // this half's latent blocks: vb0, vb0 + 1

  tc::grid_dep_launch();
  tc::grid_dep_wait();   // plan, query images and the pool come from earlier kernels
  if (c >= a.meta[0]) return;   // more CTAs than KV splits in use

  if (threadIdx.x == 0) {
    for (int i = 0; i < kF8Ring; ++i) {
      mbar_init(&bar[kF + i], 1);
      mbar_init(&bar[kE + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar[kSF + i], 1);
      mbar_init(&bar[kPF + i], 4);
      mbar_init(&bar[kPD + i], 1);
      mbar_init(&bar[kCF + i], 1);
      mbar_init(&bar[kCE + i], 4);
    }
    mbar_init(&bar[kQF], 1);
    mbar_init(&bar[kQE], 5);
    mbar_init(&bar[kOF], 4);
    mbar_init(&bar[kDR], 2);
    *abort_flag = 0;
    *conv_fail = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmB);
    tc::prefetch_tmap(&tmC);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sQ = smem_u32(smem + kOffQ8);
  const uint32_t sR = smem_u32(smem + kOffRing8);
  const int oob_row = a.num_pages * kPage + kPage;   // TMA zero-fills rows out of range
  int issued = 0, q_issued = 0, c_issued = 0;        // producer: copies in flight

  if (warp == 0) {
    // -------------------------------------------------------------- producer
    // Per segment the query image, then per tile its row scales and the five
    // ring stages (latent blocks 0..3, RoPE block), in the MMA issuer's order.
    const bool leader = tc::elect_one();
    SegIter it;
    it.init(&a, c, t);
    int sb, p0, p1, slot, k = 0, g = 0;
    bool ok = true;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      if (k > 0 && !warp_wait(&bar[kQE], (k - 1) & 1, a.status, 121)) { ok = false; break; }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
      ++q_issued;
      if (leader) {
        const uint32_t qb = smem_u32(&bar[kQF]);
        tc::mbar_arrive_expect_tx(qb, kQ8Bytes);
        const uint8_t* src = a.qimg + ((size_t)sb * a.T + t) * kQ8Bytes;
        for (uint32_t o = 0; o < (uint32_t)kQ8Bytes; o += 16384)
          tc::bulk_load(sQ + o, src + o, min(16384u, (uint32_t)kQ8Bytes - o), qb);
      }
      for (int i = 0; ok && i < n; ++i, ++g) {
        TilePages tp;
        tp.load(a, sb, p0 + i * kTile, p1);
        const int y0 = tp.row(a, 0, sb, oob_row), y1 = tp.row(a, 1, sb, oob_row);
        if (g >= 2 && !warp_wait(&bar[kCE + (g & 1)], ((g >> 1) - 1) & 1, a.status, 122)) {
          ok = false;
          break;
        }
        c_issued = g + 1;
        if (leader) {
          const uint32_t cb = smem_u32(&bar[kCF + (g & 1)]);
          const uint32_t dst = smem_u32(smem + kOffScl + (g & 1) * kSclBytes);
          tc::mbar_arrive_expect_tx(cb, kSclBytes);
          tc::tma_load_2d(dst, &tmC, 640, y0, cb);
          tc::tma_load_2d(dst + kSclBytes / 2, &tmC, 640, y1, cb);
        }
        for (int kb = 0; kb < 5; ++kb) {
          const int nr = 5 * g + kb, s = nr % kF8Ring;
          if (nr >= kF8Ring &&
              !warp_wait(&bar[kE + s], ((nr / kF8Ring) & 1) ^ 1u, a.status, 123)) {
            ok = false;
            break;
          }
          if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
          issued = nr + 1;
          if (leader) {
            const uint32_t fb = smem_u32(&bar[kF + s]);
            const uint32_t dst = sR + s * kF8Stage;
            tc::mbar_arrive_expect_tx(fb, kF8Stage);
            tc::tma_load_2d(dst, &tmB, kb * 128, y0, fb);
            tc::tma_load_2d(dst + 8192, &tmB, kb * 128, y1, fb);
          }
        }
      }
      ++k;
    }
    if (!ok) *abort_flag = 1;
  } else if (warp == 1) {
    // ---------------------------------------------------------- score MMA issuer
    // Per tile S(g) on the four latent blocks and the RoPE block; the value
    // MMAs are issued by the converters once they have filled the value
    // buffer, so that neither waits behind the other.
    const bool leader = tc::elect_one();
    constexpr uint32_t idS8 = tc::idesc_e4m3(128, kTile);
    constexpr uint32_t idSR = tc::idesc_bf16(128, kTile, false, false);
    const uint64_t dQ = tc::sdesc(sQ, 16, 1024);
    const uint64_t dR = tc::sdesc(sR, 16, 1024);
    SegIter it;
    it.init(&a, c, t);
    int sb, p0, p1, slot, k = 0, g = 0;
    bool ok = true;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      if (n == 0) continue;
      if (!warp_wait(&bar[kQF], k & 1, a.status, 124)) { ok = false; break; }
      for (int i = 0; ok && i < n; ++i, ++g) {
        // S(g) reuses the columns P(g - 2) was read from
        if (g >= 2 && !warp_wait(&bar[kPD + (g & 1)], ((g - 2) >> 1) & 1, a.status, 125)) {
          ok = false;
          break;
        }
        const uint32_t dcol = tmem + kColS + (g & 1) * kTile;
        for (int kb = 0; kb < 5; ++kb) {
          const int nr = 5 * g + kb, s = nr % kF8Ring;
          if (!warp_wait(&bar[kF + s], (nr / kF8Ring) & 1, a.status, 126)) { ok = false; break; }
          tc::fence_after_sync();
          if (leader) {
            const uint64_t b = dR + ((s * kF8Stage) >> 4);
            if (kb < 4) {
              const uint64_t q = dQ + ((kb * 16384) >> 4);
              tc::mma_ss_f8(dcol, q, b, idS8, kb > 0 ? 1u : 0u);
              tc::mma_ss_f8(dcol, q + 2, b + 2, idS8, 1u);
              tc::mma_ss_f8(dcol, q + 4, b + 4, idS8, 1u);
              tc::mma_ss_f8(dcol, q + 6, b + 6, idS8, 1u);
            } else {
              const uint64_t q = dQ + (kQ8Rope >> 4);
              tc::mma_ss(dcol, q, b, idSR, 1u);
              tc::mma_ss(dcol, q + 2, b + 2, idSR, 1u);
              tc::mma_ss(dcol, q + 4, b + 4, idSR, 1u);
              tc::mma_ss(dcol, q + 6, b + 6, idSR, 1u);
            }
            tc::mma_commit(smem_u32(&bar[kE + s]));
          }
        }
        if (!ok) break;
        if (leader) {
          tc::mma_commit(smem_u32(&bar[kSF + (g & 1)]));
          if (i == n - 1) tc::mma_commit(smem_u32(&bar[kQE]));
        }
      }
      ++k;
    }
    if (!ok) *abort_flag = 1;
    if (leader) tc::mma_commit(smem_u32(&bar[kDR]));
  } else if (warp >= 6) {
    // ---------------------------------------------------------- converters
    // Tile g's codes of this half (latent blocks vb0, vb0 + 1: 256 bytes of
    // each key's row) come straight from the pool into registers, 32
    // 16-byte pieces per thread; once PV(g - 1) has read the value buffer
    // they are widened to bf16 into it ([128 keys][256 columns] as four
    // 128-byte-swizzled blocks of 64 columns), and each register is refilled
    // with the next tile's piece as soon as it is widened, so that a tile's
    // loads are in flight while the previous tile is consumed.  Keys past
    // the visible end become zeros, so that 0 * (NaN or Inf) never reaches
    // the accumulator.
    const int ct = threadIdx.x - 192;   // 0..63
    const uint8_t* pool = reinterpret_cast<const uint8_t*>(a.cache);
    // tile walk: the (sequence, first key, visible end) of each tile
    SegIter it;
    it.init(&a, c, t);
    int sb = 0, p0 = 0, p1 = 0, slot = 0, i = 0, n = 0;
    auto next_tile = [&](int* tsb, int* tts, int* tp1, bool* tfirst) -> bool {
      while (i >= n) {
        if (!it.next(&sb, &p0, &p1, &slot)) return false;
        n = ntiles_of(p0, p1);
        i = 0;
      }
      *tsb = sb;
      *tts = p0 + i * kTile;
      *tp1 = p1;
      *tfirst = i == 0;
      ++i;
      return true;
    };
    uint4 wv[32];
    // issue the loads of one tile (zeros past its visible end)
    auto load_tile = [&](int lsb, int lts, int lp1) {
      TilePages tp;
      tp.load(a, lsb, lts, lp1);
      const int y0 = tp.row(a, 0, lsb, oob_row), y1 = tp.row(a, 1, lsb, oob_row);
      const int vis = min(kTile, lp1 - lts);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int task = ct + 64 * j;
        const int kl = task >> 10, r = (task >> 3) & 127, ch = task & 7;
        wv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (r < vis)
          wv[j] = tc::ld_nc_v4(pool + (size_t)((r < kPage ? y0 : y1 - kPage) + r) * kF8Row +
                               (vb0 + kl) * 128 + ch * 16);
      }
    };
    int csb, cts, cp1;
    bool cfirst;
    bool have = next_tile(&csb, &cts, &cp1, &cfirst);
    if (have) load_tile(csb, cts, cp1);
    bool ok = true;
    uint8_t* vbuf = smem + kOffV8;
    constexpr uint32_t idO = tc::idesc_bf16(128, 256, false, true);
    const uint64_t dV = tc::sdesc(smem_u32(vbuf), 16384, 1024);   // MN-major values
    int kseg = -1;   // segment of the current tile (segments with tiles only)
    for (int g = 0; have; ++g) {
      if (cfirst) ++kseg;
      int nsb, nts, np1;
      bool nfirst = false;
      const bool more = next_tile(&nsb, &nts, &np1, &nfirst);
      bool w = true;
      if (g >= 1)
        w = bar_wait<false>(&bar[kPD + ((g - 1) & 1)], ((g - 1) >> 1) & 1, a.status, 130);
      if (!w || *abort_flag) *conv_fail = 1;
      tc::named_sync(2, 64);
      if (*conv_fail) { ok = false; break; }   // read after the barrier: the same for all
      // the next tile's rows, validated as the producer validates them
      int ny0 = 0, ny1 = 0, nvis = 0;
      if (more) {
        TilePages tp;
        tp.load(a, nsb, nts, np1);
        ny0 = tp.row(a, 0, nsb, oob_row);
        ny1 = tp.row(a, 1, nsb, oob_row);
        nvis = min(kTile, np1 - nts);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int task = ct + 64 * j;
        const int kl = task >> 10, r = (task >> 3) & 127, ch = task & 7;
        uint4 lo, hi;
        lo.x = e4m3x2_bf16x2(__byte_perm(wv[j].x, 0u, 0x4140));
        lo.y = e4m3x2_bf16x2(__byte_perm(wv[j].x, 0u, 0x4342));
        lo.z = e4m3x2_bf16x2(__byte_perm(wv[j].y, 0u, 0x4140));
        lo.w = e4m3x2_bf16x2(__byte_perm(wv[j].y, 0u, 0x4342));
        hi.x = e4m3x2_bf16x2(__byte_perm(wv[j].z, 0u, 0x4140));
        hi.y = e4m3x2_bf16x2(__byte_perm(wv[j].z, 0u, 0x4342));
        hi.z = e4m3x2_bf16x2(__byte_perm(wv[j].w, 0u, 0x4140));
        hi.w = e4m3x2_bf16x2(__byte_perm(wv[j].w, 0u, 0x4342));
        const int col = kl * 128 + ch * 16;           // column within this half
        const int vb = col >> 6, cc = (col & 63) >> 3;
        uint8_t* dst = vbuf + vb * 16384 + r * 128;
        *reinterpret_cast<uint4*>(dst + ((cc ^ (r & 7)) << 4)) = lo;
        *reinterpret_cast<uint4*>(dst + (((cc + 1) ^ (r & 7)) << 4)) = hi;
        // refill with the next tile's piece
        wv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (more && r < nvis)
          wv[j] = tc::ld_nc_v4(pool + (size_t)((r < kPage ? ny0 : ny1 - kPage) + r) * kF8Row +
                               (vb0 + kl) * 128 + ch * 16);
      }
      tc::fence_async_smem();
      tc::named_sync(2, 64);
      if (ct == 0) {
        // O += P'(g) V(g); a segment's first PV overwrites O once the
        // previous segment's epilogue has read it
        bool w2 = true;
        if (cfirst && kseg > 0) w2 = mbar_wait(&bar[kOF], (kseg - 1) & 1, a.status, 127);
        w2 = w2 && mbar_wait(&bar[kPF + (g & 1)], (g >> 1) & 1, a.status, 128);
        if (w2) {
          tc::fence_after_sync();
          const uint32_t pcol = tmem + kColS + (g & 1) * kTile;
          tc::mma_ts(tmem, pcol, dV, idO, cfirst ? 0u : 1u);
          tc::mma_ts(tmem, pcol + 8, dV + (2048 >> 4), idO, 1u);
          tc::mma_ts(tmem, pcol + 16, dV + (4096 >> 4), idO, 1u);
          tc::mma_ts(tmem, pcol + 24, dV + (6144 >> 4), idO, 1u);
          tc::mma_ts(tmem, pcol + 32, dV + (8192 >> 4), idO, 1u);
          tc::mma_ts(tmem, pcol + 40, dV + (10240 >> 4), idO, 1u);
          tc::mma_ts(tmem, pcol + 48, dV + (12288 >> 4), idO, 1u);
          tc::mma_ts(tmem, pcol + 56, dV + (14336 >> 4), idO, 1u);
          tc::mma_commit(smem_u32(&bar[kPD + (g & 1)]));
        } else {
          *conv_fail = 1;
        }
      }
      have = more;
      cfirst = nfirst;
    }
    if (!ok) *abort_flag = 1;
    if (ct == 0) tc::mma_commit(smem_u32(&bar[kDR]));   // the value MMAs' completion
  } else {
    // ------------------------------------------------------------ softmax
    // thread = head; x = D * s per key, logits x * sq * scale (log2 domain),
    // lazy rescale as in the bf16 kernels (O and l rescaled only when the
    // maximum grows by more than 2^kRescale, so p <= 256).
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    SegIter it;
    it.init(&a, c, t);
    int sb, p0, p1, slot, g = 0, k = 0;
    bool ok = true;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      const size_t st_idx = (size_t)slot * a.T + t;   // (slot, token) of the split result
      const size_t prow = st_idx * kHeads + row;
      // one split holds the whole sequence: write o_lat here, no combine
      const bool direct = a.slot_base[sb + 1] - a.slot_base[sb] == 1;
      __nv_bfloat16* olat =
          a.o_lat + (((size_t)sb * a.T + t) * kHeads + row) * kLat + half * 256;
      float* dst = a.part_o + part_off(st_idx, row, half * 256);   // chunk j at + j * 128
      if (n == 0) {
        const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        for (int j = 0; j < 256; j += 8) {
          if (direct) *reinterpret_cast<uint4*>(olat + j) = make_uint4(0u, 0u, 0u, 0u);
          else st_v8(dst + (size_t)(j >> 3) * 128, z);
        }
        if (!direct && half == 0) a.part_lse[prow] = -INFINITY;
        continue;
      }
      ok = bar_wait<false>(&bar[kQF], k & 1, a.status, 132);
      if (__any_sync(0xffffffffu, !ok || *abort_flag)) { ok = false; break; }
      const float ah =
          a.scale_log2 * *reinterpret_cast<const float*>(smem + kOffQ8 + kQ8Scale + row * 4);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(smem_u32(&bar[kQE]));
      float m_used = -INFINITY, l = 0.f;
      for (int i = 0; i < n; ++i, ++g) {
        const uint32_t scol = trow + kColS + (g & 1) * kTile;
        ok = bar_wait<false>(&bar[kSF + (g & 1)], (g >> 1) & 1, a.status, 133);
        ok = ok && bar_wait<false>(&bar[kCF + (g & 1)], (g >> 1) & 1, a.status, 134);
        if (__any_sync(0xffffffffu, !ok || *abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        const int valid = max(0, min(kTile, p1 - (p0 + i * kTile)));
        uint32_t lo[64], hi[64];
        tc::tmem_ld64(scol, lo);
        tc::tmem_ld64(scol + 64, hi);
        const float* scl = reinterpret_cast<const float*>(smem + kOffScl + (g & 1) * kSclBytes);
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          lo[j] = __float_as_uint(__uint_as_float(lo[j]) * scl[j * 4]);
          hi[j] = __float_as_uint(__uint_as_float(hi[j]) * scl[(64 + j) * 4]);
        }
        const float mx =
            (valid == kTile ? row_max<false>(lo, hi, valid) : row_max<true>(lo, hi, valid)) * ah;
        const bool need = mx > m_used + kRescale;
        if (i == 0) {
          m_used = mx;
        } else if (__any_sync(0xffffffffu, need)) {
          // O holds PV of the segment's earlier tiles: rescale once PV(g - 1) is done
          ok = bar_wait<false>(&bar[kPD + ((g - 1) & 1)], ((g - 1) >> 1) & 1, a.status, 135);
          if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
          tc::fence_after_sync();
          const float m_new = need ? mx : m_used;
          const float f = exp2f(m_used - m_new);
          l *= f;
          for (int c0 = 0; c0 < 256; c0 += 16) {
            float v[16];
            tc::tmem_ld16(trow + c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] *= f;
            tc::tmem_st16(trow + c0, v);
          }
          m_used = m_new;
        }
        uint32_t pk[64];
        const float psum = valid == kTile
                               ? exp_pack_f8<false>(lo, hi, valid, ah, m_used, scl, pk)
                               : exp_pack_f8<true>(lo, hi, valid, ah, m_used, scl, pk);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(smem_u32(&bar[kCE + (g & 1)]));
        tc::tmem_st64(scol, pk);
        l += psum;
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(smem_u32(&bar[kPF + (g & 1)]));
      }
      if (!ok) break;
      // segment epilogue: O / l (and the log-sum-exp for the combine)
      ok = bar_wait<false>(&bar[kPD + ((g - 1) & 1)], ((g - 1) >> 1) & 1, a.status, 136);
      if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      for (int c0 = 0; c0 < 256; c0 += 16) {
        float v[16];
        tc::tmem_ld16(trow + c0, v);
        if (direct) {
          uint32_t w[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * j] * inv, v[2 * j + 1] * inv);
            w[j] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(olat + c0) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(olat + c0 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; j += 8) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(v[j + e] * inv);
            st_v8(dst + (size_t)((c0 + j) >> 3) * 128, w);
          }
        }
      }
      if (!direct && half == 0) a.part_lse[prow] = l > 0.f ? m_used + log2f(l) : -INFINITY;
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(smem_u32(&bar[kOF]));
      ++k;
    }
    if (!ok) *abort_flag = 1;
  }

  // ------------------------------------------------------------ teardown
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    // drain this CTA's own copies still in flight
    for (int i = 0; i < kF8Ring && i < issued; ++i) {
      const int u = issued - 1 - i;
      mbar_wait(&bar[kF + u % kF8Ring], (u / kF8Ring) & 1, a.status, 137, 1 << 20, 100000000ull);
    }
    for (int i = 0; i < 2 && i < c_issued; ++i) {
      const int u = c_issued - 1 - i;
      mbar_wait(&bar[kCF + (u & 1)], (u >> 1) & 1, a.status, 138, 1 << 20, 100000000ull);
    }
    if (q_issued > 0)
      mbar_wait(&bar[kQF], (q_issued - 1) & 1, a.status, 139, 1 << 20, 100000000ull);
  }
  __syncthreads();
  if (warp == 1) {
    mbar_wait(&bar[kDR], 0, a.status, 140, 1 << 20, 100000000ull);
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- quantise
// Warps [0, rows): staged bf16 row t (token m0 + t of the batch) -> its FP8
// pool row.  Warps [rows, rows + M_q * 128): the bf16 query image of
// (token, head) -> the FP8 query image (E4M3 codes of q~ with the head's
// scale, q^R / sq in bf16, sq), laid out as attend_f8_kernel keeps it.
__device__ __forceinline__ void unpack8(const uint4& u, float* x) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// E4M3 codes of x[0..15] * inv (each product rounded to fp32, then to the
// nearest E4M3 value, ties to even, saturating), in order.
__device__ __forceinline__ uint4 encode16(const float* x, float inv) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint16_t lo, hi;
    const float a0 = __fmul_rn(x[4 * i], inv), a1 = __fmul_rn(x[4 * i + 1], inv);
    const float a2 = __fmul_rn(x[4 * i + 2], inv), a3 = __fmul_rn(x[4 * i + 3], inv);
    // the first source lands in the upper byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(a1), "f"(a0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(a3), "f"(a2));
    w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float warp_amax(const float* x, int n) {
  float m = 0.f;
  for (int i = 0; i < n; ++i) m = fmaxf(m, fabsf(x[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

__global__ void __launch_bounds__(256)
f8_prepare_kernel(const __nv_bfloat16* __restrict__ stage, int rows, int m0,
                  const int32_t* __restrict__ pos, const int32_t* __restrict__ bt, int T,
                  int max_pages, int max_position, int num_pages, uint8_t* __restrict__ cache8,
                  const uint8_t* __restrict__ qimg, int M_q, uint8_t* __restrict__ q8,
                  int* status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid < rows) {
    const int r = (int)wid, m = m0 + r;
    const int p = pos[m];
    const int b = m / T, lp = p / kPage;
    if (p < 0 || p >= max_position || lp >= max_pages) {
      if (lane == 0) report(status, MLA_ERR_DEVICE_INDEX, 2000000 + m);
      return;
    }
    const int pg = bt[(size_t)b * max_pages + lp];
    if (pg < 0 || pg >= num_pages) {
      if (lane == 0) report(status, MLA_ERR_DEVICE_INDEX, 3000000 + m);
      return;
    }
    const __nv_bfloat16* src = stage + (size_t)r * kRow;
    float x[16];
    unpack8(*reinterpret_cast<const uint4*>(src + lane * 16), x);
    unpack8(*reinterpret_cast<const uint4*>(src + lane * 16 + 8), x + 8);
    const float amax = warp_amax(x, 16);
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
    uint8_t* dst = cache8 + ((size_t)pg * kPage + p % kPage) * kF8Row;
    *reinterpret_cast<uint4*>(dst + lane * 16) = encode16(x, inv);
    if (lane < 8) {
      float kr[8];
      unpack8(*reinterpret_cast<const uint4*>(src + kLat + lane * 8), kr);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h2 =
            __floats2bfloat162_rn(__fdiv_rn(kr[2 * i], sc), __fdiv_rn(kr[2 * i + 1], sc));
        w[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(dst + kLat + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if (lane == 8) {
      *reinterpret_cast<uint4*>(dst + 640) = make_uint4(__float_as_uint(sc), 0u, 0u, 0u);
    }
    return;
  }
  const long long w = wid - rows;
  if (w >= (long long)M_q * kHeads) return;
  const int m = (int)(w / kHeads), h = (int)(w % kHeads);
  const uint8_t* img = qimg + (size_t)m * kQImgBytes;
  float x[16];
  unpack8(*reinterpret_cast<const uint4*>(img + qimg_off(h, lane * 16)), x);
  unpack8(*reinterpret_cast<const uint4*>(img + qimg_off(h, lane * 16 + 8)), x + 8);
  const float amax = warp_amax(x, 16);
  const float sq = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 1.f;
  uint8_t* out = q8 + (size_t)m * kQ8Bytes;
  const int kb = lane >> 3, ch = lane & 7;
  *reinterpret_cast<uint4*>(out + kb * 16384 + h * 128 + ((ch ^ (h & 7)) << 4)) = encode16(x, inv);
  if (lane < 8) {
    float qr[8];
    unpack8(*reinterpret_cast<const uint4*>(img + qimg_off(h, kLat + lane * 8)), qr);
    uint32_t wq[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h2 =
          __floats2bfloat162_rn(__fdiv_rn(qr[2 * i], sq), __fdiv_rn(qr[2 * i + 1], sq));
      wq[i] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(out + kQ8Rope + h * 128 + ((lane ^ (h & 7)) << 4)) =
        make_uint4(wq[0], wq[1], wq[2], wq[3]);
  } else if (lane == 8) {
    *reinterpret_cast<float*>(out + kQ8Scale + h * 4) = sq;
  }
}

}  // namespace

bool f8_prepare(mla_ctx* ctx, const __nv_bfloat16* stage, int rows, int m0, const int32_t* pos,
                const int32_t* bt, int T, int max_pages, uint8_t* cache8, int num_pages,
                const __nv_bfloat16* qimg, int M_q, uint8_t* q8img, cudaStream_t st) {
  const long long warps = (long long)rows + (long long)M_q * kHeads;
  if (warps == 0) return true;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((warps + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_mark(ctx, st, "f8_prepare");
  ctx->launches += 1;
  return cudaLaunchKernelEx(&cfg, f8_prepare_kernel, stage, rows, m0, pos, bt, T, max_pages,
                            ctx->cfg.max_position, num_pages, cache8,
                            reinterpret_cast<const uint8_t*>(qimg), M_q, q8img,
                            ctx->status) == cudaSuccess;
}

bool f8_attend(mla_ctx* ctx, const uint8_t* q8img, const uint8_t* cache8, int num_pages,
               const int32_t* bt, int max_pages, int B, int T, char* ws, const WsLayout& L,
               cudaStream_t st) {
  CUtensorMap tmB, tmC;
  const uint64_t rows = (uint64_t)num_pages * kPage;
  if (!make_tmap_u8_2d(&tmB, cache8, rows, kF8Row, 128, 64, true) ||
      !make_tmap_u8_2d(&tmC, cache8, rows, kF8Row, 16, 64, false)) {
    cudaGetLastError();
    return false;
  }
  AttArgs a{};
  a.lens = reinterpret_cast<const int*>(ws + L.lens);
  a.prefix = reinterpret_cast<const int*>(ws + L.page_prefix);
  a.first_split = reinterpret_cast<const int*>(ws + L.first_split);
  a.slot_base = reinterpret_cast<const int*>(ws + L.slot_base);
  a.meta = reinterpret_cast<const int*>(ws + L.meta);
  a.bt = bt;
  a.qimg = q8img;
  a.cache = reinterpret_cast<const __nv_bfloat16*>(cache8);   // read as bytes by the converters
  a.part_o = reinterpret_cast<float*>(ws + L.part_o);
  a.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  a.o_lat = reinterpret_cast<__nv_bfloat16*>(ws + L.o_lat);
  a.status = ctx->status;
  a.B = B;
  a.T = T;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.scale_log2 = ctx->cfg.softmax_scale * 1.4426950408889634f;
  static std::atomic<uint64_t> attr_done{0};
  if (smem_attr_once(attr_done, attend_f8_kernel, (int)kF8Smem) != cudaSuccess) return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.G, T, 2);
  cfg.blockDim = dim3(kF8Threads);
  cfg.dynamicSmemBytes = kF8Smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_mark(ctx, st, "attend");
  ctx->launches += 1;
  return cudaLaunchKernelEx(&cfg, attend_f8_kernel, tmB, tmC, a) == cudaSuccess;
}

}  // namespace mla
