// Split-KV flash-decoding over the bf16 latent cache on tcgen05 tensor cores.
//
// Absorbed MLA attention (page "DeepSeek-V2：在“大力出奇迹”的AI军备竞赛中，
// 四两拨千斤", liang.world, 第二章 §2 absorption and §3 decoupled RoPE): with
// the query image Q = [W^UK_i^T q^C_i ; RoPE(q^R_i)] (128 heads x 576) and
// the cached rows C = [c^KV ; k^R] (tokens x 576),
//     s = Q C^T * scale,  a = softmax(s),  o_lat = a C[:, :512].
// The 128 heads are the M = 128 side of both MMAs:
//     S  (128 x 32 tokens)  = Q (128 x 576) . C_tile^T        -> TMEM, fp32
//     O  (128 x 256 cols)  += P (128 x 32, bf16) . C_tile[:, half]
// One CTA owns one KV split of one query token and one half (256 columns)
// of the latent output; the two halves recompute the same S (so their
// softmax statistics agree bit for bit) and keep their O half resident in
// TMEM (256 + 2 x 32 of the 512 columns).
//
// Roles (192 threads): warp 0 = TMA producer (query image by bulk copy once
// per segment, 32-token cache tiles by tiled TMA into two 128B-swizzled
// stages), warp 1 = MMA issuer + TMEM owner, warps 2-5 = softmax (thread =
// head): online softmax in the log2 domain with a lazy rescale (O and l are
// rescaled only when a row maximum grows by more than 2^8, so P <= 256),
// P written to shared memory in the 64-byte swizzled K-major layout.  At the
// end of a segment the same warps write O / l and m + log2 l for the
// log-sum-exp combine.  Every wait is bounded; on a timeout the CTA records
// MLA_ERR_TIMEOUT, drains its own loads and frees TMEM.
#include "layouts.cuh"
#include "tc_util.cuh"
#include "mla_internal.h"
#include "tmap.h"

namespace mla {
namespace {

constexpr int kTok = 32;                                   // tokens per tile
constexpr uint32_t kTileBlock = kTok * 128;                // one 64-feature box
constexpr uint32_t kTileBytes = 9 * kTileBlock;            // 36864
constexpr uint32_t kPBytes = 128 * kTok * 2;               // 8192
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffTile = kQImgBytes;                  // 147456
constexpr uint32_t kOffP = kOffTile + 2 * kTileBytes;      // 221184
constexpr uint32_t kOffBar = kOffP + kPBytes;              // 229376
constexpr uint32_t kSmem = kOffBar + 256 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 256;                            // S buffers at 256, 288
constexpr float kRescale = 8.0f;                           // log2 units

struct AttArgs {
  const int* lens;
  const int* prefix;
  const int* first_split;
  const int* slot_base;
  const int* meta;
  const int32_t* bt;
  const uint8_t* qimg;
  float* part_o;
  float* part_lse;
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
  return p1 > p0 ? (p1 - p0 + kTok - 1) / kTok : 0;
}

__device__ __forceinline__ uint32_t p_off(int r, int chunk) {
  // 64-byte swizzle: 8-row x 64 B atoms, chunk j of row r at j ^ ((r % 8) >> 1)
  return (uint32_t)((r >> 3) * 512 + (r & 7) * 64 + ((chunk ^ ((r & 7) >> 1)) << 4));
}

__device__ __forceinline__ uint64_t sdesc64(uint32_t saddr, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                       // leading byte offset (unused): 16 B
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;                       // swizzle mode: 64-byte
  return d;
}

__global__ void __launch_bounds__(192, 1)
attend_tc_kernel(const __grid_constant__ CUtensorMap tmC, const AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bar;          // [2]
  uint64_t* empty = bar + 2;     // [2]
  uint64_t* s_full = bar + 4;    // [2]
  uint64_t* q_full = bar + 6;
  uint64_t* q_empty = bar + 7;
  uint64_t* p_full = bar + 8;
  uint64_t* pv_done = bar + 9;
  uint64_t* o_free = bar + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, t = blockIdx.y, half = blockIdx.z;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&s_full[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(o_free, 128);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) tc::prefetch_tmap(&tmC);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  tc::grid_dep_wait();   // plan, query image and cache come from earlier kernels

  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint32_t sT = smem_u32(smem + kOffTile);
  const uint32_t sP = smem_u32(smem + kOffP);
  int issued = 0;   // producer: cache tiles issued

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      SegIter it;
      it.init(&a, c, t);
      int sb, p0, p1, slot, k = 0, g = 0;
      while (it.next(&sb, &p0, &p1, &slot)) {
        const int n = ntiles_of(p0, p1);
        if (n == 0) continue;
        if (k > 0 && !mbar_wait(q_empty, (k - 1) & 1, a.status, 21)) { *abort_flag = 1; break; }
        if (*abort_flag) break;
        tc::mbar_arrive_expect_tx(smem_u32(q_full), kQImgBytes);
        const uint8_t* qsrc = a.qimg + ((size_t)sb * a.T + t) * kQImgBytes;
        for (int fb = 0; fb < 9; ++fb)
          tc::bulk_load(sQ + fb * 16384, qsrc + fb * 16384, 16384, smem_u32(q_full));
        for (int i = 0; i < n; ++i, ++g) {
          const int s = g & 1;
          if (g >= 2 && !mbar_wait(&empty[s], ((g >> 1) - 1) & 1, a.status, 22)) {
            *abort_flag = 1;
            break;
          }
          if (*abort_flag) break;
          const int p = p0 + i * kTok;
          int pg = a.bt[(size_t)sb * a.max_pages + p / kPage];
          if (pg < 0 || pg >= a.num_pages) {
            report(a.status, MLA_ERR_DEVICE_INDEX, 4000000 + sb);
            pg = 0;
          }
          const int y = pg * kPage + (p % kPage);
          tc::mbar_arrive_expect_tx(smem_u32(&full[s]), kTileBytes);
          for (int fb = 0; fb < 9; ++fb)
            tc::tma_load_2d(sT + s * kTileBytes + fb * kTileBlock, &tmC, fb * 64, y,
                            smem_u32(&full[s]));
          issued = g + 1;
        }
        if (*abort_flag) break;
        ++k;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idS = tc::idesc_bf16(128, kTok, false, false);
      constexpr uint32_t idO = tc::idesc_bf16(128, 256, false, true);
      SegIter it;
      it.init(&a, c, t);
      int sb, p0, p1, slot, k = 0, g = 0;
      auto issue_s = [&](int gg) -> bool {
        const int s = gg & 1;
        if (!mbar_wait(&full[s], (gg >> 1) & 1, a.status, 23)) return false;
        tc::fence_after_sync();
        const uint32_t tile = sT + s * kTileBytes;
#pragma unroll 4
        for (int kk = 0; kk < 36; ++kk) {
          const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint32_t toff = (kk >> 2) * kTileBlock + (kk & 3) * 32;
          tc::mma_ss(tmem + kColS + s * kTok, tc::sdesc(sQ + koff, 16, 1024),
                     tc::sdesc(tile + toff, 16, 1024), idS, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(smem_u32(&s_full[s]));
        return true;
      };
      bool ok = true;
      while (ok && it.next(&sb, &p0, &p1, &slot)) {
        const int n = ntiles_of(p0, p1);
        if (n == 0) continue;
        if (!mbar_wait(q_full, k & 1, a.status, 24)) { ok = false; break; }
        for (int i = 0; i < n; ++i, ++g) {
          if (i == 0 && !(ok = issue_s(g))) break;
          if (i + 1 < n && !(ok = issue_s(g + 1))) break;
          if (i == n - 1) tc::mma_commit(smem_u32(q_empty));
          if (i == 0 && k > 0 && !(ok = mbar_wait(o_free, (k - 1) & 1, a.status, 25))) break;
          if (!(ok = mbar_wait(p_full, g & 1, a.status, 26))) break;
          if (*abort_flag) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t tile = sT + (g & 1) * kTileBytes + half * 4 * kTileBlock;
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            tc::mma_ss(tmem, sdesc64(sP + kk * 32, 512), tc::sdesc(tile + kk * 2048, kTileBlock, 1024),
                       idO, (i > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(smem_u32(&empty[g & 1]));
          tc::mma_commit(smem_u32(pv_done));
        }
        ++k;
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;          // head
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    SegIter it;
    it.init(&a, c, t);
    int sb, p0, p1, slot, g = 0;
    bool ok = true;
    while (ok && it.next(&sb, &p0, &p1, &slot)) {
      const int n = ntiles_of(p0, p1);
      const size_t prow = ((size_t)slot * a.T + t) * kHeads + row;
      float* dst = a.part_o + prow * kLat + half * 256;
      if (n == 0) {
        for (int j = 0; j < 256; j += 4)
          *reinterpret_cast<float4*>(dst + j) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (half == 0) a.part_lse[prow] = -INFINITY;
        continue;
      }
      float m_used = -INFINITY, l = 0.f;
      for (int i = 0; i < n; ++i, ++g) {
        const int s = g & 1;
        ok = mbar_wait(&s_full[s], (g >> 1) & 1, a.status, 27);
        if (__any_sync(0xffffffffu, !ok || *abort_flag)) { ok = false; break; }
        tc::fence_after_sync();
        float x[32];
        {
          float v[16];
          tc::tmem_ld16(trow + kColS + s * kTok, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) x[j] = v[j];
          tc::tmem_ld16(trow + kColS + s * kTok + 16, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) x[16 + j] = v[j];
        }
        const int valid = min(kTok, p1 - (p0 + i * kTok));
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          x[j] = j < valid ? x[j] * a.scale_log2 : -INFINITY;
          mx = fmaxf(mx, x[j]);
        }
        if (i > 0) {
          ok = mbar_wait(pv_done, (g - 1) & 1, a.status, 28);
          if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
          tc::fence_after_sync();
        }
        const bool need = mx > m_used + kRescale;
        if (i == 0) {
          m_used = mx;
        } else if (__any_sync(0xffffffffu, need)) {
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
        float psum = 0.f;
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float e0 = exp2f(x[2 * j] - m_used), e1 = exp2f(x[2 * j + 1] - m_used);
          psum += e0 + e1;
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(e0, e1);
          pk[j] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        l += psum;
        if (valid < kTok) {
          // rows past the visible end hold stale pool data: zero this half's
          // columns of them so that 0 * (Inf or NaN) cannot reach the PV MMA
          uint8_t* st0 = smem + kOffTile + s * kTileBytes + half * 4 * kTileBlock;
          const int ntail = (kTok - valid) * 4 * 8;
          for (int e = threadIdx.x - 64; e < ntail; e += 128) {
            const int r = valid + (e >> 5), blk = (e >> 3) & 3, ch = e & 7;
            *reinterpret_cast<uint4*>(st0 + blk * kTileBlock + (r >> 3) * 1024 + (r & 7) * 128 +
                                      ch * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        uint8_t* prow_s = smem + kOffP;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
          *reinterpret_cast<uint4*>(prow_s + p_off(row, ch)) =
              make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        tc::fence_async_smem();
        tc::fence_before_sync();
        tc::mbar_arrive(smem_u32(p_full));
      }
      if (!ok) break;
      // segment epilogue: O / l and the log-sum-exp
      ok = mbar_wait(pv_done, (g - 1) & 1, a.status, 29);
      if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
      tc::fence_after_sync();
      const float inv = 1.f / l;
      for (int c0 = 0; c0 < 256; c0 += 16) {
        float v[16];
        tc::tmem_ld16(trow + c0, v);
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          __stcg(reinterpret_cast<float4*>(dst + c0 + j),
                 make_float4(v[j] * inv, v[j + 1] * inv, v[j + 2] * inv, v[j + 3] * inv));
      }
      if (half == 0) a.part_lse[prow] = m_used + log2f(l);
      tc::fence_before_sync();
      tc::mbar_arrive(smem_u32(o_free));
    }
    if (!ok) *abort_flag = 1;
  }

  // ------------------------------------------------------------ teardown
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    for (int i = 0; i < 2 && i < issued; ++i) {
      const int gl = issued - 1 - i;
      mbar_wait(&full[gl & 1], (gl >> 1) & 1, a.status, 30, 1 << 20, 100000000ull);
    }
    mbar_wait(q_full, 0, a.status, 31, 1 << 20, 100000000ull);
  }
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool tc_attend(mla_ctx* ctx, const __nv_bfloat16* qimg, const __nv_bfloat16* cache,
               int num_pages, const int32_t* bt, int max_pages, int B, int T, char* ws,
               const WsLayout& L, cudaStream_t st) {
  CUtensorMap tmC;
  if (!make_tmap_bf16_2d(&tmC, cache, (uint64_t)num_pages * kPage, kRow, kRow, 64, kTok, false))
    return false;
  AttArgs a{};
  a.lens = reinterpret_cast<const int*>(ws + L.lens);
  a.prefix = reinterpret_cast<const int*>(ws + L.page_prefix);
  a.first_split = reinterpret_cast<const int*>(ws + L.first_split);
  a.slot_base = reinterpret_cast<const int*>(ws + L.slot_base);
  a.meta = reinterpret_cast<const int*>(ws + L.meta);
  a.bt = bt;
  a.qimg = reinterpret_cast<const uint8_t*>(qimg);
  a.part_o = reinterpret_cast<float*>(ws + L.part_o);
  a.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  a.status = ctx->status;
  a.B = B;
  a.T = T;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.scale_log2 = ctx->cfg.softmax_scale * 1.4426950408889634f;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmem) != cudaSuccess)
      return false;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.G, T, 2);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_mark(ctx, st, "attend");
  ctx->launches += 1;
  return cudaLaunchKernelEx(&cfg, attend_tc_kernel, tmC, a) == cudaSuccess;
}

}  // namespace mla
