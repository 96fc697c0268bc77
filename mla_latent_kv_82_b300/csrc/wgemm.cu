// Weight-streaming tensor-core GEMM (tcgen05 + TMA) for the projections of
// MLA decode:  D[f, t] = sum_k W[f, k] X[t, k]  ("swap AB": the weight rows
// are the M = 128 side of the MMA, tokens the N side), fp32 accumulation in
// TMEM.  Instances (page "DeepSeek-V2：在“大力出奇迹”的AI军备竞赛中，四两拨千斤",
// liang.world, 第二章):
//   compress   [W^DKV ; W^KR] h  -> RoPE on k^R -> paged cache row  (§2, §3)
//   absorb     W^UK_i^T q^C_i per head (W^UK folded into the query)  (§2)
//   value      W^UV_i o_lat_i per head                                (§2)
//   output     W_O [o_1; ...; o_{n_h}]                                (§1)
//
// One CTA = one 128-row weight tile x one token tile (NT = 16..256 tokens)
// x one K split.  Warp 0 issues TMA loads into a STAGES-deep ring, warp 1
// issues the MMAs (one thread) and owns TMEM, warps 2-5 run the epilogue
// (one TMEM lane = one weight row per thread).  With several K splits each
// CTA writes an fp32 partial; the last CTA of a tile (atomic counter) sums
// the partials in split order, so results do not depend on timing.
// Weight tiles are requested before griddepcontrol.wait: under programmatic
// dependent launch the weight stream starts while the previous kernel ends.
#include "layouts.cuh"
#include "tc_util.cuh"
#include "wgemm.h"
#include "launch_util.h"

namespace mla {
namespace {

// Token tiles up to 64 run two CTAs per SM.  The absorbed-query GEMM reads
// K = 128 (two chunks), so two stages are all it can use, which also lets
// two of its CTAs share an SM at any tile (measured: the append + absorbed
// query launch at 256 tokens 72 -> 51 us).  Wide tiles of the long-K
// projections keep one CTA per SM with a deep ring: halving the ring for two
// CTAs per SM, with the extra K splits that brings, was measured slower
// (W_O at 256 tokens 70 -> 82 us).  Row-major outputs with 128-token tiles
// serve the short-K projections of a prefill (K^C and V of every cached row:
// K = 512, eight chunks): three stages cover a tile's K and two CTAs share
// an SM, so one CTA's epilogue overlaps the other's MMAs.
template <int NT, int EPI = WG_ROWMAJOR> struct WgCfg {
  static constexpr bool kShortK = EPI == WG_ROWMAJOR && NT == 128;
  static constexpr int kStages = EPI == WG_QIMG ? 2
                               : kShortK ? 3
                               : NT == 16 ? 6 : NT == 32 ? 5 : NT == 64 ? 4 : NT == 128 ? 6 : 4;
  static constexpr int kMinBlocks = (EPI == WG_QIMG || NT <= 64 || kShortK) ? 2 : 1;
  static constexpr uint32_t kA = 128 * 64 * 2;
  static constexpr uint32_t kB = NT * 64 * 2;
  static constexpr uint32_t kStage = kA + kB;
  static constexpr uint32_t kTmemCols = NT < 32 ? 32 : NT;
  static constexpr uint32_t kSmem = kStages * kStage + 1024 + 512;
};

constexpr int kThreads = 192;
constexpr int kStgPitch = 136;   // bf16 per staged token row (128 + 8 pad)

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&b);
}

// One CTA's work: weight tile mt, token tile nt (of ntile), K split z.
template <int NT, int EPI, bool A_MN>
__device__ __forceinline__ void wgemm_body(const CUtensorMap& tmA, const CUtensorMap& tmA2,
                                           const CUtensorMap& tmB, const WgArgs& a, const int mt,
                                           const int nt, const int z, const int ntile) {
  using C = WgCfg<NT, EPI>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * C::kStage);
  uint64_t* empty = full + S;
  uint64_t* done = empty + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);   // abort, last, go
  int* scan_tmp = reinterpret_cast<int*>(smem + S * C::kStage + 256);     // 33 ints

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int head = mt / a.tiles_per_head, tile = mt % a.tiles_per_head;
  const int kc0 = z * a.k_chunks / a.splits, kc1 = (z + 1) * a.k_chunks / a.splits;
  const int nk = kc1 - kc0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    flags[0] = 0;
    flags[1] = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmA);
    tc::prefetch_tmap(&tmA2);
    tc::prefetch_tmap(&tmB);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int issued = 0;
  // let the next kernel's CTAs start their prologue and weight loads on free
  // SMs; they still wait (griddepcontrol.wait) before touching our outputs
  tc::grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- producer
      const bool second = !A_MN && tile >= a.a_tiles_main;
      const CUtensorMap* mA = second ? &tmA2 : &tmA;
      const int a_row = A_MN ? head * a.a_head_rows
                             : head * a.a_head_rows + (second ? tile - a.a_tiles_main : tile) * 128;
      auto load_a = [&](int i) {
        const int s = i % S, kc = kc0 + i;
        const uint32_t sa = smem_u32(smem + s * C::kStage);
        if (A_MN) {
          tc::tma_load_2d(sa, mA, tile * 128, a_row + kc * 64, smem_u32(&full[s]));
          tc::tma_load_2d(sa + 8192, mA, tile * 128 + 64, a_row + kc * 64, smem_u32(&full[s]));
        } else {
          tc::tma_load_2d(sa, mA, kc * 64, a_row, smem_u32(&full[s]));
        }
      };
      auto load_b = [&](int i) {
        const int s = i % S, kc = kc0 + i;
        const uint32_t sb = smem_u32(smem + s * C::kStage) + C::kA;
        tc::tma_load_2d(sb, &tmB, head * a.b_head_cols + kc * 64, nt * NT, smem_u32(&full[s]));
      };
      // weights first (independent of the previous kernel), then activations
      const int pre = nk < S ? nk : S;
      for (int i = 0; i < pre; ++i) {
        tc::mbar_arrive_expect_tx(smem_u32(&full[i]), C::kStage);
        load_a(i);
      }
      tc::grid_dep_wait();
      for (int i = 0; i < pre; ++i) load_b(i);
      issued = pre;
      for (int i = pre; i < nk; ++i) {
        const int s = i % S;
        if (!mbar_wait(&empty[s], ((i / S) - 1) & 1, a.status, 11)) { flags[0] = 1; break; }
        if (flags[0]) break;
        tc::mbar_arrive_expect_tx(smem_u32(&full[s]), C::kStage);
        load_a(i);
        load_b(i);
        issued = i + 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = tc::idesc_bf16(128, NT, A_MN, false);
      for (int i = 0; i < nk; ++i) {
        const int s = i % S;
        if (!mbar_wait(&full[s], (i / S) & 1, a.status, 12)) { flags[0] = 1; break; }
        if (flags[0]) break;
        tc::fence_after_sync();
        const uint32_t sa = smem_u32(smem + s * C::kStage), sb = sa + C::kA;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = A_MN ? tc::sdesc(sa + kk * 2048, 8192, 1024)
                                   : tc::sdesc(sa + kk * 32, 16, 1024);
          const uint64_t bd = tc::sdesc(sb + kk * 32, 16, 1024);
          tc::mma_ss(tmem, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(smem_u32(&empty[s]));
      }
      tc::mma_commit(smem_u32(done));
    }
  } else {
    // ---------------- epilogue: warps 2..5, thread <-> TMEM lane <-> weight row
    tc::grid_dep_wait();   // outputs may still be read by the previous kernel
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int etid = threadIdx.x - 64;   // 0..127
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    if (EPI == WG_QIMG && a.do_plan && mt == 0 && nt == 0 && z == 0)
      build_plan<128>(etid, [] { tc::named_sync(2, 128); }, scan_tmp, a.plan);
    if (!mbar_wait(done, 0, a.status, 13)) flags[0] = 1;
    tc::fence_after_sync();
    // one decision for all 128 epilogue threads before any named barrier
    tc::named_sync(1, 128);
    if (etid == 0) flags[2] = flags[0];
    tc::named_sync(1, 128);
    const bool ok = flags[2] == 0;
    float* part = nullptr;
    bool final_cta = true;
    if (ok && a.splits > 1) {
      part = a.partials + ((size_t)(mt * ntile + nt) * a.splits) * NT * 128;
      float* mine = part + (size_t)z * NT * 128;
      for (int c0 = 0; c0 < NT; c0 += 16) {
        float v[16];
        tc::tmem_ld16(trow + c0, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) __stcg(mine + (c0 + j) * 128 + row, v[j]);
      }
      __threadfence();
      tc::named_sync(1, 128);
      if (etid == 0) {
        const int prev = atomicAdd(&a.counters[mt * ntile + nt], 1);
        const int last = prev == a.splits - 1;
        if (last) a.counters[mt * ntile + nt] = 0;
        flags[1] = last;
      }
      tc::named_sync(1, 128);
      final_cta = flags[1] != 0;
      __threadfence();
    }
    if (ok && final_cta) {
      uint16_t* stg = reinterpret_cast<uint16_t*>(smem);   // stages are idle now
      const int rows_valid = (tile == a.tiles_per_head - 1) ? a.valid_rows_last : 128;
      for (int c0 = 0; c0 < NT; c0 += 16) {
        float v[16];
        if (a.splits > 1) {
          // sum the partials in split order; four splits in flight at a time
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = 0.f;
          int zz = 0;
          for (; zz + 4 <= a.splits; zz += 4) {
            float w[4][16];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float* p = part + (size_t)(zz + u) * NT * 128 + c0 * 128 + row;
#pragma unroll
              for (int j = 0; j < 16; ++j) w[u][j] = __ldcg(p + j * 128);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] += w[u][j];
          }
          for (; zz < a.splits; ++zz) {
            const float* p = part + (size_t)zz * NT * 128 + c0 * 128 + row;
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] += __ldcg(p + j * 128);
          }
        } else {
          tc::tmem_ld16(trow + c0, v);
        }
        const int t0 = nt * NT + c0;
        if (EPI == WG_APPEND && a.append_rope_tile == tile) {
          // k^R rows: interleaved RoPE pairs live in neighbouring lanes
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
            const int t = t0 + j;
            if (t < a.n_tokens && row < 64) {
              const int pos = a.pos[t];
              if (pos >= 0 && pos < a.max_position) {
                const float2 cs = a.rope_cs[(size_t)pos * (kRope / 2) + (row >> 1)];
                v[j] = (row & 1) ? fmaf(other, cs.y, v[j] * cs.x) : fmaf(-other, cs.y, v[j] * cs.x);
              }
            }
          }
        }
        // stage 16 tokens x 128 rows as bf16, then 16-byte stores per token row
#pragma unroll
        for (int j = 0; j < 16; ++j) stg[j * kStgPitch + row] = bf16_bits(v[j]);
        tc::named_sync(1, 128);
        for (int e = etid; e < 16 * 16; e += 128) {
          const int j = e >> 4, ch = e & 15;
          const int t = t0 + j;
          if (t >= a.n_tokens || ch * 8 >= rows_valid) continue;
          const uint4 val = *reinterpret_cast<const uint4*>(stg + j * kStgPitch + ch * 8);
          __nv_bfloat16* dst = nullptr;
          if (EPI == WG_ROWMAJOR && a.out_rows_per_head > 0) {
            // weight row gr belongs to output head gr / rows_per_head
            const int gr = tile * 128 + ch * 8;
            dst = a.out + (size_t)t * a.ld_out + (gr / a.out_rows_per_head) * a.out_head_cols +
                  gr % a.out_rows_per_head;
          } else if (EPI == WG_ROWMAJOR) {
            dst = a.out + (size_t)t * a.ld_out + head * a.out_head_cols + tile * 128 + ch * 8;
          } else if (EPI == WG_QIMG) {
            // 8 consecutive features of one head are one 16-byte chunk of the image
            dst = reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<uint8_t*>(a.qimg) +
                                                   (size_t)t * kQImgBytes +
                                                   qimg_off(head, tile * 128 + ch * 8));
          } else if (a.stage_rows) {   // WG_APPEND into a staging buffer, row t
            dst = a.cache + (size_t)t * kRow + tile * 128 + ch * 8;
          } else {   // WG_APPEND
            const int pos = a.pos[t];
            const int b = t / a.T;
            const int lp = pos / kPage;
            if (pos < 0 || pos >= a.max_position || lp >= a.max_pages) {
              if (ch == 0 && tile == 0) report(a.status, MLA_ERR_DEVICE_INDEX, 2000000 + t);
              continue;
            }
            const int pg = a.bt[(size_t)b * a.max_pages + lp];
            if (pg < 0 || pg >= a.num_pages) {
              if (ch == 0 && tile == 0) report(a.status, MLA_ERR_DEVICE_INDEX, 3000000 + t);
              continue;
            }
            dst = a.cache + ((size_t)pg * kPage + pos % kPage) * kRow + tile * 128 + ch * 8;
          }
          *reinterpret_cast<uint4*>(dst) = val;
        }
        tc::named_sync(1, 128);
      }
      if (EPI == WG_QIMG && tile == 0) {
        // rotated q^R of this head for the tile's tokens -> image features
        // 512..575, one 16-byte chunk (4 RoPE pairs) per step
        for (int e = etid; e < NT * 8; e += 128) {
          const int t = nt * NT + (e >> 3), ch = e & 7;
          if (t >= a.n_tokens) continue;
          const int b = t / a.T, tq = t % a.T;
          const int pos = plan_len(a.plan.seq_lens, b, a.T, kPage, a.plan.max_pages,
                                   a.max_position) - a.T + tq;
          const uint4 raw = *reinterpret_cast<const uint4*>(
              a.q + ((size_t)t * kHeads + head) * (kNope + kRope) + kNope + ch * 8);
          const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw);
          uint32_t o[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float x0 = __bfloat162float(x[2 * p]), x1 = __bfloat162float(x[2 * p + 1]);
            const float2 cs = a.rope_cs[(size_t)pos * (kRope / 2) + ch * 4 + p];
            o[p] = (uint32_t)bf16_bits(x0 * cs.x - x1 * cs.y) |
                   ((uint32_t)bf16_bits(x0 * cs.y + x1 * cs.x) << 16);
          }
          *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(a.qimg) + (size_t)t * kQImgBytes +
                                    qimg_off(head, kLat + ch * 8)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }

  // ---------------- teardown
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && flags[0]) {
    // wait (bounded) for loads still in flight before shared memory goes away
    for (int i = 0; i < S && i < issued; ++i) {
      const int last_use = issued - 1 - i;
      mbar_wait(&full[last_use % S], (last_use / S) & 1, a.status, 14, 1 << 20, 100000000ull);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int NT, int EPI, bool A_MN>
__global__ void __launch_bounds__(kThreads, (WgCfg<NT, EPI>::kMinBlocks))
wgemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
             const __grid_constant__ CUtensorMap tmB, const WgArgs a) {
  wgemm_body<NT, EPI, A_MN>(tmA, tmA2, tmB, a, blockIdx.x, blockIdx.y, blockIdx.z, gridDim.y);
}

// The compress/append GEMM (first m1 * n1 * s1 CTAs, token tile NT1) and the
// absorbed-query GEMM (token tile NT2) in one launch: they share no data, so
// one waits for nothing of the other.
template <int NT1, int NT2>
struct DualCfg {
  using C1 = WgCfg<NT1, WG_APPEND>;
  using C2 = WgCfg<NT2, WG_QIMG>;
  static constexpr int kMinBlocks = C1::kMinBlocks < C2::kMinBlocks ? C1::kMinBlocks : C2::kMinBlocks;
  static constexpr uint32_t kSmem = C1::kSmem > C2::kSmem ? C1::kSmem : C2::kSmem;
};

template <int NT1, int NT2>
__global__ void __launch_bounds__(kThreads, (DualCfg<NT1, NT2>::kMinBlocks))
wgemm_dual_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmA21,
                  const __grid_constant__ CUtensorMap tmB1, const WgArgs a1,
                  const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmA22,
                  const __grid_constant__ CUtensorMap tmB2, const WgArgs a2, const int m1,
                  const int n1, const int s1, const int m2, const int n2) {
  const int c1 = m1 * n1 * s1;
  const int bid = blockIdx.x;
  if (bid < c1) {
    wgemm_body<NT1, WG_APPEND, false>(tmA1, tmA21, tmB1, a1, bid % m1, (bid / m1) % n1,
                                      bid / (m1 * n1), n1);
  } else {
    const int b = bid - c1;
    wgemm_body<NT2, WG_QIMG, true>(tmA2, tmA22, tmB2, a2, b % m2, (b / m2) % n2, b / (m2 * n2), n2);
  }
}

template <int NT1, int NT2>
cudaError_t launch_dual_nt(const WgPlan& p1, const WgPlan& p2, cudaStream_t st, bool pdl) {
  using C = DualCfg<NT1, NT2>;
  auto kern = wgemm_dual_kernel<NT1, NT2>;
  static std::atomic<uint64_t> attr_done{0};   // per instantiation
  if (const cudaError_t e = smem_attr_once(attr_done, kern, (int)C::kSmem); e != cudaSuccess)
    return e;
  const int c1 = p1.m_tiles * p1.n_tiles * p1.args.splits;
  const int c2 = p2.m_tiles * p2.n_tiles * p2.args.splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c1 + c2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p1.tmA, p1.tmA2, p1.tmB, p1.args, p2.tmA, p2.tmA2, p2.tmB,
                            p2.args, p1.m_tiles, p1.n_tiles, p1.args.splits, p2.m_tiles,
                            p2.n_tiles);
}

template <int NT1>
cudaError_t launch_dual_nt1(const WgPlan& p1, const WgPlan& p2, cudaStream_t st, bool pdl) {
  switch (p2.nt) {
    case 16: return launch_dual_nt<NT1, 16>(p1, p2, st, pdl);
    case 32: return launch_dual_nt<NT1, 32>(p1, p2, st, pdl);
    case 64: return launch_dual_nt<NT1, 64>(p1, p2, st, pdl);
    case 128: return launch_dual_nt<NT1, 128>(p1, p2, st, pdl);
    default: return launch_dual_nt<NT1, 256>(p1, p2, st, pdl);
  }
}

template <int NT, int EPI, bool A_MN>
cudaError_t launch_nt(const WgPlan& p, cudaStream_t st, bool pdl) {
  using C = WgCfg<NT, EPI>;
  auto kern = wgemm_kernel<NT, EPI, A_MN>;
  static std::atomic<uint64_t> attr_done{0};   // per instantiation
  if (const cudaError_t e = smem_attr_once(attr_done, kern, (int)C::kSmem); e != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.m_tiles, p.n_tiles, p.args.splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p.tmA, p.tmA2, p.tmB, p.args);
}

template <int EPI, bool A_MN>
cudaError_t launch_epi(const WgPlan& p, cudaStream_t st, bool pdl) {
  switch (p.nt) {
    case 16: return launch_nt<16, EPI, A_MN>(p, st, pdl);
    case 32: return launch_nt<32, EPI, A_MN>(p, st, pdl);
    case 64: return launch_nt<64, EPI, A_MN>(p, st, pdl);
    case 128: return launch_nt<128, EPI, A_MN>(p, st, pdl);
    default: return launch_nt<256, EPI, A_MN>(p, st, pdl);
  }
}

}  // namespace

int wgemm_token_tile(int n_tokens) {
  if (n_tokens <= 16) return 16;
  if (n_tokens <= 32) return 32;
  if (n_tokens <= 64) return 64;
  if (n_tokens <= 128) return 128;
  return 256;
}

int wgemm_ctas_per_sm(int nt) { return nt <= 64 ? 2 : 1; }

cudaError_t wgemm_launch_dual(const WgPlan& append, const WgPlan& qimg, cudaStream_t st, bool pdl) {
  if (append.nt == 16) return launch_dual_nt1<16>(append, qimg, st, pdl);
  if (append.nt == 32) return launch_dual_nt1<32>(append, qimg, st, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t wgemm_launch(const WgPlan& p, int epi, bool a_mn_major, cudaStream_t st, bool pdl) {
  if (a_mn_major) return launch_epi<WG_QIMG, true>(p, st, pdl);
  if (epi == WG_APPEND) return launch_epi<WG_APPEND, false>(p, st, pdl);
  return launch_epi<WG_ROWMAJOR, false>(p, st, pdl);
}

}  // namespace mla
