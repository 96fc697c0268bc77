// Prefill (a chunk of T new tokens per sequence) in the explicit form.
//
// The pages note that absorbed decode is not always the fastest form
// (www.pptc.cn/news/140720 §6 问题三): recovering K and V pays off when many
// query tokens share them.  For a chunk of T query tokens against S cached
// tokens the absorbed form does 2·128·(576 + 512) FLOP per (query, key) pair,
// the explicit form 2·128·(192 + 128) after up-projecting every key once
// (2·2·512·16384 FLOP per key: K^C = W^UK c, V = W^UV c, page "DeepSeek-V2：
// 在“大力出奇迹”的AI军备竞赛中，四两拨千斤", liang.world, 第二章 §2).  Here:
//   gather     cached rows of each sequence -> contiguous [B, Smax, 576]
//              (rows past the sequence's length zeroed)
//   up-proj    K^C = rows W^UK^T, V = rows W^UV^T (the weight-streaming GEMM)
//   rope_q     q_rot = [q^C ; RoPE_pos(q^R)] per head (§3)
//   attention  per (128-query tile, head, sequence): S = q_rot K^T with
//              K = [K^C_i ; k^R] (192 features), causal softmax, O = P V_i,
//              on tcgen05 (S and O in TMEM, P written over S as bf16)
//   W_O        u = W_O [o_1; ...; o_128] (the weight-streaming GEMM)
#include <algorithm>

#include "layouts.cuh"
#include "tc_util.cuh"
#include "tmap.h"
#include "wgemm.h"
#include "plan_device.cuh"
#include "launch_util.h"
#include "attend_common.cuh"

namespace mla {
namespace {

using namespace att;

// ---------------------------------------------------------------- gather
// Row p of sequence b of the pool -> G[b * Smax + p] (16-byte pieces; rows
// p >= len_b are zero, so every key and value the attention touches is
// finite).  A bad page id is reported and its row written as zeros.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const __nv_bfloat16* __restrict__ cache, const int32_t* __restrict__ bt,
                   const int32_t* __restrict__ seq_lens, int B, int T, int max_pages,
                   int max_position, int num_pages, int Smax, __nv_bfloat16* __restrict__ G,
                   int* status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kPieces = kRow * 2 / 16;   // 72 pieces of 16 bytes per row
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)B * Smax * kPieces) return;
  const int piece = (int)(i % kPieces);
  const long long r = i / kPieces;
  const int b = (int)(r / Smax), p = (int)(r % Smax);
  const int len = plan_len(seq_lens, b, T, kPage, max_pages, max_position);
  if (p == 0 && piece == 0 && len != seq_lens[b]) report(status, MLA_ERR_DEVICE_INDEX, 1000000 + b);
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (p < len) {
    const int pg = bt[(size_t)b * max_pages + p / kPage];
    if (pg >= 0 && pg < num_pages) {
      v = *reinterpret_cast<const uint4*>(cache + ((size_t)pg * kPage + p % kPage) * kRow +
                                          piece * 8);
    } else if (piece == 0) {
      report(status, MLA_ERR_DEVICE_INDEX, 5000000 + b);
    }
  }
  *reinterpret_cast<uint4*>(G + (size_t)r * kRow + piece * 8) = v;
}

// ---------------------------------------------------------------- rope_q
// q_rot[m, h] = [q^C ; RoPE_pos(q^R)] with pos = len_b - T + t (m = b T + t):
// one thread per (m, head, 8 features).
__global__ void __launch_bounds__(256)
rope_q_kernel(const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ seq_lens, int B,
              int T, int max_pages, int max_position, const float2* __restrict__ rope_cs,
              __nv_bfloat16* __restrict__ q_rot) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kQ = kNope + kRope;   // 192
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)B * T * kHeads * (kQ / 8)) return;
  const int ch = (int)(i % (kQ / 8));
  const long long mh = i / (kQ / 8);
  const int m = (int)(mh / kHeads);
  const int b = m / T, t = m % T;
  const size_t off = (size_t)mh * kQ + ch * 8;
  uint4 raw = *reinterpret_cast<const uint4*>(q + off);
  if (ch * 8 >= kNope) {
    const int pos = plan_len(seq_lens, b, T, kPage, max_pages, max_position) - T + t;
    const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(&raw);
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float x0 = __bfloat162float(x[2 * p]), x1 = __bfloat162float(x[2 * p + 1]);
      const float2 cs = rope_cs[(size_t)pos * (kRope / 2) + (ch * 8 - kNope) / 2 + p];
      const __nv_bfloat162 r = __floats2bfloat162_rn(x0 * cs.x - x1 * cs.y, x0 * cs.y + x1 * cs.x);
      o[p] = *reinterpret_cast<const uint32_t*>(&r);
    }
    raw = make_uint4(o[0], o[1], o[2], o[3]);
  }
  *reinterpret_cast<uint4*>(q_rot + off) = raw;
}

// ---------------------------------------------------------------- attention
constexpr int kFQ = 128;                         // query rows per CTA
constexpr int kFK = 128;                         // keys per tile
constexpr uint32_t kFKBytes = 3 * 16384;         // K tile: 3 blocks [128 keys][64 features]
constexpr uint32_t kFVBytes = 2 * 16384;         // V tile: 2 blocks [128 keys][64 columns]
constexpr uint32_t kFOffK = 3 * 16384;           // two K stages after the Q tile
constexpr uint32_t kFOffV = kFOffK + 2 * kFKBytes;   // two V stages
constexpr uint32_t kFOffBar = kFOffV + 2 * kFVBytes;
constexpr uint32_t kFOffX = kFOffBar + 256;      // row-max exchange [2 tiles][2 halves][128], l [2][128]
constexpr uint32_t kFSmem = kFOffX + 4096 + 1024;
constexpr uint32_t kFColO = 256;                 // TMEM: S0 at 0, S1 at 128, O at 256
constexpr int kFThreads = 320;                   // producer, MMA issuer, 8 softmax warps

struct FaArgs {
  const int32_t* seq_lens;
  __nv_bfloat16* o;      // [B*T, 128*128]
  int* status;
  int B, T, Smax, max_pages, max_position;
  float scale_log2;
};

__global__ void __launch_bounds__(kFThreads, 1)
prefill_attend_kernel(const __grid_constant__ CUtensorMap tmQ,   // q_rot [B*T, 128*192]
                      const __grid_constant__ CUtensorMap tmK,   // K^C [B*Smax, 128*128]
                      const __grid_constant__ CUtensorMap tmR,   // rows [B*Smax, 576]
                      const __grid_constant__ CUtensorMap tmV,   // V [B*Smax, 128*128]
                      const FaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kFOffBar);
  // K and V stream through separate two-stage rings: K(j) is released when
  // S(j) completes and V(j) when PV(j) does, so K(j + 2) loads while the
  // softmax of tile j runs
  uint64_t* kfull = bar;         // [2] K stage loaded
  uint64_t* kempty = bar + 2;    // [2] K stage consumed (S done)
  uint64_t* s_full = bar + 4;    // [2] S of tiles of that parity done
  uint64_t* p_full = bar + 6;    // [2] P written (8 softmax warps)
  uint64_t* pv_done = bar + 8;   // [2] PV of tiles of that parity done
  uint64_t* q_full = bar + 10;
  uint64_t* drained = bar + 11;
  uint64_t* vfull = bar + 12;    // [2] V stage loaded
  uint64_t* vempty = bar + 14;   // [2] V stage consumed (PV done)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* sm_fail = reinterpret_cast<volatile int*>(tmem_slot + 2);
  float* xmax = reinterpret_cast<float*>(smem + kFOffX);   // [2][2][128]
  float* xl = xmax + 512;                                    // [2][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, head = blockIdx.y, b = blockIdx.z;
  tc::grid_dep_launch();
  tc::grid_dep_wait();   // q_rot, K^C, V and the gathered rows come from earlier kernels
  const int t0 = qt * kFQ;
  if (t0 >= a.T) return;
  const int len = plan_len(a.seq_lens, b, a.T, kPage, a.max_pages, a.max_position);
  const int q0 = len - a.T + t0;                       // position of the tile's first query
  const int qlast = len - a.T + min(t0 + kFQ - 1, a.T - 1);
  const int n = qlast / kFK + 1;                       // key tiles the tile's queries see
  const int krow0 = b * a.Smax;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(drained, 1);
    *abort_flag = 0;
    *sm_fail = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  int k_issued = 0, v_issued = 0;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    const bool el = tc::elect_one();
    if (el) {
      tc::prefetch_tmap(&tmQ);
      tc::prefetch_tmap(&tmK);
      tc::prefetch_tmap(&tmR);
      tc::prefetch_tmap(&tmV);
      tc::mbar_arrive_expect_tx(smem_u32(q_full), 3 * 16384);
      for (int blk = 0; blk < 3; ++blk)
        tc::tma_load_2d(smem_u32(smem + blk * 16384), &tmQ, head * (kNope + kRope) + blk * 64,
                        b * a.T + t0, smem_u32(q_full));
    }
    // K one tile ahead of V: K(0), K(1), V(0), K(2), V(1), ...
    for (int j = 0; j <= n; ++j) {
      if (j < n) {
        const int s = j & 1;
        if (j >= 2 && !warp_wait<false>(&kempty[s], ((j >> 1) - 1) & 1, a.status, 101)) {
          *abort_flag = 1;
          break;
        }
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        k_issued = j + 1;
        if (el) {
          const uint32_t st = smem_u32(smem + kFOffK + s * kFKBytes);
          const uint32_t fb = smem_u32(&kfull[s]);
          const int y = krow0 + j * kFK;
          tc::mbar_arrive_expect_tx(fb, kFKBytes);
          tc::tma_load_2d(st, &tmK, head * kNope, y, fb);
          tc::tma_load_2d(st + 16384, &tmK, head * kNope + 64, y, fb);
          tc::tma_load_2d(st + 32768, &tmR, kLat, y, fb);
        }
      }
      if (j >= 1) {
        const int jv = j - 1, s = jv & 1;
        if (jv >= 2 && !warp_wait<false>(&vempty[s], ((jv >> 1) - 1) & 1, a.status, 109)) {
          *abort_flag = 1;
          break;
        }
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        v_issued = jv + 1;
        if (el) {
          const uint32_t st = smem_u32(smem + kFOffV + s * kFVBytes);
          const uint32_t fb = smem_u32(&vfull[s]);
          const int y = krow0 + jv * kFK;
          tc::mbar_arrive_expect_tx(fb, kFVBytes);
          tc::tma_load_2d(st, &tmV, head * kDv, y, fb);
          tc::tma_load_2d(st + 16384, &tmV, head * kDv + 64, y, fb);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // S(j) into S buffer j & 1 (after PV(j - 2), which read P(j - 2) from
    // there), then PV(j - 1), so that S(j) overlaps the softmax of j - 1.
    const bool el = tc::elect_one();
    constexpr uint32_t idS = tc::idesc_bf16(128, kFK, false, false);
    constexpr uint32_t idO = tc::idesc_bf16(128, kDv, false, true);
    const uint64_t dQ = tc::sdesc(smem_u32(smem), 16, 1024);
    const uint64_t dR = tc::sdesc(smem_u32(smem + kFOffK), 16, 1024);
    const uint64_t dV = tc::sdesc(smem_u32(smem + kFOffV), 16384, 1024);
    bool ok = warp_wait<false>(q_full, 0, a.status, 102);
    for (int j = 0; ok && j <= n; ++j) {
      if (j < n) {
        const int s = j & 1;
        if (j >= 2 && !warp_wait<false>(&pv_done[s], ((j - 2) >> 1) & 1, a.status, 103)) {
          ok = false;
          break;
        }
        if (!warp_wait<false>(&kfull[s], (j >> 1) & 1, a.status, 104)) { ok = false; break; }
        tc::fence_after_sync();
        if (el) {
          const uint32_t d = tmem + s * kFK;
          const uint64_t dk = dR + ((s * kFKBytes) >> 4);
          // straight-line MMAs (a branch between MMAs slows their issue)
#pragma unroll
          for (int blk = 0; blk < 3; ++blk) {
            const uint64_t qa = dQ + blk * 1024, kb = dk + blk * 1024;
            tc::mma_ss(d, qa, kb, idS, blk > 0 ? 1u : 0u);
            tc::mma_ss(d, qa + 2, kb + 2, idS, 1u);
            tc::mma_ss(d, qa + 4, kb + 4, idS, 1u);
            tc::mma_ss(d, qa + 6, kb + 6, idS, 1u);
          }
          tc::mma_commit(smem_u32(&kempty[s]));
          tc::mma_commit(smem_u32(&s_full[s]));
        }
      }
      if (j >= 1) {
        const int jv = j - 1, s = jv & 1;
        if (!warp_wait<false>(&p_full[s], (jv >> 1) & 1, a.status, 105) ||
            !warp_wait<false>(&vfull[s], (jv >> 1) & 1, a.status, 110)) {
          ok = false;
          break;
        }
        if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
        tc::fence_after_sync();
        if (el) {
          const uint32_t pcol = tmem + s * kFK;
          const uint64_t vb = dV + ((s * kFVBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)   // 16 keys per K step: 8 P columns, 2 atoms of V
            tc::mma_ts(tmem + kFColO, pcol + 8 * kk, vb + kk * (2048 >> 4), idO,
                       (jv > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(smem_u32(&pv_done[s]));
          tc::mma_commit(smem_u32(&vempty[s]));
        }
      }
    }
    if (!ok) *abort_flag = 1;
    if (el) tc::mma_commit(smem_u32(drained));
  } else {
    // ---------------------------------------------------------- softmax
    // Eight warps: warps w and w + 4 share TMEM lanes 32 (w % 4).. (thread =
    // query row) and take keys 0..63 and 64..127 of each tile (and O columns
    // 0..63 and 64..127).  The two halves of a row exchange their maxima
    // through shared memory at a barrier of the 256 softmax threads, so
    // both take the same maximum and rescale decision; l is kept per half
    // and summed at the end.  Keys up to the query's own position are
    // visible.  A failed wait raises sm_fail, which every thread reads after
    // the next barrier, so all 256 leave together.
    const int q4 = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = q4 * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const int qpos = q0 + row;
    const bool live = t0 + row < a.T;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int s = j & 1;
      if (!bar_wait<false>(&s_full[s], (j >> 1) & 1, a.status, 106) || *abort_flag) *sm_fail = 1;
      tc::fence_after_sync();
      uint32_t v[64];
      tc::tmem_ld64(trow + s * kFK + half * 64, v);
      const int valid = live ? max(0, min(kFK, qpos - j * kFK + 1)) : 0;
      const int vh = max(0, min(64, valid - half * 64));   // visible keys of this half
      float mh = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c)
        if (c < vh) mh = fmaxf(mh, __uint_as_float(v[c]));
      xmax[(s * 2 + half) * 128 + row] = mh;
      tc::named_sync(1, 256);
      if (*sm_fail) { ok = false; break; }   // read after the barrier: the same for all
      const float mx = fmaxf(mh, xmax[(s * 2 + (half ^ 1)) * 128 + row]) * a.scale_log2;
      const bool need = j > 0 && mx > m_used + kRescale;
      if (j == 0) {
        m_used = mx;
      } else if (__any_sync(0xffffffffu, need)) {
        // O holds PV(0..j-1): rescale this half's columns once PV(j - 1) is done
        if (!bar_wait<false>(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, a.status, 107))
          *sm_fail = 1;
        tc::fence_after_sync();
        const float m_new = need ? mx : m_used;
        const float f = exp2f(m_used - m_new);
        l *= f;
        for (int c0 = 0; c0 < 64; c0 += 16) {
          float o[16];
          tc::tmem_ld16(trow + kFColO + half * 64 + c0, o);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) o[jj] *= f;
          tc::tmem_st16(trow + kFColO + half * 64 + c0, o);
        }
        m_used = m_new;
      }
      // P (bf16, two keys per column) over this half's S columns: keys
      // half*64 + 2i, +1 -> column half*32 + i (the S MMA of j + 2 waits for
      // PV(j) before reusing the buffer)
      uint32_t pk[32];
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int c0 = 2 * i, c1 = 2 * i + 1;
        const float e0 = c0 < vh ? tc::ex2_approx(fmaf(__uint_as_float(v[c0]), a.scale_log2, -m_used)) : 0.f;
        const float e1 = c1 < vh ? tc::ex2_approx(fmaf(__uint_as_float(v[c1]), a.scale_log2, -m_used)) : 0.f;
        psum += e0 + e1;
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(e0, e1);
        pk[i] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      l += psum;
      tc::tmem_st32(trow + s * kFK + half * 32, pk);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(smem_u32(&p_full[s]));
    }
    // epilogue: l of both halves, then O / l of this half's 64 columns
    if (ok && !bar_wait<false>(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, a.status, 108))
      *sm_fail = 1;
    xl[half * 128 + row] = l;
    tc::named_sync(1, 256);
    if (ok && !*sm_fail) {
      tc::fence_after_sync();
      const float lt = l + xl[(half ^ 1) * 128 + row];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      __nv_bfloat16* dst =
          a.o + ((size_t)(b * a.T + t0 + row)) * (kHeads * kDv) + head * kDv + half * 64;
      for (int c0 = 0; c0 < 64; c0 += 16) {
        float o[16];
        tc::tmem_ld16(trow + kFColO + half * 64 + c0, o);
        if (live) {
          uint32_t w[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * jj] * inv, o[2 * jj + 1] * inv);
            w[jj] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(dst + c0) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(dst + c0 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    } else {
      ok = false;
    }
    if (!ok) *abort_flag = 1;
  }

  // ------------------------------------------------------------ teardown
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (*abort_flag) {
      mbar_wait(q_full, 0, a.status, 111, 1 << 20, 100000000ull);
      for (int i = 0; i < 2 && i < k_issued; ++i) {
        const int u = k_issued - 1 - i;
        mbar_wait(&kfull[u & 1], (u >> 1) & 1, a.status, 112, 1 << 20, 100000000ull);
      }
      for (int i = 0; i < 2 && i < v_issued; ++i) {
        const int u = v_issued - 1 - i;
        mbar_wait(&vfull[u & 1], (u >> 1) & 1, a.status, 113, 1 << 20, 100000000ull);
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    mbar_wait(drained, 0, a.status, 114, 1 << 20, 100000000ull);
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

cudaLaunchConfig_t pdl_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                           cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

PrefillLayout prefill_layout(const mla_ctx* ctx, int B, int T, int max_pages) {
  PrefillLayout L{};
  const size_t M = (size_t)B * T;
  L.Smax = max_pages * kPage;
  const size_t R = (size_t)B * L.Smax;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = (off + bytes + 255) & ~size_t(255); return o; };
  L.rows = take(R * kRow * 2);
  L.k = take(R * kHeads * kNope * 2);
  L.v = take(R * kHeads * kDv * 2);
  L.q_rot = take(M * kHeads * (kNope + kRope) * 2);
  L.o = take(M * kHeads * kDv * 2);
  L.wg_part = take(prefill_partial_bytes(ctx, (int)R, (int)M));
  L.total = off;
  return L;
}

bool bf16_prefill_explicit(mla_ctx* ctx, const __nv_bfloat16* q, const __nv_bfloat16* cache,
                           int num_pages, const int32_t* bt, int max_pages,
                           const int32_t* seq_lens, int B, int T, __nv_bfloat16* out, char* ws,
                           const PrefillLayout& L, cudaStream_t st) {
  const int D = ctx->cfg.d_model;
  const int Smax = L.Smax;
  const int R = B * Smax, M = B * T;
  __nv_bfloat16* rows = reinterpret_cast<__nv_bfloat16*>(ws + L.rows);
  __nv_bfloat16* kbuf = reinterpret_cast<__nv_bfloat16*>(ws + L.k);
  __nv_bfloat16* vbuf = reinterpret_cast<__nv_bfloat16*>(ws + L.v);
  __nv_bfloat16* q_rot = reinterpret_cast<__nv_bfloat16*>(ws + L.q_rot);
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(ws + L.o);
  float* part = reinterpret_cast<float*>(ws + L.wg_part);
  cudaLaunchAttribute attr[1];
  // ---- gather the cached rows of every sequence
  {
    const long long n = (long long)R * (kRow * 2 / 16);
    cudaLaunchConfig_t cfg = pdl_cfg(dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, attr);
    prof_mark(ctx, st, "gather");
    ctx->launches += 1;
    if (cudaLaunchKernelEx(&cfg, gather_rows_kernel, cache, bt, seq_lens, B, T, max_pages,
                           ctx->cfg.max_position, num_pages, Smax, rows, ctx->status) !=
        cudaSuccess)
      return false;
  }
  // ---- K^C = rows W^UK^T and V = rows W^UV^T for every cached row
  if (!bf16_rowmajor_gemm(ctx, ctx->tm_wuk_rows, kHeads, kLat / 64, rows, R, kRow, kbuf,
                          kHeads * kNope, part, st, "key_up") ||
      !bf16_rowmajor_gemm(ctx, ctx->tm_wuv, kHeads, kLat / 64, rows, R, kRow, vbuf,
                          kHeads * kDv, part, st, "value_up"))
    return false;
  // ---- rotated queries
  {
    const long long n = (long long)M * kHeads * ((kNope + kRope) / 8);
    cudaLaunchConfig_t cfg = pdl_cfg(dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, attr);
    prof_mark(ctx, st, "rope_q");
    ctx->launches += 1;
    if (cudaLaunchKernelEx(&cfg, rope_q_kernel, q, seq_lens, B, T, max_pages,
                           ctx->cfg.max_position, (const float2*)ctx->rope_cs, q_rot) != cudaSuccess)
      return false;
  }
  // ---- causal attention per (query tile, head, sequence)
  {
    CUtensorMap tmQ, tmK, tmR, tmV;
    if (!make_tmap_bf16_2d(&tmQ, q_rot, M, kHeads * (kNope + kRope), kHeads * (kNope + kRope), 64,
                           kFQ, false) ||
        !make_tmap_bf16_2d(&tmK, kbuf, R, kHeads * kNope, kHeads * kNope, 64, kFK, false) ||
        !make_tmap_bf16_2d(&tmR, rows, R, kRow, kRow, 64, kFK, false) ||
        !make_tmap_bf16_2d(&tmV, vbuf, R, kHeads * kDv, kHeads * kDv, 64, kFK, false)) {
      cudaGetLastError();
      return false;
    }
    FaArgs fa{seq_lens, o, ctx->status, B, T, Smax, max_pages, ctx->cfg.max_position,
              ctx->cfg.softmax_scale * 1.4426950408889634f};
    static std::atomic<uint64_t> attr_done{0};
    if (smem_attr_once(attr_done, prefill_attend_kernel, (int)kFSmem) != cudaSuccess) return false;
    cudaLaunchConfig_t cfg =
        pdl_cfg(dim3((T + kFQ - 1) / kFQ, kHeads, B), dim3(kFThreads), kFSmem, st, attr);
    prof_mark(ctx, st, "prefill_attend");
    ctx->launches += 1;
    if (cudaLaunchKernelEx(&cfg, prefill_attend_kernel, tmQ, tmK, tmR, tmV, fa) != cudaSuccess)
      return false;
  }
  // ---- u = W_O o
  return bf16_rowmajor_gemm(ctx, ctx->tm_wo, D / 128, kHeads * kDv / 64, o, M, kHeads * kDv, out,
                            D, part, st, "out_proj");
}

}  // namespace mla
