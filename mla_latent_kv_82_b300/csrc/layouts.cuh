// Fixed data layouts shared by the bf16 kernels.
#pragma once

#include <cstdint>

namespace mla {

// DeepSeek-V2 widths served by the bf16 path.
constexpr int kHeads = 128, kNope = 128, kDv = 128, kLat = 512, kRope = 64;
constexpr int kRow = kLat + kRope;            // 576 cached elements per token
constexpr int kPage = 64;

// Query image: the absorbed query of one token, [q~ (512) ; RoPE(q^R) (64)]
// for all 128 heads, stored exactly as the attention kernel keeps it in
// shared memory: 9 feature blocks of 64, each [128 heads][128 B] with the
// 128-byte swizzle (16-byte chunk j of head r at position j ^ (r % 8)).
// One bulk copy moves it from global to shared memory unchanged.
constexpr int kQImgBytes = 9 * 128 * 128;     // 147456

__host__ __device__ __forceinline__ uint32_t qimg_off(int head, int f) {
  const int fb = f >> 6, c = f & 63;
  return (uint32_t)(fb * 16384 + (head >> 3) * 1024 + (head & 7) * 128 +
                    (((c >> 3) ^ (head & 7)) << 4) + (c & 7) * 2);
}

}  // namespace mla
