// Fixed data layouts shared by the bf16 kernels.
#pragma once

#include <cstddef>
#include <cstdint>

namespace mla {

// DeepSeek-V2 widths served by the bf16 path.
constexpr int kHeads = 128, kNope = 128, kDv = 128, kLat = 512, kRope = 64;
constexpr int kRow = kLat + kRope;            // 576 cached elements per token
constexpr int kPage = 64;

// Query image: the absorbed query of one token, [q~ (512) ; RoPE(q^R) (64)]
// for all 128 heads (147456 bytes).
//  * q~ (features 0..511) is chunk-major: 32-byte chunk j (features
//    16j..16j+15) of head r at j * 4096 + r * 32.  The attention moves it
//    into tensor memory with one thread per head, so a warp's 32 heads read
//    1 KB contiguous per load, and a writer of one head stores whole
//    32-byte sectors.
//  * RoPE(q^R) (features 512..575) is stored as the attention keeps it in
//    shared memory: [128 heads][128 B] with the 128-byte swizzle (16-byte
//    chunk c of head r at position c ^ (r % 8)), moved by one bulk copy.
constexpr int kQImgBytes = 9 * 128 * 128;     // 147456

__host__ __device__ __forceinline__ uint32_t qimg_off(int head, int f) {
  if (f < kLat) return (uint32_t)((f >> 4) * 4096 + head * 32 + (f & 15) * 2);
  const int c = f - kLat;
  return (uint32_t)(8 * 16384 + (head >> 3) * 1024 + (head & 7) * 128 +
                    (((c >> 3) ^ (head & 7)) << 4) + (c & 7) * 2);
}

// Split result of one (slot, query token): 128 heads x 512 latent columns in
// fp32 (256 KB), in groups of 16 heads (32 KB each), chunk-major inside a
// group: the 8 columns 8j..8j+7 of head r at float offset (r / 16) * 8192 +
// j * 128 + (r % 16) * 8.  The attention writes a head per thread, so a
// warp's 32 heads store two 512-byte runs per 32-byte chunk; a merge of 16
// heads reads one contiguous 32 KB group.
constexpr int kPartFloats = kHeads * kLat;    // floats per (slot, token)

__host__ __device__ __forceinline__ size_t part_off(size_t slot_token, int head, int col) {
  return slot_token * kPartFloats + (size_t)(head >> 4) * (16 * kLat) + (size_t)(col >> 3) * 128 +
         (head & 15) * 8 + (col & 7);
}

}  // namespace mla
