// philox.cuh -- the counter-based generator behind the dropout mask.
//
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
// SC 2011): ten rounds over a 128-bit counter with a 64-bit key; each round multiplies two
// counter words by fixed odd constants, swaps the halves of the products with the other two
// words xor-ed with the key, and bumps the key by Weyl constants.
//
// Dropout ("FlashAttention 与显存" §07/§09: fused into the kernel; the mask is regenerated in
// the backward pass from the generator state instead of being stored).  One generator call
// serves eight elements: element (bh, i, j) (head index, query, key) reads the 16-bit half
// j % 2 (0 = low) of word (j % 8) / 2 of philox(counter = (j / 8, i, bh, 0),
// key = (seed low, seed high)) and is kept when that half is >= t = round(p * 2^16) (at most
// 2^16 - 1); kept probabilities are scaled by 2^16 / (2^16 - t), the inverse keep probability.
#pragma once

#include <cstdint>

namespace fa {

struct DropoutParams {
  uint32_t threshold;  // t: keep when the 16-bit draw is >= t
  float scale;         // 2^16 / (2^16 - t)
  uint32_t seed_lo, seed_hi;
};

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = uint64_t(c0) * 0xD2511F53u;  // one 32 x 32 -> 64-bit product each
    const uint64_t p1 = uint64_t(c2) * 0xCD9E8D57u;
    c0 = uint32_t(p1 >> 32) ^ c1 ^ k0;
    c1 = uint32_t(p1);
    c2 = uint32_t(p0 >> 32) ^ c3 ^ k1;
    c3 = uint32_t(p0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint4(c0, c1, c2, c3);
}

// The four words behind keys 8g .. 8g+7 of query i: word m holds key 8g + 2m in its low
// half and key 8g + 2m + 1 in its high half.
__device__ __forceinline__ uint4 dropout_words(const DropoutParams& dp, uint32_t g, uint32_t i, uint32_t bh) {
  return philox4x32_10(g, i, bh, 0u, dp.seed_lo, dp.seed_hi);
}

// Keep bits of keys 8g .. 8g+7 (bit u = key 8g + u) for query i of head bh.
__device__ __forceinline__ uint32_t dropout_keep8(const DropoutParams& dp, uint32_t g, uint32_t i,
                                                  uint32_t bh) {
  const uint4 w = philox4x32_10(g, i, bh, 0u, dp.seed_lo, dp.seed_hi);
  const uint32_t t = dp.threshold;
  auto two = [t](uint32_t x) -> uint32_t { return uint32_t((x & 0xFFFFu) >= t) | (uint32_t((x >> 16) >= t) << 1); };
  return two(w.x) | (two(w.y) << 2) | (two(w.z) << 4) | (two(w.w) << 6);
}

}  // namespace fa
