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

// Keep bits of key `key` for queries qb .. qb + 8 kOctets - 1 (bit c of the result = query
// qb + c), for a thread that owns one key row.  The eight lanes holding keys 8g .. 8g+7 share
// the generator calls: lane u draws the call of query 8b + u (8 bits, one per key), the octet
// exchanges its 8 x 8 bit block by shuffles and each lane gathers its own bit column -- one
// call per lane per 8 queries.  All 32 lanes of the warp take part; lane & 7 must equal
// key & 7.
template <int kOctets>
__device__ __forceinline__ uint64_t dropout_key_bits(const DropoutParams& dp, int key, int qb, int bh, int lane) {
  static_assert(kOctets % 2 == 0 && kOctets <= 8, "up to 64 queries, in pairs of octets");
  const uint32_t u = uint32_t(lane & 7);
  const uint32_t g = uint32_t(key) >> 3;
  uint64_t out = 0;
#pragma unroll
  for (int b = 0; b < kOctets; b += 2) {
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      // row u of this octet's 8 x 8 bit block: keep bits of keys 8g .. 8g+7 for query 8(b+bb) + u
      const uint32_t row = dropout_keep8(dp, g, uint32_t(qb + 8 * (b + bb)) + u, uint32_t(bh));
      uint32_t x = row << (8 * (u & 3));
      x |= __shfl_xor_sync(0xffffffffu, x, 1);
      x |= __shfl_xor_sync(0xffffffffu, x, 2);  // rows of this quad of lanes
      const uint32_t y = __shfl_xor_sync(0xffffffffu, x, 4);
      const uint32_t lo = u < 4 ? x : y;      // rows 0-3, one per byte
      const uint32_t hi = u < 4 ? y : x;      // rows 4-7
      // column u: bit u of every byte, gathered into a nibble (the four products land on
      // distinct bits 24..27, so no carries)
      const uint32_t nlo = (((lo >> u) & 0x01010101u) * 0x01020408u) >> 24;
      const uint32_t nhi = (((hi >> u) & 0x01010101u) * 0x01020408u) >> 24;
      out |= uint64_t(nlo | (nhi << 4)) << (8 * (b + bb));
    }
  }
  return out;
}

}  // namespace fa
