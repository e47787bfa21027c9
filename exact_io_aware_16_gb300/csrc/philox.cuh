// philox.cuh — the Philox4x32-10 counter-based generator on the device, and
// the dropout keep decision built on it.
//
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC 2011): a 128-bit counter and a 64-bit key go through
// ten rounds; each round multiplies counter words 0 and 2 by two fixed odd
// 32-bit constants, keeps both halves of each 64-bit product, XORs the high
// halves with the other two words and the round key, and permutes the words;
// the key is bumped by two Weyl constants between rounds.
//
// Dropout on P (the talk's dropout applied to the attention probabilities
// before the product with V): one Philox call, counter = (j / 8, i, bh,
// offset) and key = seed, decides eight consecutive keys of row i; key j
// takes the low (even j) or high (odd j) 16 bits of word (j / 2) mod 4 and is
// kept iff they are at least thr16 = floor(p * 2^16).  Kept probabilities are
// scaled by the inverse keep probability 65536 / (65536 - thr16).
#pragma once

#include <cstdint>

namespace fa {

constexpr int kPhiloxRounds = 10;

// Kernel parameter block of dropout.  The round keys are expanded on the
// host (set_seed), so the kernels read them from the parameter bank instead
// of keeping twenty derived values in registers.
struct DropArgs {
  uint32_t rk0[kPhiloxRounds] = {};  // round r key word 0: seed_lo + r * 0x9E3779B9
  uint32_t rk1[kPhiloxRounds] = {};  // round r key word 1: seed_hi + r * 0xBB67AE85
  uint32_t offset = 0;               // counter word 3
  uint32_t thr_hi = 0;               // thr16 << 16: keep iff the 16 bits, moved up, are >= it
  float rs = 1.0f;                   // 65536 / (65536 - thr16)

  __host__ __device__ void set_seed(uint32_t k0, uint32_t k1) {
    for (int r = 0; r < kPhiloxRounds; ++r) {
      rk0[r] = k0 + 0x9E3779B9u * static_cast<uint32_t>(r);
      rk1[r] = k1 + 0xBB67AE85u * static_cast<uint32_t>(r);
    }
  }
};

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                               uint32_t c3, const DropArgs& dr) {
  constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
#pragma unroll
  for (int r = 0; r < kPhiloxRounds; ++r) {
    // one 32 x 32 -> 64-bit multiply per product gives both halves
    const uint64_t p0 = static_cast<uint64_t>(kMul0) * c0;
    const uint64_t p1 = static_cast<uint64_t>(kMul1) * c2;
    const uint32_t n0 = static_cast<uint32_t>(p1 >> 32) ^ c1 ^ dr.rk0[r];
    const uint32_t n2 = static_cast<uint32_t>(p0 >> 32) ^ c3 ^ dr.rk1[r];
    c0 = n0;
    c1 = static_cast<uint32_t>(p1);
    c2 = n2;
    c3 = static_cast<uint32_t>(p0);
  }
  return make_uint4(c0, c1, c2, c3);
}

// The two decisions carried by one 32-bit word (low half: even key, high
// half: odd key) as bits 0 and 1.  Comparing the halves moved to the top of
// the word against thr16 << 16 decides them without masking.
__device__ __forceinline__ uint32_t keep_pair(uint32_t w, uint32_t thr_hi) {
  return static_cast<uint32_t>((w << 16) >= thr_hi) | (static_cast<uint32_t>(w >= thr_hi) << 1);
}

// Keep bits of the eight elements (i, 8 jg + e), e = 0..7, as bits 0..7.
__device__ __forceinline__ uint32_t keep_byte(const DropArgs& dr, uint32_t jg, uint32_t i,
                                              uint32_t bh) {
  const uint4 w = philox4x32_10(jg, i, bh, dr.offset, dr);
  return keep_pair(w.x, dr.thr_hi) | (keep_pair(w.y, dr.thr_hi) << 2) |
         (keep_pair(w.z, dr.thr_hi) << 4) | (keep_pair(w.w, dr.thr_hi) << 6);
}

// Keep bits, transposed across a warp: lane L holds key row jrow (eight
// consecutive lanes hold eight consecutive keys starting at a multiple of 8)
// and wants the decisions for query rows i0 .. i0+31.  Each lane computes four
// counters (its octet's key group, rows i0 + 8u + L % 8 for u = 0..3): byte u
// of its word is then row L % 8 of an 8 x 8 bit block (bit c: key 8m + c).
// Three XOR-shuffle butterfly stages transpose all four blocks of the octet at
// once (stage b swaps the off-diagonal b x b sub-blocks between lanes b
// apart; the masks keep the bytes apart), leaving in byte u of lane L the
// column L % 8 of block u: bit k = row i0 + 8u + k of this lane's key.
// Returns the keep bits of rows i0 + t as bits t = 0..31.  All 32 lanes must
// call it together.
__device__ __forceinline__ uint32_t keep_word_t(const DropArgs& dr, uint32_t jrow, uint32_t i0,
                                                uint32_t bh, int lane) {
  const uint32_t r = static_cast<uint32_t>(lane) & 7u;
  uint32_t x = 0;
#pragma unroll
  for (uint32_t u = 0; u < 4; ++u) x |= keep_byte(dr, jrow >> 3, i0 + 8u * u + r, bh) << (8 * u);
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    const int b = 4 >> s;
    const uint32_t lo = s == 0 ? 0x0F0F0F0Fu : (s == 1 ? 0x33333333u : 0x55555555u);
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, b);
    x = (lane & b) ? ((x & ~lo) | ((y >> b) & lo)) : ((x & lo) | ((y << b) & ~lo));
  }
  return x;
}

}  // namespace fa
