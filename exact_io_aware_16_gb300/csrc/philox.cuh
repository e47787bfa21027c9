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
// before the product with V): element (i, j) of head bh is kept iff word
// j mod 4 of Philox(counter = (j / 4, i, bh, offset), key = seed) is at least
// thr = floor(p * 2^32); kept probabilities are scaled by 1 / (1 - p).
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
  uint32_t thr = 0;                  // keep iff word >= thr
  float rs = 1.0f;                   // 1 / (1 - p)

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
    const uint32_t hi0 = __umulhi(kMul0, c0), lo0 = kMul0 * c0;
    const uint32_t hi1 = __umulhi(kMul1, c2), lo1 = kMul1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ dr.rk0[r];
    const uint32_t n2 = hi0 ^ c3 ^ dr.rk1[r];
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return make_uint4(c0, c1, c2, c3);
}

// Keep bits of the four elements (i, 4 jg + e), e = 0..3, as bits 0..3.
__device__ __forceinline__ uint32_t keep_nibble(const DropArgs& dr, uint32_t jg, uint32_t i,
                                                uint32_t bh) {
  const uint4 w = philox4x32_10(jg, i, bh, dr.offset, dr);
  return static_cast<uint32_t>(w.x >= dr.thr) | (static_cast<uint32_t>(w.y >= dr.thr) << 1) |
         (static_cast<uint32_t>(w.z >= dr.thr) << 2) | (static_cast<uint32_t>(w.w >= dr.thr) << 3);
}

// Keep bits, transposed across a warp: lane L holds key row jrow (four
// consecutive lanes hold four consecutive keys starting at a multiple of 4)
// and wants the decisions for query rows i0 .. i0+3.  Each lane computes one
// counter (its quad's key group, row i0 + L % 4) and four ballots hand every
// lane its own key's column of the 4 x 4 block.  Returns the keep bits of
// rows i0 + r as bits r = 0..3.  All 32 lanes must call it together.
__device__ __forceinline__ uint32_t keep_nibble_t(const DropArgs& dr, uint32_t jrow, uint32_t i0,
                                                  uint32_t bh, int lane) {
  const uint32_t r = static_cast<uint32_t>(lane) & 3u;
  const uint4 w = philox4x32_10(jrow >> 2, i0 + r, bh, dr.offset, dr);
  const uint32_t b0 = __ballot_sync(0xffffffffu, w.x >= dr.thr);
  const uint32_t b1 = __ballot_sync(0xffffffffu, w.y >= dr.thr);
  const uint32_t b2 = __ballot_sync(0xffffffffu, w.z >= dr.thr);
  const uint32_t b3 = __ballot_sync(0xffffffffu, w.w >= dr.thr);
  const uint32_t mine = r == 0 ? b0 : (r == 1 ? b1 : (r == 2 ? b2 : b3));
  return (mine >> (static_cast<uint32_t>(lane) & ~3u)) & 0xFu;
}

}  // namespace fa
