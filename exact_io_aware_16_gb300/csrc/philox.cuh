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

// Calls that share three counter words.  In the first rounds some products
// depend on the shared words alone; they are formed once (the *_init
// functions) and every call then does the rest of the rounds as above.  The
// results are those of philox4x32_10, bit for bit.
//
// PhiloxRow: counter words 1..3 (query row i, bh, offset) shared, word 0 (the
// key group) varying.  Round 0's second product (kMul1 * bh) and round 1's
// first product (kMul0 * word 0 after round 0) are shared: 18 of the 20
// multiplies remain per call.
struct PhiloxRow {
  uint32_t c0_1;  // word 0 after round 0
  uint32_t c1_1;  // word 1 after round 0
  uint32_t h2, l2;  // halves of round 1's first product, kMul0 * c0_1
};

__host__ __device__ __forceinline__ PhiloxRow philox_row_init(const DropArgs& dr, uint32_t i,
                                                              uint32_t bh) {
  constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
  const uint64_t p1 = static_cast<uint64_t>(kMul1) * bh;
  PhiloxRow r;
  r.c0_1 = static_cast<uint32_t>(p1 >> 32) ^ i ^ dr.rk0[0];
  r.c1_1 = static_cast<uint32_t>(p1);
  const uint64_t p2 = static_cast<uint64_t>(kMul0) * r.c0_1;
  r.h2 = static_cast<uint32_t>(p2 >> 32);
  r.l2 = static_cast<uint32_t>(p2);
  return r;
}

// The ten rounds from round `first` on, counter (c0..c3) after round first - 1.
__host__ __device__ __forceinline__ uint4 philox_rounds_from(int first, uint32_t c0, uint32_t c1,
                                                            uint32_t c2, uint32_t c3,
                                                            const DropArgs& dr) {
  constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
#pragma unroll
  for (int r = 0; r < kPhiloxRounds; ++r) {
    if (r < first) continue;
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

// philox4x32_10(jg, i, bh, dr.offset) with r = philox_row_init(dr, i, bh).
__host__ __device__ __forceinline__ uint4 philox_row_call(const DropArgs& dr, const PhiloxRow& r,
                                                         uint32_t jg) {
  constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
  const uint64_t p0 = static_cast<uint64_t>(kMul0) * jg;  // round 0
  const uint32_t c2_1 = static_cast<uint32_t>(p0 >> 32) ^ dr.offset ^ dr.rk1[0];
  const uint32_t c3_1 = static_cast<uint32_t>(p0);
  const uint64_t p1 = static_cast<uint64_t>(kMul1) * c2_1;  // round 1
  return philox_rounds_from(2, static_cast<uint32_t>(p1 >> 32) ^ r.c1_1 ^ dr.rk0[1],
                            static_cast<uint32_t>(p1), r.h2 ^ c3_1 ^ dr.rk1[1], r.l2, dr);
}

// PhiloxCol: counter words 0, 2, 3 (key group, bh, offset) shared, word 1 (the
// query row) varying.  Both products of round 0, the second of round 1 and the
// first of round 2 are shared: 16 of the 20 multiplies remain per call.
struct PhiloxCol {
  uint32_t k0;      // word 0 after round 0 is k0 ^ i
  uint32_t l0;      // low half of round 0's first product
  uint32_t g;       // word 1 after round 1
  uint32_t h4, l4;  // halves of round 2's first product
};

__host__ __device__ __forceinline__ PhiloxCol philox_col_init(const DropArgs& dr, uint32_t jg,
                                                              uint32_t bh) {
  constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
  const uint64_t p0 = static_cast<uint64_t>(kMul0) * jg;  // round 0
  const uint64_t p1 = static_cast<uint64_t>(kMul1) * bh;
  PhiloxCol c;
  c.k0 = static_cast<uint32_t>(p1 >> 32) ^ dr.rk0[0];
  c.l0 = static_cast<uint32_t>(p0);
  const uint32_t e = static_cast<uint32_t>(p0 >> 32) ^ dr.offset ^ dr.rk1[0];  // word 2
  const uint64_t p3 = static_cast<uint64_t>(kMul1) * e;  // round 1, second product
  c.g = static_cast<uint32_t>(p3);
  const uint32_t f = static_cast<uint32_t>(p3 >> 32) ^ static_cast<uint32_t>(p1) ^ dr.rk0[1];
  const uint64_t p4 = static_cast<uint64_t>(kMul0) * f;  // round 2, first product
  c.h4 = static_cast<uint32_t>(p4 >> 32);
  c.l4 = static_cast<uint32_t>(p4);
  return c;
}

// philox4x32_10(jg, i, bh, dr.offset) with c = philox_col_init(dr, jg, bh).
__host__ __device__ __forceinline__ uint4 philox_col_call(const DropArgs& dr, const PhiloxCol& c,
                                                         uint32_t i) {
  constexpr uint32_t kMul0 = 0xD2511F53u, kMul1 = 0xCD9E8D57u;
  const uint64_t p0 = static_cast<uint64_t>(kMul0) * (c.k0 ^ i);  // round 1
  const uint32_t c2_2 = static_cast<uint32_t>(p0 >> 32) ^ c.l0 ^ dr.rk1[1];
  const uint32_t c3_2 = static_cast<uint32_t>(p0);
  const uint64_t p1 = static_cast<uint64_t>(kMul1) * c2_2;  // round 2
  return philox_rounds_from(3, static_cast<uint32_t>(p1 >> 32) ^ c.g ^ dr.rk0[2],
                            static_cast<uint32_t>(p1), c.h4 ^ c3_2 ^ dr.rk1[2], c.l4, dr);
}

// The two decisions carried by one 32-bit word (low half: even key, high
// half: odd key) as bits 0 and 1.  Comparing the halves moved to the top of
// the word against thr16 << 16 decides them without masking.
__device__ __forceinline__ uint32_t keep_pair(uint32_t w, uint32_t thr_hi) {
  return static_cast<uint32_t>((w << 16) >= thr_hi) | (static_cast<uint32_t>(w >= thr_hi) << 1);
}

// The eight decisions of one generator call's words, as bits 0..7.
__device__ __forceinline__ uint32_t keep8(const uint4& w, uint32_t thr_hi) {
  return keep_pair(w.x, thr_hi) | (keep_pair(w.y, thr_hi) << 2) |
         (keep_pair(w.z, thr_hi) << 4) | (keep_pair(w.w, thr_hi) << 6);
}

// Keep bits of the eight elements (i, 8 jg + e), e = 0..7, as bits 0..7.
__device__ __forceinline__ uint32_t keep_byte(const DropArgs& dr, uint32_t jg, uint32_t i,
                                              uint32_t bh) {
  return keep8(philox4x32_10(jg, i, bh, dr.offset, dr), dr.thr_hi);
}

// The same for the row of r = philox_row_init(dr, i, bh).
__device__ __forceinline__ uint32_t keep_byte_row(const DropArgs& dr, const PhiloxRow& r,
                                                  uint32_t jg) {
  return keep8(philox_row_call(dr, r, jg), dr.thr_hi);
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
// call it together.  pc = philox_col_init(dr, jrow / 8, bh).
__device__ __forceinline__ uint32_t keep_word_t(const DropArgs& dr, const PhiloxCol& pc,
                                                uint32_t i0, int lane) {
  const uint32_t r = static_cast<uint32_t>(lane) & 7u;
  uint32_t x = 0;
#pragma unroll
  for (uint32_t u = 0; u < 4; ++u)
    x |= keep8(philox_col_call(dr, pc, i0 + 8u * u + r), dr.thr_hi) << (8 * u);
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
