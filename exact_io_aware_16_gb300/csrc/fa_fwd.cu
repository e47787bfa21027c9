// fa_fwd.cu — fused exact-attention forward for sm_103a.
//
// One CTA computes two 128-row query tiles (a "pair") of one (batch, head):
//   * "What is Flash Attention?" 03:44-04:15 (tiling): both Q tiles are
//     loaded once and stay in shared memory while 128-row K and V tiles
//     stream through a two-stage ring (TMA, 128-byte swizzle); every K/V tile
//     serves both Q tiles.
//   * "Atencao exata ..." block-score formula S_ij = Q_i K_j^T / sqrt(d):
//     tcgen05.mma writes each 128 x 128 fp32 score tile into tensor memory.
//   * transcript 04:46-05:17 (online softmax): one warpgroup per Q tile, one
//     thread per query row (= one TMEM lane), keeps the running max m (log2
//     units of the scaled scores) and running sum l, writes
//     P~ = 2^(s*scale*log2e - m) as bf16 back over its score row, and
//     rescales the O accumulator by alpha = 2^(m_old - m_new).  The running max
//     is moved lazily: a tile's exponentials are first taken against the
//     current running max, and only when some row's P~ would exceed a bound
//     (2^16 for bf16 P~, 2^7 for e4m3) is the tile redone against a new max
//     (moved when the block max exceeds the running max by more than 8, log2
//     units); since O and l carry the same factor, O / l is unchanged.  beta
//     of the page is folded in by exponentiating against the current max
//     directly (the "l_new" formula of the mentria page).
//   * O += P~ V_j is a tcgen05.mma with the P~ operand read from tensor
//     memory and V from shared memory; O stays in tensor memory (fp32).
//   * 06:52-07:24: at the end only O = O_acc / l (bf16) and one fp32
//     statistic per row, lse = (m + log2 l) ln 2, are written.
//   * causal masking ("FlashAttention ..." talk, optional masking): query
//     tile i visits key tiles 0..i only; the mask is applied inside the
//     diagonal tile, so whole tiles above the diagonal are never loaded.
//   * dropout (the talk's dropout on P, fused with the softmax): with
//     DROPOUT each thread draws the keep bits of its row for the next key
//     tile from Philox4x32-10 (philox.cuh) while the tensor core computes the
//     scores, zeroes dropped entries of P~ before the P V product (the row
//     sum l keeps them: lse is that of P), and scales O by the inverse keep
//     probability at the end.
//
// Ping-pong schedule of the MMA warp for key tile j:
//     PV0_j, S0_{j+1}, PV1_j, S1_{j+1}
// so while warpgroup 0 turns S0 into P0 the tensor core runs PV1 and S1, and
// the other way round.  Committing S_g(j+1) also guarantees that PV_g(j) has
// completed, so a warpgroup that has seen its scores may rescale O at once.
//
// Warp roles (320 threads): warps 0-3 tile 0 and warps 4-7 tile 1
// (softmax / correction / epilogue; thread t <-> row t <-> TMEM lane t),
// warp 8 TMA producer, warp 9 TMEM allocator and MMA issuer.
#include <algorithm>
#include <mutex>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "philox.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

__device__ unsigned int g_fwd_error;

// Work-item counters of persistent launches: each launch claims one slot
// (the host hands them out in turn), its CTAs take items with atomicAdd on
// slot[0], and the last CTA to finish (slot[1] counts them) zeroes the slot
// again.  fa_fwd_reset_sched zeroes every slot after a device error, since an
// aborted launch may leave its slot dirty.
__device__ unsigned int g_fwd_sched[kSchedSlots][2];
constexpr int kItemRing = 4;  // claimed items in flight between the roles of a CTA


constexpr int kFwdThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStages = 2;

// Ring slot and phase parity of the K / V tile at ring position pos >= 0
// (unsigned: kStages is a power of two, so these are a mask and a shift).
__device__ __forceinline__ int ring_slot(int pos) {
  return static_cast<int>(static_cast<unsigned>(pos) % kStages);
}
__device__ __forceinline__ uint32_t ring_phase(int pos) {
  return (static_cast<unsigned>(pos) / kStages) & 1u;
}
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLazyRescaleLog2 = 8.0f;
// A speculative tile (exponentials against the running max, before the block
// max is known) is accepted when every row's sum of P~ is at most this bound,
// so that every P~ is too.  e4m3 P~ must stay below 448: 2^7.  bf16 P~ and
// the fp32 O and l accumulators are unharmed by P~ up to 2^16 (bf16 rounding
// is relative, and O and l carry the same factor), so a bf16 tile is accepted
// up to 2^16; a row's running max then trails its true max by at most 16
// (log2) instead of 8, and O / l is the same up to rounding.
constexpr float kSpeculateSumBoundF8 = 128.0f;
constexpr float kSpeculateSumBound = 65536.0f;

// EB: bytes per element of Q, K, V (2: bf16, 1: e4m3).  A tile is 128 rows;
// every 128-byte run of a row is one swizzled TMA box column ("chunk").
template <int D, int EB = 2>
struct FwdLayout {
  static constexpr int kChunks = D * EB / 128;
  static constexpr uint32_t kTileBytes = 128u * D * EB;
  static constexpr uint32_t kQ = 0;  // two Q tiles
  static constexpr uint32_t kK = kQ + 2 * kTileBytes;
  static constexpr uint32_t kV = kK + kStages * kTileBytes;
  static constexpr uint32_t kBar = kV + kStages * kTileBytes;
  static constexpr uint32_t kList = kBar + 256;  // block-sparse key-tile list (uint16)
  static constexpr uint32_t kSmemUsed = kList + 2 * kMaxSparseTiles + 1024;  // + align slack
  // at least 116 KB, so two CTAs never share an SM (each takes all 512 TMEM columns)
  static constexpr uint32_t kSmem = kSmemUsed > 118784u ? kSmemUsed : 118784u;
  static constexpr uint32_t kTmemCols = 512;            // S0, S1, O0, O1
  __host__ __device__ static constexpr uint32_t s_col(int g) { return 128u * g; }
  __host__ __device__ static constexpr uint32_t o_col(int g) { return 256u + D * g; }
};

struct FwdBars {
  uint64_t q_full;
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_ready[2], pv_done[2];
  uint64_t q_empty;    // the S products of an item are done with the Q tiles
  uint64_t item_full[kItemRing];  // the producer has claimed the item of this ring entry
  uint64_t o_free[2];  // softmax warpgroup g has read its O for the epilogue
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int nlist;  // block-sparse: entries of the key-tile list
  int item_ring[kItemRing];  // claimed items (-1: no more)
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, FwdBars* b,
                                          uint32_t code) {
  bool ok = mbar_wait(bar, parity, &b->abort_flag, &g_fwd_error, code);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool mma_wait(uint64_t* bar, uint32_t parity, FwdBars* b,
                                         uint32_t code) {
  return mbar_wait(bar, parity, &b->abort_flag, &g_fwd_error, code);
}

// SPARSE: the pair visits only the key tiles that at least one of its two
// query tiles keeps in the block mask (bmask[bh * mstride + qt * nk + kt] != 0,
// 128 x 128 tiles).  Warp 0 compacts them into a list in shared memory
// (entry = key tile | keep-by-tile-0 << 14 | keep-by-tile-1 << 15); for each
// list entry both query tiles compute their scores, and a query tile that
// does not keep the key tile masks all of it to -inf.
//
// FP8: Q, K and V are e4m3 (V transposed per head, [d][N], so that both
// products read K-major operands); S = Q K^T and O += P V are
// tcgen05.mma.kind::f8f6f4 (K = 32 per instruction), P~ is rounded to e4m3
// into tensor memory as the A operand of P V, and o_scale (the V descale)
// multiplies O in the epilogue.  The Q and K descales are folded into
// scale_log2 by the caller.
template <int D, bool CAUSAL, bool SPARSE, bool DROPOUT, bool FP8, bool PERSIST>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, __nv_bfloat16* __restrict__ o,
                  float* __restrict__ lse, int BH, int N, float scale_log2,
                  const uint8_t* __restrict__ bmask, long long mstride, DropArgs drop,
                  float o_scale, unsigned int* __restrict__ sched, int group_heads) {
  static_assert(!FP8 || (D == 128 && !SPARSE && !DROPOUT), "e4m3 path: d = 128, dense");
  static_assert(!(PERSIST && SPARSE), "block-sparse items each have their own CTA");
  using L = FwdLayout<D, FP8 ? 1 : 2>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  FwdBars* bars = reinterpret_cast<FwdBars*>(smem + L::kBar);
  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nq = (N + kTileM - 1) / kTileM;
  const int nk = (N + kTileN - 1) / kTileN;
  const int npairs = (nq + 1) / 2;
  // Work items: one pair of query tiles of one (b, h), numbered in the order
  // they are handed out (item_pair / item_bh below).
  const int n_items = BH * npairs;
  // PERSIST: persistent CTAs (one per SM) claim items in the order above from
  // the launch's counter slot: the TMA warp claims them and publishes each
  // through a small ring in shared memory to the MMA warp and the softmax
  // warpgroups, and the next item's loads and first score product overlap
  // the current item's epilogue.  Otherwise every item has its own CTA (item
  // blockIdx.x; block-sparse calls build its tile list before the roles
  // split).
  constexpr bool kPersist = PERSIST;
  // Items come in groups of group_heads heads (all pairs of those heads);
  // within a group pair-major, the heaviest pair (4p + 3 key tiles when
  // causal) of every head first.  Handing them out in order (the block
  // scheduler, or the persistent CTAs' counter) then balances the SMs like
  // longest-job-first, while the K / V tiles a group reads at once stay
  // within L2 (the launcher sizes the group; 1 = head-major, for the equal
  // non-causal items).
  auto item_group = [&](int item) { return item / (group_heads * npairs); };
  auto item_rank = [&](int item, int& head) {  // rank of the pair in its group, heaviest first
    const int grp = item_group(item);
    const int gs = min(group_heads, BH - grp * group_heads);
    const int r = item - grp * group_heads * npairs;
    head = grp * group_heads + r % gs;
    return r / gs;
  };
  auto item_pair = [&](int item) {
    int head;
    return npairs - 1 - item_rank(item, head);
  };
  auto item_bh = [&](int item) {
    int head;
    item_rank(item, head);
    return head;
  };
  // key tiles visited by query tile 2*pair + g
  auto item_nkv = [&](int item, int g) {
    return CAUSAL ? min(2 * item_pair(item) + 1 + g, nk) : nk;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&bars->s_full[g], 1);
      mbar_init(&bars->p_ready[g], 128);
      mbar_init(&bars->pv_done[g], 1);
      mbar_init(&bars->o_free[g], 128);
    }
    mbar_init(&bars->q_empty, 1);
    for (int r = 0; r < kItemRing; ++r) mbar_init(&bars->item_full[r], 1);
    mbar_init(&bars->drain, 1);
    // an earlier CTA already recorded a pipeline timeout: exit without work
    bars->abort_flag = (*static_cast<volatile unsigned int*>(&g_fwd_error) != 0) ? 1 : 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (bars->abort_flag) return;
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::kList);
  if (SPARSE && warp == 0) {
    const int pair = item_pair(blockIdx.x), bh = item_bh(blockIdx.x);
    const uint8_t* m0 = bmask + bh * mstride + static_cast<long long>(2 * pair) * nk;
    const bool has1 = 2 * pair + 1 < nq;  // the pair's second tile may lie past N
    int count = 0;
    for (int base = 0; base < nk; base += 32) {
      const int j = base + lane;
      bool u0 = false, u1 = false;
      if (j < nk) {
        u0 = m0[j] != 0 && (!CAUSAL || j <= 2 * pair);
        u1 = has1 && m0[nk + j] != 0 && (!CAUSAL || j <= 2 * pair + 1);
      }
      const unsigned bal = __ballot_sync(0xffffffffu, u0 || u1);
      if (u0 || u1)
        list[count + __popc(bal & ((1u << lane) - 1u))] =
            static_cast<uint16_t>(j | (u0 ? 1 << 14 : 0) | (u1 ? 1 << 15 : 0));
      count += __popc(bal);
    }
    if (lane == 0) bars->nlist = count;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  // number of list positions each query tile of an item runs through (a
  // prefix of the pair's list), and the key tile at a position
  auto item_n = [&](int item, int g) { return SPARSE ? bars->nlist : item_nkv(item, g); };
  auto kv_of = [&](int p) -> int { return SPARSE ? (list[p] & 0x3FFF) : p; };
  // The t-th item of this CTA as the consumers see it (-1: no more).  `wait`
  // is the role's bounded wait on the ring entry.
  auto consumer_item = [&](int t, auto&& wait) -> int {
    if (!kPersist) return t == 0 ? static_cast<int>(blockIdx.x) : -1;
    if (!wait(&bars->item_full[t % kItemRing], (t / kItemRing) & 1)) return -1;
    return bars->item_ring[t % kItemRing];
  };

  if (warp == kTmaWarp) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int kvb = 0;  // K / V tiles loaded for earlier items (ring position)
      bool ok = true;
      for (int t = 0; ok; ++t) {
        // claim the next item and publish it to the other roles
        int item;
        if (kPersist) {
          const unsigned int c = atomicAdd(&sched[0], 1u);
          item = c < static_cast<unsigned int>(n_items) ? static_cast<int>(c) : -1;
          bars->item_ring[t % kItemRing] = item;
          mbar_arrive(&bars->item_full[t % kItemRing]);
        } else {
          item = t == 0 ? static_cast<int>(blockIdx.x) : -1;
        }
        if (item < 0) break;
        const int pair = item_pair(item), bh = item_bh(item);
        const int n1 = item_n(item, 1);
        auto load_q = [&]() {
          mbar_arrive_expect_tx(&bars->q_full, 2 * L::kTileBytes);
#pragma unroll
          for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_3d(smem + L::kQ + g * L::kTileBytes + c * 16384, &tq, &bars->q_full,
                          c * 64, (2 * pair + g) * kTileM, bh);
        };
        // a CTA's first item: Q right away; later items: the first K tile
        // first (its ring slot is free early), then Q once the previous item's
        // score products are done with the Q buffer
        if (t == 0 && n1 > 0) load_q();
        for (int j = 0; j < n1; ++j) {
          const int s = ring_slot(kvb + j);
          const uint32_t ph = ring_phase(kvb + j);
          const int kt = kv_of(j);
          if (!mbar_wait(&bars->k_empty[s], ph ^ 1, &bars->abort_flag, &g_fwd_error, 0x101)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->k_full[s], L::kTileBytes);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(smem + L::kK + s * L::kTileBytes + c * 16384, &tk, &bars->k_full[s],
                        c * 64, kt * kTileN, bh);
          if (j == 0 && t > 0) {
            if (!mbar_wait(&bars->q_empty, (t - 1) & 1, &bars->abort_flag, &g_fwd_error, 0x103)) {
              ok = false;
              break;
            }
            load_q();
          }
          if (!mbar_wait(&bars->v_empty[s], ph ^ 1, &bars->abort_flag, &g_fwd_error, 0x102)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->v_full[s], L::kTileBytes);
          if (FP8) {  // V^T tile: d rows of 128 keys
            tma_load_3d(smem + L::kV + s * L::kTileBytes, &tv, &bars->v_full[s], kt * kTileN, 0,
                        bh);
          } else {
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_3d(smem + L::kV + s * L::kTileBytes + c * 16384, &tv, &bars->v_full[s],
                          c * 64, kt * kTileN, bh);
          }
        }
        kvb += n1;
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
      constexpr uint32_t idesc_f8 = idesc_e4m3_f32(128, 128);
      // S_g = Q_g K^T from the K tile at ring position pos (no commit)
      auto issue_s = [&](int g, int pos) {
        const uint32_t kbase = sK + ring_slot(pos) * L::kTileBytes;
        const uint32_t qbase = sQ + g * L::kTileBytes;
        if (FP8) {  // K = 32 e4m3 = 32 bytes per instruction, one 128-byte chunk
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            umma_ss_f8(tmem + L::s_col(g), sdesc_sw128(qbase + kk * 32, 16, 1024),
                       sdesc_sw128(kbase + kk * 32, 16, 1024), idesc_f8, kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            umma_ss(tmem + L::s_col(g), sdesc_sw128(qbase + off, 16, 1024),
                    sdesc_sw128(kbase + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          }
        }
      };
      // O_g (+)= P_g V from the V tile at ring position pos; `first` starts O
      // afresh (no commit)
      auto issue_pv = [&](int g, int pos, bool first) {
        const uint32_t vbase = sV + ring_slot(pos) * L::kTileBytes;
        if (FP8) {  // A = P~ e4m3, 8 tensor-memory columns per 32 keys; B = V^T K-major
#pragma unroll
          for (int kk = 0; kk < kTileN / 32; ++kk)
            umma_ts_f8(tmem + L::o_col(g), tmem + L::s_col(g) + kk * 8,
                       sdesc_sw128(vbase + kk * 32, 16, 1024), idesc_f8,
                       (!first || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            umma_ts(tmem + L::o_col(g), tmem + L::s_col(g) + kk * 8,
                    sdesc_sw128(vbase + kk * 2048, 16384, 1024), idesc_pv,
                    (!first || kk > 0) ? 1u : 0u);
        }
      };
      // One item: t = items before it in this CTA, kvb = its first K / V ring
      // position, base0 / base1 = tiles each softmax warpgroup finished before
      // it.  Returns false after a pipeline timeout.
      //
      // For key tile j the products go out in two bursts, PV0_j S0_{j+1} and
      // PV1_j S1_{j+1}, each preceded by the waits for everything it reads,
      // so that no wait sits between the two products of a burst: a blocking
      // wait of this thread between products leaves the tensor core idle
      // after the earlier ones complete.  Group 1's P is usually ready by the
      // time group 0's burst has gone out, so it is first tested without
      // blocking, and when it is ready its burst follows at once.
      auto mma_item = [&](const int item, const int t, const int kvb, const int base0,
                          const int base1) -> bool {
        const int n0 = item_n(item, 0), n1 = item_n(item, 1);
        if (n1 == 0) return true;  // block-sparse item without key tiles (its only item)
        bool ok = mma_wait(&bars->q_full, t & 1, bars, 0x201) &&
             mma_wait(&bars->k_full[ring_slot(kvb)], ring_phase(kvb), bars, 0x202);
        if (!ok) return false;
        tc_fence_after_sync();
        issue_s(0, kvb);
        umma_commit(&bars->s_full[0]);
        issue_s(1, kvb);
        umma_commit(&bars->s_full[1]);
        umma_commit(&bars->k_empty[ring_slot(kvb)]);
        for (int j = 0; j < n1; ++j) {
          const int pos = kvb + j;
          const int s = ring_slot(pos);
          const uint32_t ph = ring_phase(pos);
          const int sn = ring_slot(pos + 1);
          const uint32_t phn = ring_phase(pos + 1);
          bool pre1 = false;
          if (j < n0) {
            // burst of group 0: P0_j, V_j, and K_{j+1} for S0_{j+1} (or for
            // S1_{j+1} alone when group 0 ends here)
            ok = mma_wait(&bars->p_ready[0], (base0 + j) & 1, bars, 0x203) &&
                 mma_wait(&bars->v_full[s], ph, bars, 0x204) &&
                 (j > 0 || t == 0 || mma_wait(&bars->o_free[0], (t - 1) & 1, bars, 0x209)) &&
                 (j + 1 >= n1 || mma_wait(&bars->k_full[sn], phn, bars, 0x205));
            if (!ok) break;
            tc_fence_after_sync();
            issue_pv(0, pos, j == 0);
            umma_commit(&bars->pv_done[0]);
            if (j + 1 < n0) issue_s(0, pos + 1);
            pre1 = mbar_test_wait(&bars->p_ready[1], (base1 + j) & 1) &&
                   (j > 0 || t == 0 || mbar_test_wait(&bars->o_free[1], (t - 1) & 1));
            if (j + 1 < n0) umma_commit(&bars->s_full[0]);
          }
          // burst of group 1: P1_j (V_j and K_{j+1} are in when group 0 had
          // this tile)
          if (!pre1) {
            ok = mma_wait(&bars->p_ready[1], (base1 + j) & 1, bars, 0x206) &&
                 (j < n0 || mma_wait(&bars->v_full[s], ph, bars, 0x207)) &&
                 (j > 0 || t == 0 || mma_wait(&bars->o_free[1], (t - 1) & 1, bars, 0x20a)) &&
                 (j < n0 || j + 1 >= n1 || mma_wait(&bars->k_full[sn], phn, bars, 0x208));
            if (!ok) break;
          }
          tc_fence_after_sync();
          issue_pv(1, pos, j == 0);
          umma_commit(&bars->v_empty[s]);
          if (j + 1 < n1) issue_s(1, pos + 1);
          umma_commit(&bars->pv_done[1]);
          if (j + 1 < n1) {
            umma_commit(&bars->s_full[1]);
            umma_commit(&bars->k_empty[sn]);
          }
        }
        // every score product of the item has been issued: the Q tiles are
        // free once they complete
        umma_commit(&bars->q_empty);
        return ok;
      };
      if (kPersist) {
        auto mwait = [&](uint64_t* bar, uint32_t par) { return mma_wait(bar, par, bars, 0x20b); };
        int kvb = 0, base0 = 0, base1 = 0;
        for (int t = 0;; ++t) {
          const int item = consumer_item(t, mwait);
          if (item < 0 || !mma_item(item, t, kvb, base0, base1)) break;
          kvb += item_n(item, 1);
          base0 += item_n(item, 0);
          base1 += item_n(item, 1);
        }
      } else {
        mma_item(static_cast<int>(blockIdx.x), 0, 0, 0, 0);
      }
      umma_commit(&bars->drain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warpgroups
    const int g = warp >> 2;           // which query tile of the pair
    const int t = threadIdx.x & 127;   // row within the tile, TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t scol = tmem + lane_off + L::s_col(g);
    const uint32_t ocol = tmem + lane_off + L::o_col(g);
    // one item of this warpgroup; tb = tiles it finished in earlier items
    // (barrier phases).  Returns false after a pipeline timeout.
    auto softmax_item = [&](const int item, const int tb) -> bool {
    bool ok = true;
    const int pair = item_pair(item), bh = item_bh(item);
    const int row = (2 * pair + g) * kTileM + t;
    const int nkv = item_n(item, g);
    const int q0 = (2 * pair + g) * kTileM;
    // the generator's products that depend on this row's counter words alone
    const PhiloxRow prow = DROPOUT ? philox_row_init(drop, static_cast<uint32_t>(row),
                                                     static_cast<uint32_t>(bh))
                                   : PhiloxRow{};
    float m_run = -INFINITY;  // running (lazily moved) max of s * scale * log2(e)
    float l_run = 0.0f;
    for (int j = 0; j < nkv; ++j) {
      // dropout keep bits of this row for the 128 keys of the tile (bit c of
      // kb[c / 32] for key kv0 + c), drawn before the scores are waited for
      uint32_t kb[4] = {0u, 0u, 0u, 0u};
      if (DROPOUT) {
        const uint32_t jg0 = static_cast<uint32_t>(kv_of(j) * kTileN) >> 3;
        // four words of keep bits, four generator calls (interleaved) per
        // word; a rolled outer loop keeps the code small (fully unrolled, the
        // sixteen calls cost instruction-fetch stalls: 620 against 677 TFLOP/s
        // for the 8K causal forward at p = 0.1); each word enters at kb[3] and
        // moves down, so the array is never indexed at run time
#pragma unroll 1
        for (int w = 0; w < 4; ++w) {
          uint32_t acc = 0;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            acc |= keep_byte_row(drop, prow, jg0 + 4 * w + u) << (8 * u);
          kb[0] = kb[1]; kb[1] = kb[2]; kb[2] = kb[3]; kb[3] = acc;
        }
        reg_pin(kb);  // drawn here, before the wait, not next to their use
      }
      if (!warp_wait(&bars->s_full[g], (tb + j) & 1, bars, 0x301)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t sr[128];
      const int kv0 = kv_of(j) * kTileN;
      // a key tile this query tile does not keep: every score is masked
      const bool keep = !SPARSE || ((list[j] >> (14 + g)) & 1);
      const bool need_mask = !keep || (CAUSAL && kv0 + kTileN - 1 > q0) || (kv0 + kTileN > N);
      // this row's 128 scores from tensor memory, masked where needed
      auto load_scores = [&]() {
        tmem_ld32(scol + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld32(scol + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
        tmem_ld32(scol + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
        tmem_ld_wait();
        reg_pin(sr);
        if (need_mask) {
          const int lim_causal = CAUSAL ? (row - kv0) : 0x7fffffff;  // col index <= lim visible
          const int lim_n = N - 1 - kv0;
          const int lim = keep ? (lim_causal < lim_n ? lim_causal : lim_n) : -1;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > lim) sr[c] = __float_as_uint(-INFINITY);
        }
      };
      load_scores();
      // Once the rows have a finite running max, the tile's exponentials are
      // first taken against it without looking at the block max (the row max
      // is off the common path).  If every row's sum of P~ is then within the
      // bound (kSpeculateSumBound, e4m3: kSpeculateSumBoundF8), so is every
      // P~, and the tile stands.  Otherwise (rare) it is redone the exact way:
      // scores reloaded, block max, and the running max moved when some row's
      // block max exceeds it by more than 8 (log2 units, kLazyRescaleLog2).
      float sum = 0.0f;
      // exponentials of this row's scores against the running max (P~ packed
      // into sr) and their sum
      auto exp_tile = [&]() {
        const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
        // exponent arguments and row sums two lanes at a time (packed fp32 FMA / add)
        const float2 sc2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(-m_use, -m_use);
        float2 sp[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};  // partial row sums
        if (FP8) {
          // P~ as e4m3, four per word: quad c overwrites sr[c], already consumed
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x01 = __ffma2_rn(
                make_float2(__uint_as_float(sr[4 * c]), __uint_as_float(sr[4 * c + 1])), sc2, nm2);
            const float2 x23 = __ffma2_rn(
                make_float2(__uint_as_float(sr[4 * c + 2]), __uint_as_float(sr[4 * c + 3])), sc2,
                nm2);
            const float2 p01 = make_float2(ex2_approx(x01.x), ex2_approx(x01.y));
            const float2 p23 = make_float2(ex2_approx(x23.x), ex2_approx(x23.y));
            sp[(2 * c) & 3] = __fadd2_rn(sp[(2 * c) & 3], p01);
            sp[(2 * c + 1) & 3] = __fadd2_rn(sp[(2 * c + 1) & 3], p23);
            sr[c] = pack_e4m3x4(p01.x, p01.y, p23.x, p23.y);
          }
        } else {
          // P~ packed in place: pair c overwrites sr[c], already consumed.  The
          // row sum adds each pair (p0 + p1) into partial sum (c / 2) % 4, x for
          // even c and y for odd c.  Two pairs at a time, with packed fma / add
          // (each lane rounded as the scalar op, so the sums are the same bit
          // for bit), except in the persistent causal d = 128 kernel, whose item
          // state leaves no registers for them (it spilled and ran 8 % slower at
          // N = 2048; the dropout kernels spill a little too but gain 2.5 %).
          constexpr bool kPairs = !(PERSIST && CAUSAL && D == 128);
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float p[4];
            if (kPairs) {
              const float2 x0 = __ffma2_rn(
                  make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc2, nm2);
              const float2 x1 = __ffma2_rn(
                  make_float2(__uint_as_float(sr[2 * c + 2]), __uint_as_float(sr[2 * c + 3])), sc2,
                  nm2);
              p[0] = ex2_approx(x0.x);
              p[1] = ex2_approx(x0.y);
              p[2] = ex2_approx(x1.x);
              p[3] = ex2_approx(x1.y);
              const float2 pair = __fadd2_rn(make_float2(p[0], p[2]), make_float2(p[1], p[3]));
              sp[(c >> 1) & 3] = __fadd2_rn(sp[(c >> 1) & 3], pair);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                p[e] = ex2_approx(fmaf(__uint_as_float(sr[2 * c + e]), scale_log2, -m_use));
              sp[(c >> 1) & 3].x += p[0] + p[1];
              sp[(c >> 1) & 3].y += p[2] + p[3];
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float p0 = p[2 * h], p1 = p[2 * h + 1];
              const int cc = c + h;
              if (DROPOUT) {
                const uint32_t bits = kb[cc >> 4] >> ((2 * cc) & 31);
                sr[cc] = pack_bf16x2((bits & 1u) ? p0 : 0.0f, (bits & 2u) ? p1 : 0.0f);
              } else {
                sr[cc] = pack_bf16x2(p0, p1);
              }
            }
          }
        }
        const float2 s01 = __fadd2_rn(sp[0], sp[1]);
        const float2 s23 = __fadd2_rn(sp[2], sp[3]);
        const float2 s4 = __fadd2_rn(s01, s23);
        sum = s4.x + s4.y;
      };
      bool move = false;
      float alpha = 1.0f;
      bool exact = !__all_sync(0xffffffffu, m_run != -INFINITY);
      constexpr float kBound = FP8 ? kSpeculateSumBoundF8 : kSpeculateSumBound;
      // the block max of the scores, and the running max moved when some row
      // of the warp needs it
      auto move_max = [&]() {
        const float m_blk = row_max128(sr) * scale_log2;
        move = __any_sync(0xffffffffu, m_blk > m_run + kLazyRescaleLog2);
        if (move) {
          const float m_new = fmaxf(m_run, m_blk);
          alpha = ex2_approx(m_run - m_new);  // 0 on the first tile
          l_run *= alpha;
          m_run = m_new;
        }
      };
      if (DROPOUT || FP8 || SPARSE) {
        // two copies of the exponential loop (the speculative and the exact
        // pass); one shared copy in a loop, as below, measured slower here:
        // 9 % with dropout (the keep bits live across it), 7.6 % for e4m3,
        // 0.7 % block-sparse
        if (!exact) {
          exp_tile();
          // speculation held unless some row's sum exceeds the bound (or is not finite)
          if (__any_sync(0xffffffffu, !(sum <= kBound))) {
            load_scores();  // the speculative pass overwrote sr with P~
            exact = true;
          }
        }
        if (exact) {
          move_max();
          exp_tile();
        }
      } else {
        // one copy of the exponential loop, run once, or twice when the
        // speculative pass fails (the smaller kernel spills less and ran 1-4 %
        // faster)
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
          if (exact) move_max();
          exp_tile();
          if (exact) break;
          // speculation held unless some row's sum exceeds the bound (or is not finite)
          if (!__any_sync(0xffffffffu, !(sum <= kBound))) break;
          load_scores();  // the speculative pass overwrote sr with P~
          exact = true;
        }
      }
      tmem_st32(scol + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      if (!FP8) tmem_st32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      if (move && j > 0) {
        // PV_g(j-1) completed before S_g(j) was reported, and PV_g(j) is not
        // issued before p_ready: O is stable here
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(ocol + c * 32, r);
          tmem_ld_wait();
          reg_pin(r);
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 o2 = __fmul2_rn(
                make_float2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1])), a2);
            r[2 * e] = __float_as_uint(o2.x);
            r[2 * e + 1] = __float_as_uint(o2.y);
          }
          tmem_st32(ocol + c * 32, r);
        }
      }
      l_run += sum;
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars->p_ready[g]);
    }
    // ------------------------------------------------ epilogue
    if (SPARSE && nkv == 0) {
      // no key tile at all: O = 0, lse = -inf (tensor memory is never read)
      if (row < N) {
        uint4* dst = reinterpret_cast<uint4*>(o + (static_cast<size_t>(bh) * N + row) * D);
#pragma unroll
        for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
        lse[static_cast<size_t>(bh) * N + row] = -INFINITY;
      }
    } else if (ok && (ok = warp_wait(&bars->pv_done[g], (tb + nkv - 1) & 1, bars, 0x303))) {
      tc_fence_after_sync();
      // a row with no visible key (block-sparse) has l = 0: O = 0, lse = -inf;
      // with dropout the kept terms carry the factor 1 / (1 - p)
      const float inv_l =
          l_run > 0.0f ? (DROPOUT ? drop.rs : 1.0f) * (FP8 ? o_scale : 1.0f) / l_run : 0.0f;
      // Rows of this lane's 4-lane group are stored together, row by row (32
      // columns at a time: the softmax warps' registers are scarce).  The
      // persistent causal kernel, which carries its item state across the
      // epilogue, has no registers left for the transpose and stores its own
      // row (measured: the transpose there spills and costs 7 % at N = 2048).
      constexpr bool kGroupStore = !(PERSIST && CAUSAL);
      const int r0 = kGroupStore ? row - (lane & 3) : row;
      const int grp_rows = min(kGroupStore ? 4 : 1, N - r0);
      __nv_bfloat16* ogrp = o + (static_cast<size_t>(bh) * N + (grp_rows > 0 ? r0 : 0)) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(ocol + c * 32, r);
        tmem_ld_wait();
        reg_pin(r);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv_l, __uint_as_float(r[2 * e + 1]) * inv_l);
        if (kGroupStore) {
          store_rows<4>(w, ogrp + c * 32, D, grp_rows);
        } else if (grp_rows > 0) {
          uint4* dst = reinterpret_cast<uint4*>(ogrp + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      if (row < N)
        lse[static_cast<size_t>(bh) * N + row] =
            l_run > 0.0f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
    }
    // O_g has been read: the next item's first P V may overwrite it
    tc_fence_before_sync();
    mbar_arrive(&bars->o_free[g]);
    return ok;
    };
    if (kPersist) {
      auto swait = [&](uint64_t* bar, uint32_t par) { return warp_wait(bar, par, bars, 0x304); };
      int tb = 0;
      for (int tt = 0;; ++tt) {
        const int item = consumer_item(tt, swait);
        if (item < 0 || !softmax_item(item, tb)) break;
        tb += item_n(item, g);
      }
    } else {
      softmax_item(static_cast<int>(blockIdx.x), 0);
    }
  }

  // ------------------------------------------------ teardown
  if (warp == kMmaWarp) {
    // every MMA this CTA issued has completed before TMEM is released
    mbar_wait(&bars->drain, 0, &bars->abort_flag, &g_fwd_error, 0x205);
  }
  if (bars->abort_flag) {
    // let any bulk copy already in flight land before the CTA exits
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kTmemCols);
  }
  // the last CTA of a persistent launch leaves its counter slot zeroed
  if (kPersist && threadIdx.x == 0 && atomicAdd(&sched[1], 1u) == gridDim.x - 1) {
    atomicExch(&sched[0], 0u);
    atomicExch(&sched[1], 0u);
  }
}

// Heads per group of the item order: causal calls take as many heads as keep
// the K / V tiles of a group within half of the 129 MB L2 (the pairs of a
// group go heaviest first across its heads); non-causal calls 1 (head-major).
int group_heads(const FwdArgs& a) {
  if (!a.causal) return 1;
  const double kv_head = 2.0 * a.N * a.d * (a.fp8 ? 1.0 : 2.0);
  const double g = (64.0 * 1024 * 1024) / kv_head;
  return static_cast<int>(g < 1.0 ? 1.0 : (g > a.BH ? a.BH : g));
}

// Counter slots of this file's persistent launches (see SchedRing).
SchedRing g_sched_ring;

cudaError_t claim_slot(cudaStream_t s, unsigned int** out) {
  return claim_sched_slot(g_sched_ring, reinterpret_cast<const void*>(&g_fwd_sched), s, out);
}

template <int D, bool CAUSAL, bool SPARSE, bool DROPOUT, bool FP8 = false, bool PERSIST = false>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t s) {
  auto kern = fa_fwd_kernel<D, CAUSAL, SPARSE, DROPOUT, FP8, PERSIST>;
  constexpr uint32_t smem = FwdLayout<D, FP8 ? 1 : 2>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long nq = (a.N + kTileM - 1) / kTileM;
  const long long items = (nq + 1) / 2 * a.BH;
  if (items > 0x7fffffffll) return cudaErrorInvalidValue;
  // Non-causal items all weigh the same: persistent CTAs, one per SM, take
  // them in turn.  Causal items weigh 3 .. 2 nq - 1 key tiles, and the hardware
  // block scheduler, handing out the heaviest-first order one item per CTA as
  // SMs free up, balances them far better than any fixed assignment; block-
  // sparse items likewise get one CTA each.
  constexpr bool kPersist = PERSIST;
  const long long blocks = kPersist ? std::min<long long>(items, a.num_sms) : items;
  unsigned int* sched = nullptr;
  if (kPersist) {
    if (a.num_sms < 1) return cudaErrorInvalidValue;
    if ((e = claim_slot(s, &sched)) != cudaSuccess) return e;
  }
  kern<<<static_cast<unsigned>(blocks), kFwdThreads, smem, s>>>(
      *a.tq, *a.tk, *a.tv, static_cast<__nv_bfloat16*>(a.o), a.lse, a.BH, a.N, a.scale_log2,
      a.bmask, a.mstride, a.drop, a.o_scale, sched, group_heads(a));
  return cudaGetLastError();
}

template <bool SPARSE, bool DROPOUT, bool PERSIST = false>
cudaError_t launch_forward_s(const FwdArgs& a, cudaStream_t s) {
  if (a.d == 64)
    return a.causal ? launch_fwd_t<64, true, SPARSE, DROPOUT, false, PERSIST>(a, s)
                    : launch_fwd_t<64, false, SPARSE, DROPOUT, false, PERSIST>(a, s);
  return a.causal ? launch_fwd_t<128, true, SPARSE, DROPOUT, false, PERSIST>(a, s)
                  : launch_fwd_t<128, false, SPARSE, DROPOUT, false, PERSIST>(a, s);
}

// Dense sequences up to this length run persistent CTAs: with few key tiles
// per item the per-item start-up and epilogue are a large share of the work,
// and overlapping them pays; longer sequences keep one CTA per item, whose
// leaner code runs the long key loops faster.  Measured on GB300 (d = 128,
// causal, one CTA per item against persistent, with the packed softmax
// arithmetic): 876 / 900 TFLOP/s at N = 2048, 1098 / 1090 at 4096, 1254 /
// 1210 at 8192.
constexpr int kPersistMaxN = 2048;

bool fwd_persist(const FwdArgs& a) {
  return !a.bmask && a.num_sms > 0 && a.N <= kPersistMaxN;
}

}  // namespace

cudaError_t launch_forward(const FwdArgs& a, cudaStream_t s) {
  if (a.fp8) {  // d = 128, dense, no dropout (checked by the caller)
    return a.causal ? launch_fwd_t<128, true, false, false, true>(a, s)
                    : launch_fwd_t<128, false, false, false, true>(a, s);
  }
  const bool persist = fwd_persist(a);
  if (a.dropout) {
    if (persist) return launch_forward_s<false, true, true>(a, s);
    return a.bmask ? launch_forward_s<true, true>(a, s) : launch_forward_s<false, true>(a, s);
  }
  if (persist) return launch_forward_s<false, false, true>(a, s);
  return a.bmask ? launch_forward_s<true, false>(a, s) : launch_forward_s<false, false>(a, s);
}

cudaError_t fwd_reset_sched(cudaStream_t s) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_fwd_sched);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p, 0, sizeof(g_fwd_sched), s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

cudaError_t fwd_read_clear_error(uint32_t* out, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_fwd_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_fwd_error, &zero, sizeof(zero));
  }
  *out = v;
  return e;
}

}  // namespace fa
