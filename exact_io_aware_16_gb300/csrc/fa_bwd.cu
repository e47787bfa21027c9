// fa_bwd.cu — recompute backward of exact attention for sm_103a.
//
// "What is Flash Attention?" 06:52-07:24: P is not stored; it is rebuilt tile
// by tile from Q, K and the per-row statistic (here lse = m + ln l) with the
// same tiling loop, trading FLOPs for HBM traffic.  The gradient formulas are
// the chain rule through the exact definition (the pages state only that the
// gradients are the same as standard attention's, 08:26):
//   P = exp(scale * Q K^T - lse),  dV = P^T dO,  dP = dO V^T,
//   D_i = sum_c dO_ic O_ic,  dS = P o (dP - D),  dQ = scale dS K,
//   dK = scale dS^T Q.
//
// Three kernels:
//   * bwd_pre:  D = rowsum(dO o O), fp32, HBM-bound.
//   * bwd_dkdv: one CTA per (batch*head, 128-row key tile).  K_j and V_j stay
//     in shared memory; 128-row Q_i / dO_i tiles stream through a two-stage
//     TMA ring.  Scores are computed transposed, S^T = K_j Q_i^T, so the key
//     row is the TMEM lane: each of 128 threads owns one key row, forms
//     P^T and dS^T for its row and writes them back as bf16 over S^T / dP^T
//     in tensor memory, where they are the A operand of
//     dV += P^T dO_i and dK += dS^T Q_i (accumulators live in TMEM).
//   * bwd_dq:   one CTA per (batch*head, 128-row query tile).  Q_i, dO_i stay
//     resident; K_j / V_j stream.  S = Q_i K_j^T and dP = dO_i V_j^T give dS
//     per query row; dQ += dS K_j accumulates in TMEM.
// Causal tiles above the diagonal are skipped in both kernels; the mask is
// applied inside the diagonal tile only.
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <type_traits>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "philox.cuh"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

__device__ unsigned int g_bwd_error;

// Work-item counters of persistent launches (as in the forward): each launch
// claims a slot, its CTAs take items with atomicAdd on slot[0], the last CTA
// to finish (slot[1] counts them) zeroes the slot; bwd_reset_sched zeroes all
// slots after a device error.
__device__ unsigned int g_bwd_sched[kSchedSlots][2];
constexpr int kItemRing = 4;  // claimed items in flight between the roles of a CTA

constexpr int kBwdThreads = 320;
constexpr int kStages = 2;  // streamed-tile ring at d = 128 (shared memory allows no more)
// d = 64: a four-stage ring, where the scores of the next step are issued
// before the current step's products and need their tiles a step earlier
constexpr int kStages64 = 4;
constexpr float kLog2e = 1.44269504088896340736f;

// ============================================================ D pre-pass
// Each group of d/8 consecutive threads owns one row: every thread loads 8
// bf16 of O and of dO (one 16-byte vector each), forms the partial dot product
// in fp32, and the group reduces with warp shuffles.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const uint4* __restrict__ o,
                                                         const uint4* __restrict__ dO,
                                                         float* __restrict__ Dout,
                                                         long long rows) {
  constexpr int kPerRow = D / 8;  // threads per row: 8 or 16
  const long long gt = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = gt / kPerRow;
  float acc = 0.0f;
  if (row < rows) {
    const uint4 a = o[gt];
    const uint4 b = dO[gt];
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa2 = __bfloat1622float2(pa[e]);
      const float2 fb2 = __bfloat1622float2(pb[e]);
      acc = fmaf(fa2.x, fb2.x, acc);
      acc = fmaf(fa2.y, fb2.y, acc);
    }
  }
#pragma unroll
  for (int off = kPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && (gt % kPerRow) == 0) Dout[row] = acc;
}

// ============================================================ shared pieces
// Warp roles of both recompute kernels (320 threads):
//   warps 0-7  two compute warpgroups; warpgroup g owns score columns
//              [64g, 64g+64) of every row, thread t of a warpgroup owns TMEM
//              lane (row) t, so the 128 columns of a tile are processed by two
//              warps per SM sub-partition;
//   warp 8     TMA producer;
//   warp 9     TMEM allocator and MMA issuer.
constexpr int kComputeThreads = 256;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;

template <int D>
struct BwdLayout {
  static constexpr int kRing = D == 64 ? kStages64 : kStages;
  static constexpr int kChunks = D / 64;
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  // dkdv: K, V resident; Q, dO streamed.  dq: Q, dO resident; K, V streamed.
  static constexpr uint32_t kRes0 = 0;
  static constexpr uint32_t kRes1 = kRes0 + kTileBytes;
  static constexpr uint32_t kStr0 = kRes1 + kTileBytes;                // [stage] tiles
  static constexpr uint32_t kStr1 = kStr0 + kRing * kTileBytes;       // [stage] tiles
  static constexpr uint32_t kVec = kStr1 + kRing * kTileBytes;         // lse/D vectors
  static constexpr uint32_t kBar = kVec + kRing * 2 * 128 * 4;
  static constexpr uint32_t kList = kBar + 256;  // block-sparse tile list (uint16)
  static constexpr uint32_t kSmemUsed = kList + 2 * kMaxSparseTiles + 1024;
  // at least 116 KB, so two CTAs never share an SM (each takes all 512 TMEM columns)
  static constexpr uint32_t kSmem = kSmemUsed > 118784u ? kSmemUsed : 118784u;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSCol = 0;     // S (or S^T); P bf16 packed inside each half
  static constexpr uint32_t kDPCol = 128;  // dP (or dP^T); dS bf16 packed inside each half
  static constexpr uint32_t kAcc0 = 256;   // dV (dkdv) or dQ~ (dq)
  static constexpr uint32_t kAcc1 = 256 + D;  // dK (dkdv) or B = P K (dq)
  // d = 64: the accumulators leave columns 384..511 free, a second score
  // buffer: step g's scores (and P over them) sit in buffer g % 2, so the next
  // step's score product need not wait for this step's P to be consumed
  static constexpr bool kDoubleS = D == 64;
  __host__ __device__ static constexpr uint32_t s_col(int step) {
    return (kDoubleS && (step & 1)) ? 384u : kSCol;
  }
};

struct BwdBars {
  uint64_t res_full;
  uint64_t str_full[kStages], str_empty[kStages];
  uint64_t s_full, dp_full, p_ready, ds_ready;
  uint64_t dx_ready;
  uint64_t acc_done;
  uint64_t res_empty;  // persistent: the item's products are done with the resident tiles
  uint64_t acc_free;   // persistent: the epilogue has read the accumulators
  uint64_t item_full[kItemRing];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int nlist;  // block-sparse: entries of the tile list
  int item_ring[kItemRing];  // claimed items (-1: no more)
  // d = 64 only: ring stages 2 and 3, and the "scores ready" / "P ready"
  // barriers of score buffer 1 (each buffer has its own: with step g + 1's
  // scores issued before step g's P is consumed, one barrier could complete a
  // second phase before the waiter of the first has seen it)
  uint64_t str_full_hi[2], str_empty_hi[2];
  uint64_t s_full_1, p_ready_1;
};

static_assert(sizeof(BwdBars) <= 256, "barrier block overruns its shared-memory slot");

// Barriers of ring stage s, and of score buffer b, in a ring of R stages
template <int R>
__device__ __forceinline__ uint64_t* str_full_bar(BwdBars* b, int s) {
  if constexpr (R == 2) return &b->str_full[s];
  else return s < 2 ? &b->str_full[s] : &b->str_full_hi[s - 2];
}
template <int R>
__device__ __forceinline__ uint64_t* str_empty_bar(BwdBars* b, int s) {
  if constexpr (R == 2) return &b->str_empty[s];
  else return s < 2 ? &b->str_empty[s] : &b->str_empty_hi[s - 2];
}
// step g's "scores ready" / "P ready" barrier and its parity
template <bool DS>
__device__ __forceinline__ uint64_t* s_full_bar(BwdBars* b, int g) {
  if constexpr (DS) return (g & 1) ? &b->s_full_1 : &b->s_full;
  else return &b->s_full;
}
template <bool DS>
__device__ __forceinline__ uint64_t* p_ready_bar(BwdBars* b, int g) {
  if constexpr (DS) return (g & 1) ? &b->p_ready_1 : &b->p_ready;
  else return &b->p_ready;
}
template <bool DS>
__host__ __device__ constexpr uint32_t s_parity(int g) { return DS ? ((g >> 1) & 1) : (g & 1); }

// Adds `bytes` to the transaction count of the current phase of `bar`
// without arriving (the arrival comes separately, after staged data).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Ring slot and phase parity of the streamed tile at ring position pos >= 0
// (R stages, a power of two; 2 unless stated).
template <int R = kStages>
__device__ __forceinline__ int ring_slot(int pos) {
  return static_cast<int>(static_cast<unsigned>(pos) % R);
}
template <int R = kStages>
__device__ __forceinline__ uint32_t ring_phase(int pos) {
  return (static_cast<unsigned>(pos) / R) & 1u;
}

// Block-sparse tile list, built by warp 0 with ballots: the tiles t in
// [t_begin, t_end) for which mask[t * t_stride] != 0 (so t is a query tile
// for the dK/dV kernel and a key tile for the dQ kernel), in order.
__device__ __forceinline__ void build_list(uint16_t* list, int* count_out, const uint8_t* mask,
                                           long long t_stride, int t_begin, int t_end) {
  const int lane = static_cast<int>(lane_id());
  int count = 0;
  for (int base = t_begin; base < t_end; base += 32) {
    const int t = base + lane;
    const bool use = t < t_end && mask[t * t_stride] != 0;
    const unsigned bal = __ballot_sync(0xffffffffu, use);
    if (use) list[count + __popc(bal & ((1u << lane) - 1u))] = static_cast<uint16_t>(t);
    count += __popc(bal);
  }
  if (lane == 0) *count_out = count;
}

__device__ __forceinline__ bool bwd_warp_wait(uint64_t* bar, uint32_t parity, BwdBars* b,
                                              uint32_t code) {
  bool ok = mbar_wait(bar, parity, &b->abort_flag, &g_bwd_error, code);
  return __all_sync(0xffffffffu, ok);
}

// Returns false (uniformly for the CTA) when an earlier CTA of this library
// already recorded a pipeline timeout: the CTA then exits without work.
__device__ __forceinline__ bool bwd_init(BwdBars* bars, int warp, uint32_t cols) {
  if (threadIdx.x == 0) {
    mbar_init(&bars->res_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->str_full[s], 1);
      mbar_init(&bars->str_empty[s], 1);
      mbar_init(&bars->str_full_hi[s], 1);
      mbar_init(&bars->str_empty_hi[s], 1);
    }
    mbar_init(&bars->s_full_1, 1);
    mbar_init(&bars->p_ready_1, kComputeThreads);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_ready, kComputeThreads);
    mbar_init(&bars->ds_ready, kComputeThreads);
    mbar_init(&bars->dx_ready, kComputeThreads);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->res_empty, 1);
    mbar_init(&bars->acc_free, kComputeThreads);
    for (int r = 0; r < kItemRing; ++r) mbar_init(&bars->item_full[r], 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = (*static_cast<volatile unsigned int*>(&g_bwd_error) != 0) ? 1 : 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (bars->abort_flag) return false;
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  return true;
}

__device__ __forceinline__ void bwd_teardown(BwdBars* bars, int warp, uint32_t tmem,
                                             uint32_t cols) {
  if (warp == kMmaWarp) mbar_wait(&bars->drain, 0, &bars->abort_flag, &g_bwd_error, 0x2ff);
  if (bars->abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, cols);
  }
}

// Producer of one work item (the whole TMA warp): two resident tiles, then
// two streamed tiles per step at ring positions sb, sb + 1, ...  When `lse`
// is given (dK/dV kernel), the warp also stages the streamed query tile's
// lse * log2(e) (+inf past N) and D (0 past N) in shared memory before lane 0
// arrives on the stage's barrier, so they travel with the tiles.  t > 0 (a
// persistent CTA's later item): the first streamed tile goes first, then the
// resident tiles once the previous item's products are done with them.
// Returns false (uniformly for the warp) after a pipeline timeout.
template <int D>
__device__ __forceinline__ bool bwd_producer_item(uint8_t* smem, BwdBars* bars,
                                                  const CUtensorMap* r0, const CUtensorMap* r1,
                                                  int res_row0, const CUtensorMap* s0,
                                                  const CUtensorMap* s1, int first_tile,
                                                  int ntiles, int bh, const float* lse_bh,
                                                  const float* D_bh, int N, const uint16_t* list,
                                                  int t, int sb) {
  using L = BwdLayout<D>;
  const int lane = static_cast<int>(lane_id());
  if (ntiles == 0) return true;  // nothing to compute: load nothing
  auto load_res = [&]() {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars->res_full, 2 * L::kTileBytes);
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_3d(smem + L::kRes0 + c * 16384, r0, &bars->res_full, c * 64, res_row0, bh);
        tma_load_3d(smem + L::kRes1 + c * 16384, r1, &bars->res_full, c * 64, res_row0, bh);
      }
    }
  };
  if (t == 0) load_res();
  for (int n = 0; n < ntiles; ++n) {
    const int s = ring_slot<L::kRing>(sb + n);
    const uint32_t ph = ring_phase<L::kRing>(sb + n);
    bool ok = mbar_wait(str_empty_bar<L::kRing>(bars, s), ph ^ 1, &bars->abort_flag, &g_bwd_error,
                        0x101);
    if (!__all_sync(0xffffffffu, ok)) return false;
    const int row0 = (list ? static_cast<int>(list[n]) : first_tile + n) * 128;
    // the tiles first, then (while they are in flight) the staged vectors; the
    // stage's one arrival comes last, after both
    if (lane == 0) {
      mbar_expect_tx(str_full_bar<L::kRing>(bars, s), 2 * L::kTileBytes);
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_3d(smem + L::kStr0 + s * L::kTileBytes + c * 16384, s0, str_full_bar<L::kRing>(bars, s),
                    c * 64, row0, bh);
        tma_load_3d(smem + L::kStr1 + s * L::kTileBytes + c * 16384, s1, str_full_bar<L::kRing>(bars, s),
                    c * 64, row0, bh);
      }
    }
    if (lse_bh != nullptr) {
      float* vec = reinterpret_cast<float*>(smem + L::kVec) + s * 256;  // [lse2 | D]
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = lane + 32 * e;
        const int q = row0 + i;
        vec[i] = (q < N) ? lse_bh[q] * kLog2e : INFINITY;
        vec[128 + i] = (q < N) ? D_bh[q] : 0.0f;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(str_full_bar<L::kRing>(bars, s));
    __syncwarp();
    if (n == 0 && t > 0) {
      ok = mbar_wait(&bars->res_empty, (t - 1) & 1, &bars->abort_flag, &g_bwd_error, 0x102);
      if (!__all_sync(0xffffffffu, ok)) return false;
      load_res();
      __syncwarp();
    }
  }
  return true;
}

// The item claimed t-th by a persistent CTA (-1: no more), from the TMA warp
// (claims with atomicAdd on the launch's counter and publishes) or from a
// consumer (waits for the ring entry); `wait` is the caller's bounded wait.
__device__ __forceinline__ int bwd_claim_item(BwdBars* bars, unsigned int* sched, int n_items,
                                              int t) {
  int item = 0;
  if (lane_id() == 0) {
    const unsigned int c = atomicAdd(&sched[0], 1u);
    item = c < static_cast<unsigned int>(n_items) ? static_cast<int>(c) : -1;
    bars->item_ring[t % kItemRing] = item;
    mbar_arrive(&bars->item_full[t % kItemRing]);
  }
  return __shfl_sync(0xffffffffu, item, 0);
}

// The last CTA of a persistent launch leaves its counter slot zeroed.
__device__ __forceinline__ void bwd_release_sched(unsigned int* sched) {
  if (threadIdx.x == 0 && atomicAdd(&sched[1], 1u) == gridDim.x - 1) {
    atomicExch(&sched[0], 0u);
    atomicExch(&sched[1], 0u);
  }
}

// K-major operand descriptor for k-step kk of a [128 rows][D] swizzled tile.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
}
// MN-major operand descriptor (rows of the tile are the K dimension) for k-step kk.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, int kk) {
  return sdesc_sw128(base + kk * 2048, 16384, 1024);
}
// TMEM column of k-step kk (16 score columns) of a bf16 operand packed inside
// the two 64-column halves of a 128-column fp32 region: half g holds score
// columns [64g, 64g+64) packed in its first 32 columns.
__device__ __forceinline__ uint32_t packed_a_col(int kk) {
  return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8);
}

// Load 64 fp32 columns [addr, addr+64) of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld64(uint32_t addr, uint32_t (&r)[64]) {
  tmem_ld32(addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
  tmem_ld32(addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
  tmem_ld_wait();
  reg_pin(r);
}

__device__ __forceinline__ void tmem_st16(uint32_t addr, const uint32_t (&w)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(addr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
      "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]),
      "r"(w[15])
      : "memory");
}

// Store 64 fp32 accumulator columns [addr, addr+64) of this lane's row as bf16
// (times `mul`), written together with the rows of this lane's 8-lane group:
// grp_dst / ld / grp_rows as for store_rows.
__device__ __forceinline__ void store_acc_half(uint32_t addr, float mul, __nv_bfloat16* grp_dst,
                                               long long ld, int grp_rows) {
  uint32_t w[32];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t r[32];
    tmem_ld32(addr + c * 32, r);
    tmem_ld_wait();
    reg_pin(r);
#pragma unroll
    for (int e = 0; e < 16; ++e)
      w[16 * c + e] =
          pack_bf16x2(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
  }
  store_rows<8>(w, grp_dst, ld, grp_rows);
}

// ============================================================ dK / dV
// SPARSE: only the query tiles whose block-mask entry for this key tile is
// set are visited (a compact list built by warp 0).
//
// DROPOUT (dropout on P with keep matrix Z and rs the inverse keep
// probability):
// dV = rs (P o Z)^T dO and dS = P o (rs Z o dP - D); P itself (undropped)
// stays in registers for dS, P o Z goes to the dV product, rs is applied when
// dV is stored.  The keep bits of a key row come transposed from the
// generator's row-major counters (keep_word_t).
template <int D, bool CAUSAL, bool SPARSE, bool DROPOUT, bool PERSIST>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq,
                       const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv,
                       const __grid_constant__ CUtensorMap tdo, const float* __restrict__ lse,
                       const float* __restrict__ Dvec, __nv_bfloat16* __restrict__ dk,
                       __nv_bfloat16* __restrict__ dv, int BH, int N, float scale,
                       float scale_log2, const uint8_t* __restrict__ bmask, long long mstride,
                       DropArgs drop, int group_heads, unsigned int* __restrict__ sched) {
  static_assert(!(PERSIST && SPARSE), "block-sparse tiles each have their own CTA");
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + L::kBar);
  const float* vec = reinterpret_cast<const float*>(smem + L::kVec);  // [stage][lse2 | D][128]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nt = (N + 127) / 128;
  // Work items: one key tile of one (b, h), numbered in the order they are
  // handed out: in groups of group_heads heads, tile-major within a group,
  // key tile 0 (the heaviest when causal) of every head first.  Handing them
  // out in order balances the SMs like longest-job-first while the Q / dO
  // tiles a group streams stay within L2 (the launcher sizes the group; 1 =
  // head-major).  PERSIST: persistent CTAs claim items from the launch's
  // counter slot (the TMA warp claims, a ring in shared memory publishes
  // them); otherwise CTA = item blockIdx.x.
  const int n_items = BH * nt;
  auto item_rank = [&](int item, int& head) {
    const int grp = item / (group_heads * nt);
    const int gs = min(group_heads, BH - grp * group_heads);
    const int r = item - grp * group_heads * nt;
    head = grp * group_heads + r % gs;
    return r / gs;
  };
  auto item_bh = [&](int item) {
    int head;
    item_rank(item, head);
    return head;
  };
  auto item_kt = [&](int item) {
    int head;
    return item_rank(item, head);
  };
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::kList);
  if (SPARSE && warp == 0) {  // column kt of the mask: query tiles i >= i_first
    const int bh = item_bh(blockIdx.x), kt = item_kt(blockIdx.x);
    build_list(list, &bars->nlist, bmask + bh * mstride + kt, nt, CAUSAL ? kt : 0, nt);
  }

  if (!bwd_init(bars, warp, L::kTmemCols)) return;
  const uint32_t tmem = bars->tmem_base;
  auto item_first = [&](int item) { return CAUSAL ? item_kt(item) : 0; };  // first query tile
  auto item_iters = [&](int item) { return SPARSE ? bars->nlist : nt - item_first(item); };
  auto consumer_item = [&](int t, auto&& wait) -> int {
    if (!wait(&bars->item_full[t % kItemRing], (t / kItemRing) & 1)) return -1;
    return bars->item_ring[t % kItemRing];
  };

  if (warp == kTmaWarp) {
    auto produce = [&](int item, int t, int sb) {
      const int bh = item_bh(item);
      return bwd_producer_item<D>(smem, bars, &tk, &tv, item_kt(item) * 128, &tq, &tdo,
                                  item_first(item), item_iters(item), bh,
                                  lse + static_cast<size_t>(bh) * N,
                                  Dvec + static_cast<size_t>(bh) * N, N,
                                  SPARSE ? list : nullptr, t, sb);
    };
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
    }
    if (PERSIST) {
      for (int t = 0, sb = 0;; ++t) {
        const int item = bwd_claim_item(bars, sched, n_items, t);
        if (item < 0 || !produce(item, t, sb)) break;
        sb += item_iters(item);
      }
    } else {
      produce(static_cast<int>(blockIdx.x), 0, 0);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
      const uint32_t sK = smem_u32(smem + L::kRes0);
      const uint32_t sV = smem_u32(smem + L::kRes1);
      auto sQ = [&](int pos) { return smem_u32(smem + L::kStr0 + ring_slot(pos) * L::kTileBytes); };
      auto sdO = [&](int pos) { return smem_u32(smem + L::kStr1 + ring_slot(pos) * L::kTileBytes); };
      // S^T = K Q^T and dP^T = V dO^T of the streamed tile at ring position
      // pos (the commit is the caller's)
      auto issue_s = [&](int pos) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + L::kSCol, kmajor_desc(sK, kk), kmajor_desc(sQ(pos), kk), idesc_s,
                  kk > 0 ? 1u : 0u);
      };
      auto issue_dp = [&](int pos) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + L::kDPCol, kmajor_desc(sV, kk), kmajor_desc(sdO(pos), kk), idesc_s,
                  kk > 0 ? 1u : 0u);
      };
      // one item: t = items before it in this CTA, sb = ring position of its
      // first streamed tile, nb = steps before it (barrier phases)
      auto mma_item = [&](const int item, const int t, const int sb, const int nb) -> bool {
        const int n_iters = item_iters(item);
        if (n_iters == 0) return true;
        bool ok = mbar_wait(&bars->res_full, t & 1, &bars->abort_flag, &g_bwd_error, 0x201) &&
                  mbar_wait(&bars->str_full[ring_slot(sb)], ring_phase(sb), &bars->abort_flag,
                            &g_bwd_error, 0x202);
        if (!ok) return false;
        tc_fence_after_sync();
        issue_s(sb);
        umma_commit(&bars->s_full);
        issue_dp(sb);
        umma_commit(&bars->dp_full);
        // order per step: dV_n, S^T_{n+1}, dK_n, dP^T_{n+1}, so that the exps of
        // step n+1 overlap dK_n and dP^T_{n+1} on the tensor core.  They go out
        // as two bursts (dV_n S^T_{n+1}, dK_n dP^T_{n+1}) with the waits for
        // what a burst reads ahead of it where the barriers have already
        // completed: a blocking wait of this thread between two products
        // leaves the tensor core idle once the earlier one completes.
        for (int n = 0; n < n_iters; ++n) {
          const int pos = sb + n;
          const bool more = n + 1 < n_iters;
          // dV += P^T dO_n   (A = P^T bf16 in TMEM, B = dO_n MN-major, K = 128 queries);
          // the first one of an item overwrites the accumulators the previous
          // item's epilogue read
          if (!mbar_wait(&bars->p_ready, (nb + n) & 1, &bars->abort_flag, &g_bwd_error, 0x203) ||
              (n == 0 && t > 0 &&
               !mbar_wait(&bars->acc_free, (t - 1) & 1, &bars->abort_flag, &g_bwd_error, 0x206))) {
            ok = false;
            break;
          }
          const bool next_in =
              !more || mbar_test_wait(&bars->str_full[ring_slot(pos + 1)], ring_phase(pos + 1));
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + L::kAcc0, tmem + L::kSCol + packed_a_col(kk), mnmajor_desc(sdO(pos), kk),
                    idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
          if (more) {
            if (!next_in) {
              if (!mbar_wait(&bars->str_full[ring_slot(pos + 1)], ring_phase(pos + 1),
                             &bars->abort_flag, &g_bwd_error, 0x205)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
            }
            issue_s(pos + 1);
          }
          // dK += dS^T Q_n   (A = dS^T bf16 in TMEM, B = Q_n MN-major)
          const bool ds_in = mbar_test_wait(&bars->ds_ready, (nb + n) & 1);
          if (more) umma_commit(&bars->s_full);
          if (!ds_in &&
              !mbar_wait(&bars->ds_ready, (nb + n) & 1, &bars->abort_flag, &g_bwd_error, 0x204)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + L::kAcc1, tmem + L::kDPCol + packed_a_col(kk), mnmajor_desc(sQ(pos), kk),
                    idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars->str_empty[ring_slot(pos)]);
          if (more) {
            issue_dp(pos + 1);
            umma_commit(&bars->dp_full);
          }
        }
        if (ok) umma_commit(&bars->acc_done);
        umma_commit(&bars->res_empty);  // K, V free once the products above complete
        return ok;
      };
      // d = 64 (two score buffers, four-stage ring): the next step's scores
      // go first, into the other score buffer (the P there was read by the dV
      // of the step before, issued earlier), so that they are ready when the
      // compute warps finish a step; the ring has their tiles in well ahead.
      // Otherwise as mma_item.
      auto slot4 = [](int pos) { return ring_slot<L::kRing>(pos); };
      auto phase4 = [](int pos) { return ring_phase<L::kRing>(pos); };
      auto sQ4 = [&](int pos) { return smem_u32(smem + L::kStr0 + slot4(pos) * L::kTileBytes); };
      auto sdO4 = [&](int pos) { return smem_u32(smem + L::kStr1 + slot4(pos) * L::kTileBytes); };
      auto mma_item_ds = [&](const int item, const int t, const int sb, const int nb) -> bool {
        const int n_iters = item_iters(item);
        if (n_iters == 0) return true;
        auto issue_s4 = [&](int pos, uint32_t col) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + col, kmajor_desc(sK, kk), kmajor_desc(sQ4(pos), kk), idesc_s,
                    kk > 0 ? 1u : 0u);
        };
        auto issue_dp4 = [&](int pos) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + L::kDPCol, kmajor_desc(sV, kk), kmajor_desc(sdO4(pos), kk), idesc_s,
                    kk > 0 ? 1u : 0u);
        };
        bool ok = mbar_wait(&bars->res_full, t & 1, &bars->abort_flag, &g_bwd_error, 0x201) &&
                  mbar_wait(str_full_bar<L::kRing>(bars, slot4(sb)), phase4(sb), &bars->abort_flag,
                            &g_bwd_error, 0x202);
        if (!ok) return false;
        tc_fence_after_sync();
        issue_s4(sb, L::s_col(nb));
        umma_commit(s_full_bar<true>(bars, nb));
        issue_dp4(sb);
        umma_commit(&bars->dp_full);
        for (int n = 0; n < n_iters; ++n) {
          const int pos = sb + n;
          const bool more = n + 1 < n_iters;
          if (more) {
            if (!mbar_wait(str_full_bar<L::kRing>(bars, slot4(pos + 1)), phase4(pos + 1),
                           &bars->abort_flag, &g_bwd_error, 0x208)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_s4(pos + 1, L::s_col(nb + n + 1));
            umma_commit(s_full_bar<true>(bars, nb + n + 1));
          }
          if (!mbar_wait(p_ready_bar<true>(bars, nb + n), s_parity<true>(nb + n), &bars->abort_flag,
                         &g_bwd_error, 0x203) ||
              (n == 0 && t > 0 &&
               !mbar_wait(&bars->acc_free, (t - 1) & 1, &bars->abort_flag, &g_bwd_error, 0x206))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + L::kAcc0, tmem + L::s_col(nb + n) + packed_a_col(kk),
                    mnmajor_desc(sdO4(pos), kk), idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
          if (!mbar_test_wait(&bars->ds_ready, (nb + n) & 1) &&
              !mbar_wait(&bars->ds_ready, (nb + n) & 1, &bars->abort_flag, &g_bwd_error, 0x204)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + L::kAcc1, tmem + L::kDPCol + packed_a_col(kk), mnmajor_desc(sQ4(pos), kk),
                    idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
          umma_commit(str_empty_bar<L::kRing>(bars, slot4(pos)));
          if (more) {
            issue_dp4(pos + 1);
            umma_commit(&bars->dp_full);
          }
        }
        if (ok) umma_commit(&bars->acc_done);
        umma_commit(&bars->res_empty);
        return ok;
      };
      if (PERSIST) {
        auto mwait = [&](uint64_t* bar, uint32_t par) {
          return mbar_wait(bar, par, &bars->abort_flag, &g_bwd_error, 0x207);
        };
        for (int t = 0, sb = 0, nb = 0;; ++t) {
          const int item = consumer_item(t, mwait);
          if (item < 0 ||
              !(L::kDoubleS ? mma_item_ds(item, t, sb, nb) : mma_item(item, t, sb, nb)))
            break;
          sb += item_iters(item);
          nb += item_iters(item);
        }
      } else if (L::kDoubleS) {
        mma_item_ds(static_cast<int>(blockIdx.x), 0, 0, 0);
      } else {
        mma_item(static_cast<int>(blockIdx.x), 0, 0, 0);
      }
      umma_commit(&bars->drain);
    }
    __syncwarp();
  } else {
    // ---------------------------------------- compute warpgroups (warps 0-7)
    const int T = threadIdx.x;  // 0..255
    const int g = T >> 7;       // column half
    const int tr = T & 127;     // key row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t col0 = 64u * g;
    // one item: t = items before it in this CTA, nb = steps before it (ring
    // positions and barrier phases).  Returns false after a pipeline timeout.
    auto compute_item = [&](const int item, const int t, const int nb) -> bool {
    bool ok = true;
    const int bh = item_bh(item), kt = item_kt(item);
    const int k0 = kt * 128;
    const int krow = k0 + tr;
    const int n_iters = item_iters(item);
    // the generator's products that depend on this key row's counter words alone
    const PhiloxCol pcol = DROPOUT ? philox_col_init(drop, static_cast<uint32_t>(krow) >> 3,
                                                     static_cast<uint32_t>(bh))
                                   : PhiloxCol{};
    for (int n = 0; n < n_iters; ++n) {
      const int it = SPARSE ? static_cast<int>(list[n]) : item_first(item) + n;
      const int q0 = it * 128;
      // lse * log2(e) and D of this query tile, staged with the tiles
      const float* lse2_s = vec + ring_slot<L::kRing>(nb + n) * 256;
      const float* D_s = lse2_s + 128;
      // dropout keep bits of this key row for query rows q0 + col0 + c (bit c
      // of kb[c / 32]), drawn before the scores are waited for
      uint32_t kb[2] = {0u, 0u};
      if (DROPOUT) {
#pragma unroll
        for (int w = 0; w < 2; ++w)
          kb[w] = keep_word_t(drop, pcol, static_cast<uint32_t>(q0) + col0 + 32u * w, lane);
        reg_pin(kb);  // drawn here, before the wait, not next to their use
      }
      if (!bwd_warp_wait(s_full_bar<L::kDoubleS>(bars, nb + n), s_parity<L::kDoubleS>(nb + n),
                         bars, 0x301)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      // P^T for this key row and query columns [col0, col0+64)
      uint32_t pr[64];
      tmem_ld64(tmem + lane_off + L::s_col(nb + n) + col0, pr);
      // only the diagonal tile needs the causal mask (query rows past N have
      // lse = +inf staged, so their P is 0 without one); the test is uniform
      // across the warp
      const bool diag = CAUSAL && (it == kt);
      const float4* lse4 = reinterpret_cast<const float4*>(lse2_s + col0);
      const float2 sc2 = make_float2(scale_log2, scale_log2);
      auto exp_cols = [&](auto masked) {
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l4 = lse4[c4];
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // two columns per packed fma
            const int c = 4 * c4 + 2 * h;
            const float2 nl = h ? make_float2(-l4.z, -l4.w) : make_float2(-l4.x, -l4.y);
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(pr[c]), __uint_as_float(pr[c + 1])), sc2, nl);
            float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
            if (masked) {  // query before key
              if (q0 + static_cast<int>(col0) + c < krow) p0 = 0.0f;
              if (q0 + static_cast<int>(col0) + c + 1 < krow) p1 = 0.0f;
            }
            pr[c] = __float_as_uint(p0);
            pr[c + 1] = __float_as_uint(p1);
          }
        }
      };
      if (diag)
        exp_cols(std::true_type{});
      else
        exp_cols(std::false_type{});
      {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float p0 = __uint_as_float(pr[2 * c]), p1 = __uint_as_float(pr[2 * c + 1]);
          if (DROPOUT) {  // P o Z for the dV product
            const uint32_t bits = kb[c >> 4] >> ((2 * c) & 31);
            pk[c] = pack_bf16x2((bits & 1u) ? p0 : 0.0f, (bits & 2u) ? p1 : 0.0f);
          } else {
            pk[c] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st32(tmem + lane_off + L::s_col(nb + n) + col0, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(p_ready_bar<L::kDoubleS>(bars, nb + n));
      if (!bwd_warp_wait(&bars->dp_full, (nb + n) & 1, bars, 0x304)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      // dS^T = P^T o (dP^T - D), 32 columns at a time, packed bf16 in place
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + L::kDPCol + col0 + c2 * 32, r);
        tmem_ld_wait();
        reg_pin(r);
        uint32_t w[16];
        const float4* d4 = reinterpret_cast<const float4*>(D_s + col0 + c2 * 32);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 dd = d4[e4];
          const int c = c2 * 32 + 4 * e4;
          float dp[4] = {__uint_as_float(r[4 * e4]), __uint_as_float(r[4 * e4 + 1]),
                         __uint_as_float(r[4 * e4 + 2]), __uint_as_float(r[4 * e4 + 3])};
          if (DROPOUT) {  // dP of the dropped product: rs Z o (dO V^T)
            const uint32_t bits = kb[c >> 5] >> (c & 31);
#pragma unroll
            for (int e = 0; e < 4; ++e) dp[e] = ((bits >> e) & 1u) ? dp[e] * drop.rs : 0.0f;
          }
          // dS^T = P^T (dP^T - D), two columns per packed op (each lane
          // rounded as the scalar ops)
          const float2 ds01 = __fmul2_rn(
              make_float2(__uint_as_float(pr[c]), __uint_as_float(pr[c + 1])),
              __fadd2_rn(make_float2(dp[0], dp[1]), make_float2(-dd.x, -dd.y)));
          const float2 ds23 = __fmul2_rn(
              make_float2(__uint_as_float(pr[c + 2]), __uint_as_float(pr[c + 3])),
              __fadd2_rn(make_float2(dp[2], dp[3]), make_float2(-dd.z, -dd.w)));
          w[2 * e4] = pack_bf16x2(ds01.x, ds01.y);
          w[2 * e4 + 1] = pack_bf16x2(ds23.x, ds23.y);
        }
        tmem_st16(tmem + lane_off + L::kDPCol + col0 + c2 * 16, w);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars->ds_ready);
    }
    if (SPARSE && n_iters == 0) {
      // no query tile keeps this key tile: dK = dV = 0 (tensor memory is never read)
      if (krow < N) {
        const size_t off = (static_cast<size_t>(bh) * N + krow) * D;
        uint4* pk = reinterpret_cast<uint4*>(dk + off + (D == 128 ? col0 : 0));
        uint4* pv = reinterpret_cast<uint4*>(dv + off + (D == 128 ? col0 : 0));
        const int nvec = (D == 128 ? 64 : (g == 0 ? 64 : 0)) / 8;
        for (int e = 0; e < nvec; ++e) {
          pk[e] = make_uint4(0u, 0u, 0u, 0u);
          pv[e] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    } else if (ok && (ok = bwd_warp_wait(&bars->acc_done, t & 1, bars, 0x302))) {
      tc_fence_after_sync();
      // rows of this lane's 8-lane group (stored together, row by row)
      const int r0 = krow - (lane & 7);
      const int grp_rows = min(8, N - r0);
      const size_t off = (static_cast<size_t>(bh) * N + (grp_rows > 0 ? r0 : 0)) * D;
      // d = 128: warpgroup g stores columns [64g, 64g+64) of dV and dK;
      // d = 64: warpgroup 0 stores dV, warpgroup 1 stores dK
      const float dv_mul = DROPOUT ? drop.rs : 1.0f;
      if (D == 128) {
        store_acc_half(tmem + lane_off + L::kAcc0 + col0, dv_mul, dv + off + col0, D, grp_rows);
        store_acc_half(tmem + lane_off + L::kAcc1 + col0, scale, dk + off + col0, D, grp_rows);
      } else if (g == 0) {
        store_acc_half(tmem + lane_off + L::kAcc0, dv_mul, dv + off, D, grp_rows);
      } else {
        store_acc_half(tmem + lane_off + L::kAcc1, scale, dk + off, D, grp_rows);
      }
    }
    // the accumulators have been read: the next item may overwrite them
    tc_fence_before_sync();
    mbar_arrive(&bars->acc_free);
    return ok;
    };
    if (PERSIST) {
      auto cwait = [&](uint64_t* bar, uint32_t par) { return bwd_warp_wait(bar, par, bars, 0x305); };
      for (int t = 0, nb = 0;; ++t) {
        const int item = consumer_item(t, cwait);
        if (item < 0 || !compute_item(item, t, nb)) break;
        nb += item_iters(item);
      }
    } else {
      compute_item(static_cast<int>(blockIdx.x), 0, 0);
    }
  }
  bwd_teardown(bars, warp, tmem, L::kTmemCols);
  if (PERSIST) bwd_release_sched(sched);
}

// ============================================================ dQ
// dS needs D_i before the loop over key tiles has seen the whole row, so the
// loop uses the pre-pass estimate D~_i = rowsum(dO o O) (O stored in bf16) and
// accumulates, alongside dQ~ = scale sum_j P_ij (dP_ij - D~_i) k_j, the exact
// definition D_i = sum_j P_ij dP_ij (fp32) and B_i = sum_j P_ij k_j (one more
// MMA).  The epilogue corrects dQ = dQ~ - scale (D_i - D~_i) B_i, which removes
// the error that bf16 rounding of O puts into D~, and writes D_i back over
// D~_i for the dK/dV kernel that runs next.
// SPARSE: only the key tiles this query tile keeps in the block mask are
// visited (a compact list built by warp 0).
//
// DROPOUT: dP becomes rs Z o (dO V^T) (the exact D and dS use it); B = P K
// keeps the undropped P, since dS = P o (dP - D) is linear in D.
template <int D, bool CAUSAL, bool SPARSE, bool DROPOUT, bool PERSIST>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv,
                     const __grid_constant__ CUtensorMap tdo, const float* __restrict__ lse,
                     float* __restrict__ Dvec, __nv_bfloat16* __restrict__ dq, int BH, int N,
                     float scale, float scale_log2, const uint8_t* __restrict__ bmask,
                     long long mstride, DropArgs drop, int group_heads,
                     unsigned int* __restrict__ sched) {
  static_assert(!(PERSIST && SPARSE), "block-sparse tiles each have their own CTA");
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + L::kBar);
  float* dx_base = reinterpret_cast<float*>(smem + L::kVec);  // [item parity][2 halves][128 rows]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nt = (N + 127) / 128;
  // Work items: one query tile of one (b, h), numbered in the order they are
  // handed out: in groups of group_heads heads, tile-major within a group,
  // the heaviest (last, qt + 1 key tiles when causal) query tile of every
  // head first (longest-job-first balancing, with the K / V tiles a group
  // streams within L2; 1 = head-major).  PERSIST: persistent CTAs claim
  // items from the launch's counter slot; otherwise CTA = item blockIdx.x.
  const int n_items = BH * nt;
  auto item_rank = [&](int item, int& head) {
    const int grp = item / (group_heads * nt);
    const int gs = min(group_heads, BH - grp * group_heads);
    const int r = item - grp * group_heads * nt;
    head = grp * group_heads + r % gs;
    return r / gs;
  };
  auto item_bh = [&](int item) {
    int head;
    item_rank(item, head);
    return head;
  };
  auto item_qt = [&](int item) {
    int head;
    return nt - 1 - item_rank(item, head);
  };
  constexpr uint32_t kDQ = L::kAcc0;  // dQ~ accumulator
  constexpr uint32_t kB = L::kAcc1;   // B = P K accumulator
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::kList);
  if (SPARSE && warp == 0) {  // row qt of the mask: key tiles j < qt + 1 (causal) or < nt
    const int bh = item_bh(blockIdx.x), qt = item_qt(blockIdx.x);
    build_list(list, &bars->nlist, bmask + bh * mstride + static_cast<long long>(qt) * nt, 1, 0,
               CAUSAL ? qt + 1 : nt);
  }

  if (!bwd_init(bars, warp, L::kTmemCols)) return;
  const uint32_t tmem = bars->tmem_base;
  auto item_iters = [&](int item) {
    return SPARSE ? bars->nlist : (CAUSAL ? item_qt(item) + 1 : nt);
  };
  auto kt_of = [&](int n) -> int { return SPARSE ? static_cast<int>(list[n]) : n; };
  auto consumer_item = [&](int t, auto&& wait) -> int {
    if (!wait(&bars->item_full[t % kItemRing], (t / kItemRing) & 1)) return -1;
    return bars->item_ring[t % kItemRing];
  };

  if (warp == kTmaWarp) {
    auto produce = [&](int item, int t, int sb) {
      return bwd_producer_item<D>(smem, bars, &tq, &tdo, item_qt(item) * 128, &tk, &tv, 0,
                                  item_iters(item), item_bh(item), nullptr, nullptr, N,
                                  SPARSE ? list : nullptr, t, sb);
    };
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      tma_prefetch_desc(&tdo);
    }
    if (PERSIST) {
      for (int t = 0, sb = 0;; ++t) {
        const int item = bwd_claim_item(bars, sched, n_items, t);
        if (item < 0 || !produce(item, t, sb)) break;
        sb += item_iters(item);
      }
    } else {
      produce(static_cast<int>(blockIdx.x), 0, 0);
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, false, true);
      const uint32_t sQ = smem_u32(smem + L::kRes0);
      const uint32_t sdO = smem_u32(smem + L::kRes1);
      auto sK = [&](int pos) { return smem_u32(smem + L::kStr0 + ring_slot(pos) * L::kTileBytes); };
      auto sV = [&](int pos) { return smem_u32(smem + L::kStr1 + ring_slot(pos) * L::kTileBytes); };
      // S = Q K^T  and  dP = dO V^T of the streamed tile at ring position pos
      // (the commit is the caller's)
      auto issue_s = [&](int pos) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + L::kSCol, kmajor_desc(sQ, kk), kmajor_desc(sK(pos), kk), idesc_s,
                  kk > 0 ? 1u : 0u);
      };
      auto issue_dp = [&](int pos) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + L::kDPCol, kmajor_desc(sdO, kk), kmajor_desc(sV(pos), kk), idesc_s,
                  kk > 0 ? 1u : 0u);
      };
      // one item: t = items before it in this CTA, sb = ring position of its
      // first streamed tile (= steps before it: barrier phases)
      auto mma_item = [&](const int item, const int t, const int sb) -> bool {
        const int n_iters = item_iters(item);
        if (n_iters == 0) return true;
        bool ok = mbar_wait(&bars->res_full, t & 1, &bars->abort_flag, &g_bwd_error, 0x211) &&
                  mbar_wait(&bars->str_full[ring_slot(sb)], ring_phase(sb), &bars->abort_flag,
                            &g_bwd_error, 0x212);
        if (!ok) return false;
        tc_fence_after_sync();
        issue_s(sb);
        umma_commit(&bars->s_full);
        issue_dp(sb);
        umma_commit(&bars->dp_full);
        // order per step: B_n, S_{n+1}, dQ~_n, dP_{n+1}, as two bursts with the
        // waits ahead of them where the barriers have already completed (as in
        // the dK/dV kernel)
        for (int n = 0; n < n_iters; ++n) {
          const int pos = sb + n;
          const bool more = n + 1 < n_iters;
          // B += P K_n   (A = P bf16 in TMEM over S, B = K_n MN-major); the
          // first one of an item overwrites the accumulators the previous
          // item's epilogue read
          if (!mbar_wait(&bars->p_ready, pos & 1, &bars->abort_flag, &g_bwd_error, 0x214) ||
              (n == 0 && t > 0 &&
               !mbar_wait(&bars->acc_free, (t - 1) & 1, &bars->abort_flag, &g_bwd_error, 0x216))) {
            ok = false;
            break;
          }
          const bool next_in =
              !more || mbar_test_wait(&bars->str_full[ring_slot(pos + 1)], ring_phase(pos + 1));
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + kB, tmem + L::kSCol + packed_a_col(kk), mnmajor_desc(sK(pos), kk),
                    idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
          if (more) {
            if (!next_in) {
              if (!mbar_wait(&bars->str_full[ring_slot(pos + 1)], ring_phase(pos + 1),
                             &bars->abort_flag, &g_bwd_error, 0x215)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
            }
            issue_s(pos + 1);
          }
          // dQ~ += dS~ K_n   (A = dS~ bf16 in TMEM over dP)
          const bool ds_in = mbar_test_wait(&bars->ds_ready, pos & 1);
          if (more) umma_commit(&bars->s_full);
          if (!ds_in &&
              !mbar_wait(&bars->ds_ready, pos & 1, &bars->abort_flag, &g_bwd_error, 0x213)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + kDQ, tmem + L::kDPCol + packed_a_col(kk), mnmajor_desc(sK(pos), kk),
                    idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars->str_empty[ring_slot(pos)]);
          if (more) {
            issue_dp(pos + 1);
            umma_commit(&bars->dp_full);
          }
        }
        if (ok) umma_commit(&bars->acc_done);
        umma_commit(&bars->res_empty);  // Q, dO free once the products above complete
        return ok;
      };
      // d = 64 (two score buffers, four-stage ring): the next step's scores
      // go first, as in the dK/dV kernel.  Otherwise as mma_item.
      auto slot4 = [](int pos) { return ring_slot<L::kRing>(pos); };
      auto phase4 = [](int pos) { return ring_phase<L::kRing>(pos); };
      auto sK4 = [&](int pos) { return smem_u32(smem + L::kStr0 + slot4(pos) * L::kTileBytes); };
      auto sV4 = [&](int pos) { return smem_u32(smem + L::kStr1 + slot4(pos) * L::kTileBytes); };
      auto mma_item_ds = [&](const int item, const int t, const int sb) -> bool {
        const int n_iters = item_iters(item);
        if (n_iters == 0) return true;
        auto issue_s4 = [&](int pos, uint32_t col) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + col, kmajor_desc(sQ, kk), kmajor_desc(sK4(pos), kk), idesc_s,
                    kk > 0 ? 1u : 0u);
        };
        auto issue_dp4 = [&](int pos) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss(tmem + L::kDPCol, kmajor_desc(sdO, kk), kmajor_desc(sV4(pos), kk), idesc_s,
                    kk > 0 ? 1u : 0u);
        };
        bool ok = mbar_wait(&bars->res_full, t & 1, &bars->abort_flag, &g_bwd_error, 0x211) &&
                  mbar_wait(str_full_bar<L::kRing>(bars, slot4(sb)), phase4(sb), &bars->abort_flag,
                            &g_bwd_error, 0x212);
        if (!ok) return false;
        tc_fence_after_sync();
        issue_s4(sb, L::s_col(sb));
        umma_commit(s_full_bar<true>(bars, sb));
        issue_dp4(sb);
        umma_commit(&bars->dp_full);
        for (int n = 0; n < n_iters; ++n) {
          const int pos = sb + n;
          const bool more = n + 1 < n_iters;
          if (more) {
            if (!mbar_wait(str_full_bar<L::kRing>(bars, slot4(pos + 1)), phase4(pos + 1),
                           &bars->abort_flag, &g_bwd_error, 0x218)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_s4(pos + 1, L::s_col(pos + 1));
            umma_commit(s_full_bar<true>(bars, pos + 1));
          }
          if (!mbar_wait(p_ready_bar<true>(bars, pos), s_parity<true>(pos), &bars->abort_flag,
                         &g_bwd_error, 0x214) ||
              (n == 0 && t > 0 &&
               !mbar_wait(&bars->acc_free, (t - 1) & 1, &bars->abort_flag, &g_bwd_error, 0x216))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + kB, tmem + L::s_col(pos) + packed_a_col(kk), mnmajor_desc(sK4(pos), kk),
                    idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
          if (!mbar_test_wait(&bars->ds_ready, pos & 1) &&
              !mbar_wait(&bars->ds_ready, pos & 1, &bars->abort_flag, &g_bwd_error, 0x213)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ts(tmem + kDQ, tmem + L::kDPCol + packed_a_col(kk), mnmajor_desc(sK4(pos), kk),
                    idesc_acc, (n > 0 || kk > 0) ? 1u : 0u);
          umma_commit(str_empty_bar<L::kRing>(bars, slot4(pos)));
          if (more) {
            issue_dp4(pos + 1);
            umma_commit(&bars->dp_full);
          }
        }
        if (ok) umma_commit(&bars->acc_done);
        umma_commit(&bars->res_empty);
        return ok;
      };
      if (PERSIST) {
        auto mwait = [&](uint64_t* bar, uint32_t par) {
          return mbar_wait(bar, par, &bars->abort_flag, &g_bwd_error, 0x217);
        };
        for (int t = 0, sb = 0;; ++t) {
          const int item = consumer_item(t, mwait);
          if (item < 0 || !(L::kDoubleS ? mma_item_ds(item, t, sb) : mma_item(item, t, sb)))
            break;
          sb += item_iters(item);
        }
      } else if (L::kDoubleS) {
        mma_item_ds(static_cast<int>(blockIdx.x), 0, 0);
      } else {
        mma_item(static_cast<int>(blockIdx.x), 0, 0);
      }
      umma_commit(&bars->drain);
    }
    __syncwarp();
  } else {
    const int T = threadIdx.x;
    const int g = T >> 7;
    const int tr = T & 127;  // query row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t col0 = 64u * g;
    // one item: t = items before it in this CTA, nb = steps before it (barrier
    // phases).  Returns false after a pipeline timeout.
    auto compute_item = [&](const int item, const int t, const int nb) -> bool {
    const int bh = item_bh(item), q0 = item_qt(item) * 128;
    const int n_iters = item_iters(item);
    const int row = q0 + tr;
    const bool rvalid = row < N;
    const float lse2 = rvalid ? lse[static_cast<size_t>(bh) * N + row] * kLog2e : 0.0f;
    const float Dt = rvalid ? Dvec[static_cast<size_t>(bh) * N + row] : 0.0f;  // D~
    // the generator's products that depend on this row's counter words alone
    const PhiloxRow prow = DROPOUT ? philox_row_init(drop, static_cast<uint32_t>(row),
                                                     static_cast<uint32_t>(bh))
                                   : PhiloxRow{};
    // this half's part of the exact D = sum_j P_ij dP_ij (four partial sums)
    float2 dx2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    bool ok = true;
    for (int n = 0; n < n_iters; ++n) {
      // dropout keep bits of this row for keys kt_of(n) * 128 + col0 + c
      // (bit c of kb[c / 32]), drawn before the scores are waited for
      uint32_t kb[2] = {0u, 0u};
      if (DROPOUT) {
        const uint32_t jg0 = (static_cast<uint32_t>(kt_of(n)) * 128u + col0) >> 3;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          kb[u >> 2] |= keep_byte_row(drop, prow, jg0 + u) << (8 * (u & 3));
        reg_pin(kb);  // drawn here, before the wait, not next to their use
      }
      if (!bwd_warp_wait(s_full_bar<L::kDoubleS>(bars, nb + n), s_parity<L::kDoubleS>(nb + n),
                         bars, 0x311)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t pr[64];
      tmem_ld64(tmem + lane_off + L::s_col(nb + n) + col0, pr);
      const int kv0 = kt_of(n) * 128;
      // only the diagonal tile (causal) and a ragged last tile need a mask:
      // the test is uniform across the warp, so other tiles skip it
      const bool need_mask = (CAUSAL && kv0 + 127 > q0) || (kv0 + 128 > N);
      // exponent argument s * scale * log2(e) - lse * log2(e), two columns
      // per packed fma (each lane rounded as the scalar fma)
      const float2 sc2 = make_float2(scale_log2, scale_log2);
      const float2 nl2 = make_float2(-lse2, -lse2);
      auto exp_cols = [&](auto masked, int lim) {
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 x =
              __ffma2_rn(make_float2(__uint_as_float(pr[c]), __uint_as_float(pr[c + 1])), sc2, nl2);
          float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
          if (masked) {
            if (c > lim) p0 = 0.0f;
            if (c + 1 > lim) p1 = 0.0f;
          }
          pr[c] = __float_as_uint(p0);
          pr[c + 1] = __float_as_uint(p1);
        }
      };
      if (need_mask) {
        const int lim_c = CAUSAL ? (row - kv0) : 0x7fffffff;
        const int lim_n = N - 1 - kv0;
        exp_cols(std::true_type{}, (lim_c < lim_n ? lim_c : lim_n) - static_cast<int>(col0));
      } else {
        exp_cols(std::false_type{}, 0);
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c)
          pk[c] = pack_bf16x2(__uint_as_float(pr[2 * c]), __uint_as_float(pr[2 * c + 1]));
        tmem_st32(tmem + lane_off + L::s_col(nb + n) + col0, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(p_ready_bar<L::kDoubleS>(bars, nb + n));
      if (!bwd_warp_wait(&bars->dp_full, (nb + n) & 1, bars, 0x314)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float2 nD2 = make_float2(-Dt, -Dt);
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + L::kDPCol + col0 + c2 * 32, r);
        tmem_ld_wait();
        reg_pin(r);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c = c2 * 32 + 2 * e;
          const float2 pp = make_float2(__uint_as_float(pr[c]), __uint_as_float(pr[c + 1]));
          float2 dd = make_float2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
          if (DROPOUT) {  // dP of the dropped product: rs Z o (dO V^T)
            const uint32_t bits = kb[c >> 5] >> (c & 31);
            dd.x = (bits & 1u) ? dd.x * drop.rs : 0.0f;
            dd.y = (bits & 2u) ? dd.y * drop.rs : 0.0f;
          }
          // exact D: columns 2e and 2e + 1 feed partial sums (e & 1) x / y;
          // dS = P (dP - D~), packed (each lane rounded as the scalar ops)
          dx2[e & 1] = __ffma2_rn(pp, dd, dx2[e & 1]);
          const float2 ds = __fmul2_rn(pp, __fadd2_rn(dd, nD2));
          w[e] = pack_bf16x2(ds.x, ds.y);
        }
        tmem_st16(tmem + lane_off + L::kDPCol + col0 + c2 * 16, w);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars->ds_ready);
    }
    if (SPARSE && n_iters == 0) {
      // no key tile kept: dQ = 0 and the row's D is 0 (tensor memory is never read)
      if (rvalid) {
        const size_t off = (static_cast<size_t>(bh) * N + row) * D;
        uint4* p = reinterpret_cast<uint4*>(dq + off + (D == 128 ? col0 : 0));
        const int nvec = (D == 128 ? 64 : (g == 0 ? 64 : 0)) / 8;
        for (int e = 0; e < nvec; ++e) p[e] = make_uint4(0u, 0u, 0u, 0u);
        if (g == 0) Dvec[static_cast<size_t>(bh) * N + row] = 0.0f;
      }
      return ok;
    }
    // combine the two halves' parts of D (bounded wait); the buffer
    // alternates between items
    float* dx_s = dx_base + (t & 1) * 256;
    if (ok) {
      dx_s[g * 128 + tr] = (dx2[0].x + dx2[0].y) + (dx2[1].x + dx2[1].y);
      mbar_arrive(&bars->dx_ready);
      ok = bwd_warp_wait(&bars->dx_ready, t & 1, bars, 0x313);
    }
    if (ok && (ok = bwd_warp_wait(&bars->acc_done, t & 1, bars, 0x312))) {
      tc_fence_after_sync();
      const float Dfull = dx_s[tr] + dx_s[128 + tr];
      const float corr = Dfull - Dt;
      // rows of this lane's 8-lane group (stored together, row by row)
      const int r0 = row - (lane & 7);
      const int grp_rows = min(8, N - r0);
      const size_t off = (static_cast<size_t>(bh) * N + (grp_rows > 0 ? r0 : 0)) * D;
      // d = 128: warpgroup g stores dq columns [64g, 64g+64); d = 64: warpgroup 0 only
      if (D == 128 || g == 0) {
        const uint32_t c0 = (D == 128) ? col0 : 0u;
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t a[32], b[32];
          tmem_ld32(tmem + lane_off + kDQ + c0 + c * 32, a);
          tmem_ld32(tmem + lane_off + kB + c0 + c * 32, b);
          tmem_ld_wait();
          reg_pin(a);
          reg_pin(b);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float x0 =
                scale * fmaf(-corr, __uint_as_float(b[2 * e]), __uint_as_float(a[2 * e]));
            const float x1 =
                scale * fmaf(-corr, __uint_as_float(b[2 * e + 1]), __uint_as_float(a[2 * e + 1]));
            w[16 * c + e] = pack_bf16x2(x0, x1);
          }
        }
        store_rows<8>(w, dq + off + c0, D, grp_rows);
      }
      if (g == 0 && rvalid) Dvec[static_cast<size_t>(bh) * N + row] = Dfull;
    }
    // the accumulators have been read: the next item may overwrite them
    tc_fence_before_sync();
    mbar_arrive(&bars->acc_free);
    return ok;
    };
    if (PERSIST) {
      auto cwait = [&](uint64_t* bar, uint32_t par) { return bwd_warp_wait(bar, par, bars, 0x315); };
      for (int t = 0, nb = 0;; ++t) {
        const int item = consumer_item(t, cwait);
        if (item < 0 || !compute_item(item, t, nb)) break;
        nb += item_iters(item);
      }
    } else {
      compute_item(static_cast<int>(blockIdx.x), 0, 0);
    }
  }
  bwd_teardown(bars, warp, tmem, L::kTmemCols);
  if (PERSIST) bwd_release_sched(sched);
}

template <typename Kern>
cudaError_t prep(Kern k, uint32_t smem) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

// Heads per group of the tile order (both kernels stream two [N][d] bf16
// tensors per head): causal calls take as many heads as keep a group's
// streamed tiles within half of the 129 MB L2; non-causal calls 1
// (head-major: the tiles are equal).
int bwd_group_heads(const BwdArgs& a) {
  if (!a.causal) return 1;
  const double per_head = 2.0 * a.N * a.d * 2.0;
  const double g = (64.0 * 1024 * 1024) / per_head;
  return static_cast<int>(g < 1.0 ? 1.0 : (g > a.BH ? a.BH : g));
}

// Counter slots of this file's persistent launches (see SchedRing).
SchedRing g_sched_ring;

cudaError_t claim_slot(cudaStream_t s, unsigned int** out) {
  return claim_sched_slot(g_sched_ring, reinterpret_cast<const void*>(&g_bwd_sched), s, out);
}

// Grid of a backward launch: persistent (one CTA per SM, items claimed from
// a counter slot) or one CTA per item.
template <bool PERSIST>
cudaError_t bwd_grid(const BwdArgs& a, cudaStream_t s, unsigned* blocks, unsigned int** sched) {
  const long long items = static_cast<long long>((a.N + 127) / 128) * a.BH;
  if (items > 0x7fffffffll) return cudaErrorInvalidValue;
  *sched = nullptr;
  if (!PERSIST) {
    *blocks = static_cast<unsigned>(items);
    return cudaSuccess;
  }
  if (a.num_sms < 1) return cudaErrorInvalidValue;
  *blocks = static_cast<unsigned>(std::min<long long>(items, a.num_sms));
  return claim_slot(s, sched);
}

template <int D, bool CAUSAL, bool SPARSE, bool DROPOUT, bool PERSIST>
cudaError_t launch_dkdv_t(const BwdArgs& a, cudaStream_t s) {
  auto kern = fa_bwd_dkdv_kernel<D, CAUSAL, SPARSE, DROPOUT, PERSIST>;
  constexpr uint32_t smem = BwdLayout<D>::kSmem;
  cudaError_t e = prep(kern, smem);
  if (e != cudaSuccess) return e;
  unsigned blocks = 0;
  unsigned int* sched = nullptr;
  if ((e = bwd_grid<PERSIST>(a, s, &blocks, &sched)) != cudaSuccess) return e;
  kern<<<blocks, kBwdThreads, smem, s>>>(
      *a.tq, *a.tk, *a.tv, *a.tdo, a.lse, a.D, static_cast<__nv_bfloat16*>(a.dk),
      static_cast<__nv_bfloat16*>(a.dv), a.BH, a.N, a.scale, a.scale_log2, a.bmask, a.mstride,
      a.drop, bwd_group_heads(a), sched);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool SPARSE, bool DROPOUT, bool PERSIST>
cudaError_t launch_dq_t(const BwdArgs& a, cudaStream_t s) {
  auto kern = fa_bwd_dq_kernel<D, CAUSAL, SPARSE, DROPOUT, PERSIST>;
  constexpr uint32_t smem = BwdLayout<D>::kSmem;
  cudaError_t e = prep(kern, smem);
  if (e != cudaSuccess) return e;
  unsigned blocks = 0;
  unsigned int* sched = nullptr;
  if ((e = bwd_grid<PERSIST>(a, s, &blocks, &sched)) != cudaSuccess) return e;
  kern<<<blocks, kBwdThreads, smem, s>>>(
      *a.tq, *a.tk, *a.tv, *a.tdo, a.lse, a.D, static_cast<__nv_bfloat16*>(a.dq), a.BH, a.N,
      a.scale, a.scale_log2, a.bmask, a.mstride, a.drop, bwd_group_heads(a), sched);
  return cudaGetLastError();
}

// Persistent backward CTAs: the next tile's first copies and the current
// tile's epilogue overlap, which pays most where tiles are short.  Measured on
// GB300 (persistent against one CTA per tile, causal unless noted): +6 % at
// B4 H16 N4096 d128, +2-3 % at N = 8192 and 16384, +2.5 % at N = 8192 d64,
// even at 32768 and non-causal 8192.  Dense calls all run persistent.
bool bwd_persist(const BwdArgs& a) { return a.num_sms > 0; }

template <bool SPARSE, bool DROPOUT, bool PERSIST>
cudaError_t launch_dkdv_p(const BwdArgs& a, cudaStream_t s) {
  if (a.d == 64)
    return a.causal ? launch_dkdv_t<64, true, SPARSE, DROPOUT, PERSIST>(a, s)
                    : launch_dkdv_t<64, false, SPARSE, DROPOUT, PERSIST>(a, s);
  return a.causal ? launch_dkdv_t<128, true, SPARSE, DROPOUT, PERSIST>(a, s)
                  : launch_dkdv_t<128, false, SPARSE, DROPOUT, PERSIST>(a, s);
}

template <bool SPARSE, bool DROPOUT, bool PERSIST>
cudaError_t launch_dq_p(const BwdArgs& a, cudaStream_t s) {
  if (a.d == 64)
    return a.causal ? launch_dq_t<64, true, SPARSE, DROPOUT, PERSIST>(a, s)
                    : launch_dq_t<64, false, SPARSE, DROPOUT, PERSIST>(a, s);
  return a.causal ? launch_dq_t<128, true, SPARSE, DROPOUT, PERSIST>(a, s)
                  : launch_dq_t<128, false, SPARSE, DROPOUT, PERSIST>(a, s);
}

template <bool SPARSE, bool DROPOUT>
cudaError_t launch_dkdv_s(const BwdArgs& a, cudaStream_t s) {
  if (!SPARSE && bwd_persist(a)) return launch_dkdv_p<false, DROPOUT, true>(a, s);
  return launch_dkdv_p<SPARSE, DROPOUT, false>(a, s);
}

template <bool SPARSE, bool DROPOUT>
cudaError_t launch_dq_s(const BwdArgs& a, cudaStream_t s) {
  if (!SPARSE && bwd_persist(a)) return launch_dq_p<false, DROPOUT, true>(a, s);
  return launch_dq_p<SPARSE, DROPOUT, false>(a, s);
}

}  // namespace

cudaError_t launch_bwd_preprocess(const void* o, const void* dO, float* D, long long rows, int d,
                                  cudaStream_t s) {
  const long long threads = rows * (d / 8);
  const long long blocks = (threads + 255) / 256;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  if (d == 64)
    fa_bwd_pre_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<const uint4*>(o), static_cast<const uint4*>(dO), D, rows);
  else
    fa_bwd_pre_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<const uint4*>(o), static_cast<const uint4*>(dO), D, rows);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t s) {
  if (a.dropout)
    return a.bmask ? launch_dkdv_s<true, true>(a, s) : launch_dkdv_s<false, true>(a, s);
  return a.bmask ? launch_dkdv_s<true, false>(a, s) : launch_dkdv_s<false, false>(a, s);
}

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t s) {
  if (a.dropout)
    return a.bmask ? launch_dq_s<true, true>(a, s) : launch_dq_s<false, true>(a, s);
  return a.bmask ? launch_dq_s<true, false>(a, s) : launch_dq_s<false, false>(a, s);
}

cudaError_t bwd_reset_sched(cudaStream_t s) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_sched);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(p, 0, sizeof(g_bwd_sched), s);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(s);
}

cudaError_t bwd_read_clear_error(uint32_t* out, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_bwd_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_bwd_error, &zero, sizeof(zero));
  }
  *out = v;
  return e;
}

}  // namespace fa
