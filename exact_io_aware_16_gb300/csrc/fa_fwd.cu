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
//     is only moved when a row's block max exceeds it by more than 2^8
//     (kLazyRescaleLog2): until then P~ <= 2^8 against the stale max, and since
//     O and l are scaled by the same factor, O / l is unchanged.  beta of the
//     page is folded in by exponentiating against the current max directly
//     (the "l_new" formula of the mentria page).
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

constexpr int kFwdThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStages = 2;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLazyRescaleLog2 = 8.0f;

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
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int nlist;  // block-sparse: entries of the key-tile list
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
template <int D, bool CAUSAL, bool SPARSE, bool DROPOUT, bool FP8>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, __nv_bfloat16* __restrict__ o,
                  float* __restrict__ lse, int BH, int N, float scale_log2,
                  const uint8_t* __restrict__ bmask, long long mstride, DropArgs drop,
                  float o_scale) {
  static_assert(!FP8 || (D == 128 && !SPARSE && !DROPOUT), "e4m3 path: d = 128, dense");
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
  // head-major order (the query tiles of one head run together and share its
  // K / V tiles in L2); within a head the heaviest (last) pair first
  const int pair = npairs - 1 - static_cast<int>(blockIdx.x % npairs);
  const int bh = static_cast<int>(blockIdx.x / npairs);
  // key tiles visited by query tile 2*pair + g
  const int nkv0 = CAUSAL ? min(2 * pair + 1, nk) : nk;
  const int nkv1 = CAUSAL ? min(2 * pair + 2, nk) : nk;

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
    }
    mbar_init(&bars->drain, 1);
    // an earlier CTA already recorded a pipeline timeout: exit without work
    bars->abort_flag = (*static_cast<volatile unsigned int*>(&g_fwd_error) != 0) ? 1 : 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (bars->abort_flag) return;
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::kList);
  if (SPARSE && warp == 0) {
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
  // number of list positions each query tile runs through (a prefix of the
  // pair's list), and the key tile at a position
  const int n0 = SPARSE ? bars->nlist : nkv0;
  const int n1 = SPARSE ? bars->nlist : nkv1;
  auto kv_of = [&](int p) -> int { return SPARSE ? (list[p] & 0x3FFF) : p; };

  if (warp == kTmaWarp) {
    // ------------------------------------------------ TMA producer
    if (lane == 0 && n1 > 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_expect_tx(&bars->q_full, 2 * L::kTileBytes);
#pragma unroll
      for (int g = 0; g < 2; ++g)
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(smem + L::kQ + g * L::kTileBytes + c * 16384, &tq, &bars->q_full, c * 64,
                      (2 * pair + g) * kTileM, bh);
      for (int j = 0; j < n1; ++j) {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        const int kt = kv_of(j);
        if (!mbar_wait(&bars->k_empty[s], ph ^ 1, &bars->abort_flag, &g_fwd_error, 0x101)) break;
        mbar_arrive_expect_tx(&bars->k_full[s], L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(smem + L::kK + s * L::kTileBytes + c * 16384, &tk, &bars->k_full[s], c * 64,
                      kt * kTileN, bh);
        if (!mbar_wait(&bars->v_empty[s], ph ^ 1, &bars->abort_flag, &g_fwd_error, 0x102)) break;
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
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
      constexpr uint32_t idesc_f8 = idesc_e4m3_f32(128, 128);
      auto issue_s = [&](int g, int j) {
        const uint32_t kbase = sK + (j % kStages) * L::kTileBytes;
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
        umma_commit(&bars->s_full[g]);
      };
      auto issue_pv = [&](int g, int j) {
        const uint32_t vbase = sV + (j % kStages) * L::kTileBytes;
        if (FP8) {  // A = P~ e4m3, 8 tensor-memory columns per 32 keys; B = V^T K-major
#pragma unroll
          for (int kk = 0; kk < kTileN / 32; ++kk)
            umma_ts_f8(tmem + L::o_col(g), tmem + L::s_col(g) + kk * 8,
                       sdesc_sw128(vbase + kk * 32, 16, 1024), idesc_f8,
                       (j > 0 || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < kTileN / 16; ++kk)
            umma_ts(tmem + L::o_col(g), tmem + L::s_col(g) + kk * 8,
                    sdesc_sw128(vbase + kk * 2048, 16384, 1024), idesc_pv,
                    (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars->pv_done[g]);
      };
      bool ok = n1 > 0 && mma_wait(&bars->q_full, 0, bars, 0x201) &&
                mma_wait(&bars->k_full[0], 0, bars, 0x202);
      tc_fence_after_sync();
      if (ok) {
        issue_s(0, 0);
        issue_s(1, 0);
        umma_commit(&bars->k_empty[0]);
      }
      for (int j = 0; ok && j < n1; ++j) {
        const int s = j % kStages;
        const uint32_t ph = (j / kStages) & 1;
        const int sn = (j + 1) % kStages;
        const uint32_t phn = ((j + 1) / kStages) & 1;
        bool v_ready = false, k_next_ready = false;
        if (j < n0) {
          ok = mma_wait(&bars->p_ready[0], j & 1, bars, 0x203) &&
               mma_wait(&bars->v_full[s], ph, bars, 0x204);
          if (!ok) break;
          v_ready = true;
          tc_fence_after_sync();
          issue_pv(0, j);
          if (j + 1 < n0) {
            if (!mma_wait(&bars->k_full[sn], phn, bars, 0x205)) { ok = false; break; }
            k_next_ready = true;
            tc_fence_after_sync();
            issue_s(0, j + 1);
          }
        }
        ok = mma_wait(&bars->p_ready[1], j & 1, bars, 0x206) &&
             (v_ready || mma_wait(&bars->v_full[s], ph, bars, 0x207));
        if (!ok) break;
        tc_fence_after_sync();
        issue_pv(1, j);
        umma_commit(&bars->v_empty[s]);
        if (j + 1 < n1) {
          if (!k_next_ready && !mma_wait(&bars->k_full[sn], phn, bars, 0x208)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_s(1, j + 1);
          umma_commit(&bars->k_empty[sn]);
        }
      }
      umma_commit(&bars->drain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warpgroups
    const int g = warp >> 2;           // which query tile of the pair
    const int t = threadIdx.x & 127;   // row within the tile, TMEM lane
    const int row = (2 * pair + g) * kTileM + t;
    const int nkv = g ? n1 : n0;
    const int q0 = (2 * pair + g) * kTileM;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t scol = tmem + lane_off + L::s_col(g);
    const uint32_t ocol = tmem + lane_off + L::o_col(g);
    float m_run = -INFINITY;  // running (lazily moved) max of s * scale * log2(e)
    float l_run = 0.0f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      // dropout keep bits of this row for the 128 keys of the tile (bit c of
      // kb[c / 32] for key kv0 + c), drawn before the scores are waited for
      uint32_t kb[4] = {0u, 0u, 0u, 0u};
      if (DROPOUT) {
        const uint32_t jg0 = static_cast<uint32_t>(kv_of(j) * kTileN) >> 3;
#pragma unroll
        for (int u = 0; u < 16; ++u)
          kb[u >> 2] |= keep_byte(drop, jg0 + u, static_cast<uint32_t>(row),
                                  static_cast<uint32_t>(bh)) << (8 * (u & 3));
        reg_pin(kb);  // drawn here, before the wait, not next to their use
      }
      if (!warp_wait(&bars->s_full[g], j & 1, bars, 0x301)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t sr[128];
      tmem_ld32(scol + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld32(scol + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
      tmem_ld32(scol + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
      tmem_ld_wait();
      reg_pin(sr);
      const int kv0 = kv_of(j) * kTileN;
      // a key tile this query tile does not keep: every score is masked
      const bool keep = !SPARSE || ((list[j] >> (14 + g)) & 1);
      const bool need_mask = !keep || (CAUSAL && kv0 + kTileN - 1 > q0) || (kv0 + kTileN > N);
      if (need_mask) {
        const int lim_causal = CAUSAL ? (row - kv0) : 0x7fffffff;  // col index <= lim visible
        const int lim_n = N - 1 - kv0;
        const int lim = keep ? (lim_causal < lim_n ? lim_causal : lim_n) : -1;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) sr[c] = __float_as_uint(-INFINITY);
      }
      const float m_blk = row_max128(sr) * scale_log2;
      // move the running max only when some row of the warp needs it
      const bool move = __any_sync(0xffffffffu, m_blk > m_run + kLazyRescaleLog2);
      float alpha = 1.0f;
      if (move) {
        const float m_new = fmaxf(m_run, m_blk);
        alpha = ex2_approx(m_run - m_new);  // 0 on the first tile
        l_run *= alpha;
        m_run = m_new;
      }
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
        // P~ packed in place: pair c overwrites sr[c], already consumed.  Scalar
        // arithmetic here: packed pairs of all 128 live scores cost registers.
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c]), scale_log2, -m_use));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c + 1]), scale_log2, -m_use));
          if (c & 1)
            sp[(c >> 1) & 3].y += p0 + p1;
          else
            sp[(c >> 1) & 3].x += p0 + p1;
          if (DROPOUT) {
            const uint32_t bits = kb[c >> 4] >> ((2 * c) & 31);
            sr[c] = pack_bf16x2((bits & 1u) ? p0 : 0.0f, (bits & 2u) ? p1 : 0.0f);
          } else {
            sr[c] = pack_bf16x2(p0, p1);
          }
        }
      }
      const float2 s01 = __fadd2_rn(sp[0], sp[1]);
      const float2 s23 = __fadd2_rn(sp[2], sp[3]);
      const float2 s4 = __fadd2_rn(s01, s23);
      const float sum = s4.x + s4.y;
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
    } else if (ok && warp_wait(&bars->pv_done[g], (nkv - 1) & 1, bars, 0x303)) {
      tc_fence_after_sync();
      // a row with no visible key (block-sparse) has l = 0: O = 0, lse = -inf;
      // with dropout the kept terms carry the factor 1 / (1 - p)
      const float inv_l =
          l_run > 0.0f ? (DROPOUT ? drop.rs : 1.0f) * (FP8 ? o_scale : 1.0f) / l_run : 0.0f;
      __nv_bfloat16* orow = o + (static_cast<size_t>(bh) * N + row) * D;
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
        if (row < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      if (row < N)
        lse[static_cast<size_t>(bh) * N + row] =
            l_run > 0.0f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
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
}

template <int D, bool CAUSAL, bool SPARSE, bool DROPOUT, bool FP8 = false>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t s) {
  auto kern = fa_fwd_kernel<D, CAUSAL, SPARSE, DROPOUT, FP8>;
  constexpr uint32_t smem = FwdLayout<D, FP8 ? 1 : 2>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long nq = (a.N + kTileM - 1) / kTileM;
  const long long blocks = (nq + 1) / 2 * a.BH;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(blocks), kFwdThreads, smem, s>>>(
      *a.tq, *a.tk, *a.tv, static_cast<__nv_bfloat16*>(a.o), a.lse, a.BH, a.N, a.scale_log2,
      a.bmask, a.mstride, a.drop, a.o_scale);
  return cudaGetLastError();
}

template <bool SPARSE, bool DROPOUT>
cudaError_t launch_forward_s(const FwdArgs& a, cudaStream_t s) {
  if (a.d == 64)
    return a.causal ? launch_fwd_t<64, true, SPARSE, DROPOUT>(a, s)
                    : launch_fwd_t<64, false, SPARSE, DROPOUT>(a, s);
  return a.causal ? launch_fwd_t<128, true, SPARSE, DROPOUT>(a, s)
                  : launch_fwd_t<128, false, SPARSE, DROPOUT>(a, s);
}

}  // namespace

cudaError_t launch_forward(const FwdArgs& a, cudaStream_t s) {
  if (a.fp8) {  // d = 128, dense, no dropout (checked by the caller)
    return a.causal ? launch_fwd_t<128, true, false, false, true>(a, s)
                    : launch_fwd_t<128, false, false, false, true>(a, s);
  }
  if (a.dropout)
    return a.bmask ? launch_forward_s<true, true>(a, s) : launch_forward_s<false, true>(a, s);
  return a.bmask ? launch_forward_s<true, false>(a, s) : launch_forward_s<false, false>(a, s);
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
