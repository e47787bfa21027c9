// fa_decode.cu — attention of a few new query rows against a long key/value
// cache (the decode step of autoregressive inference; "What is Flash
// Attention?" closes, 11:33, on the KV cache as the next place the same
// memory thinking applies).
//
// Query i (0 <= i < Nq) sits at cache position Nk - Nq + i; with the causal
// mask it sees keys 0 .. Nk - Nq + i.  The step reads every key and value
// once and does ~Nq FLOPs per byte: it is bound by HBM bandwidth, and the
// products still run on the tensor core, so that no query count runs out of
// CUDA-core FMA throughput.
//
// Two kernels:
//   * decode_split_tc: the key axis is cut into ranges, one CTA per
//     (bh, range).  The Nq query rows are one 128-row tcgen05 A operand
//     (rows past Nq read as zero through the TMA bounds), so S = Q K^T of a
//     64-key tile is one M = 128, N = 64 MMA into tensor memory; only lanes
//     < Nq are used.  K and V tiles stream through a TMA ring; two score
//     buffers let the tensor core compute S of tile t+2 while warp 0 turns S
//     of tile t into P (online softmax of transcript 04:46-05:17, one lane
//     per query row, lazy rescale as in the forward kernel) and O += P V (TS
//     MMA, P bf16 in tensor memory) runs behind it.  The CTA writes a partial
//     output o_s = O / l and lse_s = m + ln l to the workspace.  Each CTA
//     takes 256 tensor-memory columns (S0, S1, O) and at least 80 KB of
//     shared memory, so two CTAs share an SM and the grid is one wave of two
//     CTAs per SM.  Roles: warp 0 softmax + epilogue, warp 1 TMA producer,
//     warp 2 tensor-memory allocator + MMA issuer.
//   * decode_combine: merges the partials of each query with the same
//     running-max update: L = max_s lse_s, w_s = e^(lse_s - L),
//     o = sum_s w_s o_s / sum_s w_s, lse = L + ln sum_s w_s.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

__device__ unsigned int g_dtc_error;

constexpr int kTcThreads = 96;
constexpr int kTcTmaWarp = 1;
constexpr int kTcMmaWarp = 2;
constexpr int kTcTile = 64;  // keys per tile
constexpr uint32_t kTcTmemCols = 256;
constexpr float kTcLn2 = 0.69314718055994530942f;
constexpr float kTcLazyRescaleLog2 = 8.0f;

template <int D>
struct TcLayout {
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr uint32_t kQChunk = 128u * 128u;     // 128 rows x 128 bytes
  static constexpr uint32_t kKvChunk = 64u * 128u;     // 64 rows x 128 bytes
  static constexpr uint32_t kQBytes = kQChunk * (D / 64);
  static constexpr uint32_t kKvBytes = kKvChunk * (D / 64);
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kQBytes;
  static constexpr uint32_t kV = kK + kStages * kKvBytes;
  static constexpr uint32_t kBar = kV + kStages * kKvBytes;
  static constexpr uint32_t kUsed = kBar + 256 + 1024;  // + alignment slack
  // at least 80 KB: no more than two CTAs (2 x 256 tensor-memory columns) per SM
  static constexpr uint32_t kSmem = kUsed > 81920u ? kUsed : 81920u;
  static constexpr uint32_t kOCol = 128;  // S0 at 0, S1 at 64, O at 128
};

struct TcBars {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_ready, pv_done, drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, TcBars* b, uint32_t code) {
  return mbar_wait(bar, parity, &b->abort_flag, &g_dtc_error, code);
}

template <int D>
__global__ void __launch_bounds__(kTcThreads)
    decode_split_tc(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, float* __restrict__ part_o,
                    float* __restrict__ part_lse, int Nq, int Nk, int S, int chunk,
                    float scale_log2, int causal) {
  using L = TcLayout<D>;
  constexpr int kSt = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  TcBars* bars = reinterpret_cast<TcBars*>(smem + L::kBar);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = static_cast<int>(blockIdx.x / S);
  const int s = static_cast<int>(blockIdx.x % S);
  const int k_begin = s * chunk;
  const int k_end = min(Nk, k_begin + chunk);
  const int n = (k_end - k_begin + kTcTile - 1) / kTcTile;  // >= 1: ranges are never empty

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int st = 0; st < kSt; ++st) {
      mbar_init(&bars->k_full[st], 1);
      mbar_init(&bars->k_empty[st], 1);
      mbar_init(&bars->v_full[st], 1);
      mbar_init(&bars->v_empty[st], 1);
    }
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    mbar_init(&bars->p_ready, 32);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->drain, 1);
    // an earlier CTA already recorded a pipeline timeout: exit without work
    bars->abort_flag = (*static_cast<volatile unsigned int*>(&g_dtc_error) != 0) ? 1 : 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (bars->abort_flag) return;
  if (warp == kTcMmaWarp) {
    tmem_alloc(&bars->tmem_base, kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);

  if (warp == kTcTmaWarp) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_expect_tx(&bars->q_full, L::kQBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + L::kQ + c * L::kQChunk, &tq, &bars->q_full, c * 64, 0, bh);
      for (int t = 0; t < n; ++t) {
        const int st = t % kSt;
        const uint32_t ph = (t / kSt) & 1;
        const int row0 = k_begin + t * kTcTile;
        if (!tc_wait(&bars->k_empty[st], ph ^ 1, bars, 0x401)) break;
        mbar_arrive_expect_tx(&bars->k_full[st], L::kKvBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kK + st * L::kKvBytes + c * L::kKvChunk, &tk, &bars->k_full[st],
                      c * 64, row0, bh);
        if (!tc_wait(&bars->v_empty[st], ph ^ 1, bars, 0x402)) break;
        mbar_arrive_expect_tx(&bars->v_full[st], L::kKvBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + L::kV + st * L::kKvBytes + c * L::kKvChunk, &tv, &bars->v_full[st],
                      c * 64, row0, bh);
      }
    }
    __syncwarp();
  } else if (warp == kTcMmaWarp) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTcTile, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
      auto issue_s = [&](int t) {  // S(t) = Q K_t^T into score buffer t & 1
        const uint32_t kbase = sK + (t % kSt) * L::kKvBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + (t & 1) * kTcTile,
                  sdesc_sw128(sQ + (kk >> 2) * L::kQChunk + (kk & 3) * 32, 16, 1024),
                  sdesc_sw128(kbase + (kk >> 2) * L::kKvChunk + (kk & 3) * 32, 16, 1024),
                  idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(&bars->s_full[t & 1]);
        umma_commit(&bars->k_empty[t % kSt]);
      };
      bool ok = tc_wait(&bars->q_full, 0, bars, 0x411) && tc_wait(&bars->k_full[0], 0, bars, 0x412);
      tc_fence_after_sync();
      if (ok) issue_s(0);
      if (ok && n > 1) {
        ok = tc_wait(&bars->k_full[1 % kSt], (1 / kSt) & 1, bars, 0x413);
        tc_fence_after_sync();
        if (ok) issue_s(1);
      }
      for (int t = 0; ok && t < n; ++t) {
        // O += P(t) V(t): A = P bf16 in score buffer t & 1, B = V tile MN-major
        if (!tc_wait(&bars->p_ready, t & 1, bars, 0x414) ||
            !tc_wait(&bars->v_full[t % kSt], (t / kSt) & 1, bars, 0x415)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t vbase = sV + (t % kSt) * L::kKvBytes;
#pragma unroll
        for (int kk = 0; kk < kTcTile / 16; ++kk)
          umma_ts(tmem + L::kOCol, tmem + (t & 1) * kTcTile + kk * 8,
                  sdesc_sw128(vbase + kk * 2048, L::kKvChunk, 1024), idesc_pv,
                  (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars->pv_done);
        umma_commit(&bars->v_empty[t % kSt]);
        // S(t+2) reuses buffer t & 1: it runs after PV(t) has read P(t)
        if (t + 2 < n) {
          if (!tc_wait(&bars->k_full[(t + 2) % kSt], ((t + 2) / kSt) & 1, bars, 0x416)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_s(t + 2);
        }
      }
      umma_commit(&bars->drain);
    }
    __syncwarp();
  } else {  // warp 0
    // ------------------------------------------------ softmax: lane = query row
    const int row = lane;  // rows >= Nq see zero queries; their results are dropped
    const int last_visible = causal ? (Nk - Nq + row) : (Nk - 1);
    const uint32_t lane_off = 0;  // warp 0 reads tensor-memory lanes 0..31
    float m_run = -INFINITY;
    float l_run = 0.0f;
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      if (!__all_sync(0xffffffffu, tc_wait(&bars->s_full[t & 1], (t >> 1) & 1, bars, 0x421))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t scol = tmem + lane_off + (t & 1) * kTcTile;
      uint32_t sr[64];
      tmem_ld32(scol, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(scol + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld_wait();
      reg_pin(sr);
      const int kb0 = k_begin + t * kTcTile;
      // key kb0 + c is visible iff c <= lim
      const int lim = min(k_end - 1, last_visible) - kb0;
      if (__any_sync(0xffffffffu, lim < kTcTile - 1)) {
#pragma unroll
        for (int c = 0; c < kTcTile; ++c)
          if (c > lim) sr[c] = __float_as_uint(-INFINITY);
      }
      float mp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mp[e] = __uint_as_float(sr[e]);
#pragma unroll
      for (int c = 8; c < kTcTile; c += 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) mp[e] = fmaxf(mp[e], __uint_as_float(sr[c + e]));
      const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                             fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      const float m_blk = mx * scale_log2;
      const bool move = __any_sync(0xffffffffu, m_blk > m_run + kTcLazyRescaleLog2);
      float alpha = 1.0f;
      if (move) {
        const float m_new = fmaxf(m_run, m_blk);
        alpha = ex2_approx(m_run - m_new);  // 0 on the first move
        l_run *= alpha;
        m_run = m_new;
      }
      const float m_use = (m_run == -INFINITY) ? 0.0f : m_run;
      float sp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < kTcTile / 2; ++c) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c]), scale_log2, -m_use));
        const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c + 1]), scale_log2, -m_use));
        sp[c & 7] += p0 + p1;
        sr[c] = pack_bf16x2(p0, p1);
      }
      l_run += ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      tmem_st32(scol, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      // PV(t-1) must be done before O is rescaled (and before PV(t) is issued)
      if (t > 0 && !__all_sync(0xffffffffu, tc_wait(&bars->pv_done, (t - 1) & 1, bars, 0x422))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (move && t > 0) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + L::kOCol + c * 32, r);
          tmem_ld_wait();
          reg_pin(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tmem_st32(tmem + lane_off + L::kOCol + c * 32, r);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&bars->p_ready);
    }
    // ------------------------------------------------ epilogue: partial o and lse
    if (ok && __all_sync(0xffffffffu, tc_wait(&bars->pv_done, (n - 1) & 1, bars, 0x423))) {
      tc_fence_after_sync();
      const float inv_l = l_run > 0.0f ? 1.0f / l_run : 0.0f;
      const long long prow = (static_cast<long long>(bh) * S + s) * Nq + row;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + L::kOCol + c * 32, r);
        tmem_ld_wait();
        reg_pin(r);
        if (row < Nq) {
          float4* dst = reinterpret_cast<float4*>(part_o + prow * D + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(r[4 * e]) * inv_l, __uint_as_float(r[4 * e + 1]) * inv_l,
                                 __uint_as_float(r[4 * e + 2]) * inv_l,
                                 __uint_as_float(r[4 * e + 3]) * inv_l);
        }
      }
      if (row < Nq) part_lse[prow] = l_run > 0.0f ? (m_run + log2f(l_run)) * kTcLn2 : -INFINITY;
    }
  }

  // ------------------------------------------------ teardown
  if (warp == kTcMmaWarp) mbar_wait(&bars->drain, 0, &bars->abort_flag, &g_dtc_error, 0x4ff);
  if (bars->abort_flag) {
    // let any bulk copy already in flight land before the CTA exits
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

// One warp per (bh, query): merge the S partial results.
template <int D>
__global__ void __launch_bounds__(256)
    decode_combine(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                   __nv_bfloat16* __restrict__ o, float* __restrict__ lse, long long rows, int Nq,
                   int S) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const long long bh = row / Nq;
  const int i = static_cast<int>(row % Nq);
  float L = -INFINITY;
  for (int s = 0; s < S; ++s) L = fmaxf(L, part_lse[(bh * S + s) * Nq + i]);
  constexpr int kCols = D / 32;
  float acc[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) acc[c] = 0.0f;
  float wsum = 0.0f;
  if (L != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float ls = part_lse[(bh * S + s) * Nq + i];
      const float w = (ls == -INFINITY) ? 0.0f : __expf(ls - L);
      wsum += w;
      const float* src = part_o + ((bh * S + s) * Nq + i) * D + lane * kCols;
#pragma unroll
      for (int c = 0; c < kCols; ++c) acc[c] = fmaf(w, src[c], acc[c]);
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
  __nv_bfloat16* dst = o + row * D + lane * kCols;
#pragma unroll
  for (int c = 0; c < kCols; ++c) dst[c] = __float2bfloat16_rn(acc[c] * inv);
  if (lane == 0) lse[row] = wsum > 0.0f ? L + logf(wsum) : -INFINITY;
}

template <int D>
cudaError_t launch_decode_t(const DecodeArgs& a, const CUtensorMap* tq, const CUtensorMap* tk,
                            const CUtensorMap* tv, cudaStream_t st) {
  constexpr uint32_t smem = TcLayout<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(decode_split_tc<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long blocks = static_cast<long long>(a.BH) * a.S;
  const long long rows = static_cast<long long>(a.BH) * a.Nq;
  if (blocks > 0x7fffffffll || (rows + 7) / 8 > 0x7fffffffll) return cudaErrorInvalidValue;
  decode_split_tc<D><<<static_cast<unsigned>(blocks), kTcThreads, smem, st>>>(
      *tq, *tk, *tv, a.part_o, a.part_lse, a.Nq, a.Nk, a.S, a.chunk,
      a.scale * 1.44269504088896340736f, a.causal);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  decode_combine<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
      a.part_o, a.part_lse, static_cast<__nv_bfloat16*>(a.o), a.lse, rows, a.Nq, a.S);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap* tq, const CUtensorMap* tk,
                          const CUtensorMap* tv, cudaStream_t s) {
  return a.d == 64 ? launch_decode_t<64>(a, tq, tk, tv, s) : launch_decode_t<128>(a, tq, tk, tv, s);
}

cudaError_t dtc_read_clear_error(uint32_t* out, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_dtc_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_dtc_error, &zero, sizeof(zero));
  }
  *out = v;
  return e;
}

}  // namespace fa
