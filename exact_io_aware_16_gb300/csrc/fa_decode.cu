// fa_decode.cu — attention of a few new query rows against a long key/value
// cache (the decode step of autoregressive inference; "What is Flash
// Attention?" closes, 11:33, on the KV cache as the next place the same
// memory thinking applies).
//
// Query i (0 <= i < Nq) sits at cache position Nk - Nq + i; with the causal
// mask it sees keys 0 .. Nk - Nq + i.  With Nq <= 16 the step reads every key
// and value once and does ~4 Nq FLOPs per byte: it is bound by HBM bandwidth,
// so it runs on CUDA cores, not on the tensor core.
//
// Two kernels:
//   * decode_split: the key axis is cut into S ranges; CTA (bh, s) streams its
//     range in 64-key tiles through shared memory and keeps, per query, the
//     running max m and sum l of the online softmax (transcript 04:46-05:17)
//     with the rescaled output accumulator; it writes a partial output
//     o_s = acc / l and lse_s = m + ln l to the workspace.
//   * decode_combine: merges the S partials of each query with the same
//     running-max update: L = max_s lse_s, w_s = e^(lse_s - L),
//     o = sum_s w_s o_s / sum_s w_s, lse = L + ln sum_s w_s.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecTile = 64;  // keys per shared-memory tile
constexpr float kDecLog2e = 1.44269504088896340736f;
constexpr float kDecLn2 = 0.69314718055994530942f;

template <int D>
struct DecSmem {
  float q[kMaxDecodeQueries][D];        // q * scale * log2(e)
  uint4 k[2][kDecTile][D / 8];          // double buffer; chunk c of row j at c ^ (j & 7)
  uint4 v[2][kDecTile][D / 8];
  float part[4][kMaxDecodeQueries][kDecTile];  // partial dots of 4 head-dim quarters
  float p[kMaxDecodeQueries][kDecTile];        // probabilities
  float m[kMaxDecodeQueries], l[kMaxDecodeQueries], alpha[kMaxDecodeQueries];
};

// 16-byte global -> shared copy that bypasses registers; src_bytes = 0
// writes zeros (rows past the key range).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

template <int D>
__global__ void __launch_bounds__(kDecThreads)
    decode_split(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                 const __nv_bfloat16* __restrict__ v, float* __restrict__ part_o,
                 float* __restrict__ part_lse, int Nq, int Nk, int S, int chunk,
                 float scale_log2, int causal) {
  extern __shared__ __align__(16) uint8_t dsmem[];
  DecSmem<D>& sm = *reinterpret_cast<DecSmem<D>*>(dsmem);
  const int t = threadIdx.x;
  const int warp = t >> 5, lane = t & 31;
  const long long bh = blockIdx.x / S;
  const int s = static_cast<int>(blockIdx.x % S);
  const int k_begin = s * chunk;
  const int k_end = min(Nk, k_begin + chunk);
  const __nv_bfloat16* qb = q + bh * Nq * D;
  const uint4* kb = reinterpret_cast<const uint4*>(k + bh * Nk * D);
  const uint4* vb = reinterpret_cast<const uint4*>(v + bh * Nk * D);

  for (int e = t; e < kMaxDecodeQueries * D; e += kDecThreads) {
    const int i = e / D, c = e % D;
    sm.q[i][c] = (i < Nq) ? __bfloat162float(qb[i * D + c]) * scale_log2 : 0.0f;
  }
  if (t < kMaxDecodeQueries) {
    sm.m[t] = -INFINITY;
    sm.l[t] = 0.0f;
  }
  // PV layout: warp w owns keys [8w, 8w + 8) of each tile; lane owns kCols
  // head-dim columns; every thread accumulates all Nq query rows
  constexpr int kCols = D / 32;
  float acc[kMaxDecodeQueries][kCols];
#pragma unroll
  for (int i = 0; i < kMaxDecodeQueries; ++i)
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[i][c] = 0.0f;

  constexpr int kChunks = D / 8;
  // issue the copies of one 64-key tile of K and V into buffer b
  auto load_tile = [&](int kt0, int b) {
    for (int e = t; e < kDecTile * kChunks; e += kDecThreads) {
      const int j = e / kChunks, c = e % kChunks;
      const int key = kt0 + j;
      const bool in = key < k_end;
      const long long src = static_cast<long long>(in ? key : k_begin) * kChunks + c;
      cp_async16(&sm.k[b][j][c ^ (j & 7)], kb + src, in ? 16 : 0);
      cp_async16(&sm.v[b][j][c], vb + src, in ? 16 : 0);
    }
    cp_async_commit();
  };
  load_tile(k_begin, 0);
  int buf = 0;
  for (int kt0 = k_begin; kt0 < k_end; kt0 += kDecTile, buf ^= 1) {
    cp_async_wait_all();
    __syncthreads();  // tile kt0 landed in `buf`; the other buffer is free (and q is ready)
    if (kt0 + kDecTile < k_end) load_tile(kt0 + kDecTile, buf ^ 1);  // overlaps this tile
    // ---- partial scores: thread = (key jj, head-dim quarter ds), all Nq rows
    {
      const int jj = t & (kDecTile - 1);
      const int ds = t >> 6;
      constexpr int kQ = kChunks / 4;  // 16-byte chunks per quarter
      float kf[kQ * 8];
#pragma unroll
      for (int c = 0; c < kQ; ++c) {
        const int cc = ds * kQ + c;
        const uint4 kw = sm.k[buf][jj][cc ^ (jj & 7)];
        kf[8 * c + 0] = bf16lo(kw.x); kf[8 * c + 1] = bf16hi(kw.x);
        kf[8 * c + 2] = bf16lo(kw.y); kf[8 * c + 3] = bf16hi(kw.y);
        kf[8 * c + 4] = bf16lo(kw.z); kf[8 * c + 5] = bf16hi(kw.z);
        kf[8 * c + 6] = bf16lo(kw.w); kf[8 * c + 7] = bf16hi(kw.w);
      }
#pragma unroll
      for (int i = 0; i < kMaxDecodeQueries; ++i) {
        if (i >= Nq) break;
        const float* qr = &sm.q[i][ds * kQ * 8];
        float dot = 0.0f;
#pragma unroll
        for (int e = 0; e < kQ * 8; ++e) dot = fmaf(qr[e], kf[e], dot);
        sm.part[ds][i][jj] = dot;
      }
    }
    __syncthreads();
    // ---- online softmax per query row (warp w: rows w, w + 8)
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int i = warp + 8 * a;
      if (i >= Nq) break;
      float sc[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int jj = lane + 32 * h;
        const int key = kt0 + jj;
        const bool vis = key < k_end && (!causal || key <= Nk - Nq + i);
        const float dot = (sm.part[0][i][jj] + sm.part[1][i][jj]) +
                          (sm.part[2][i][jj] + sm.part[3][i][jj]);
        sc[h] = vis ? dot : -INFINITY;
      }
      float mx = fmaxf(sc[0], sc[1]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_old = sm.m[i];
      const float m_new = fmaxf(m_old, mx);
      const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
      const float p0 = ex2_approx(sc[0] - m_use), p1 = ex2_approx(sc[1] - m_use);
      float sum = p0 + p1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      sm.p[i][lane] = p0;
      sm.p[i][lane + 32] = p1;
      __syncwarp();
      if (lane == 0) {
        const float al = (m_old == -INFINITY) ? 0.0f : ex2_approx(m_old - m_use);
        sm.alpha[i] = al;
        sm.l[i] = sm.l[i] * al + sum;
        sm.m[i] = m_new;
      }
    }
    __syncthreads();
    // ---- O += P V over this warp's 8 keys (rescale first)
#pragma unroll
    for (int i = 0; i < kMaxDecodeQueries; ++i) {
      if (i >= Nq) break;
      const float al = sm.alpha[i];
#pragma unroll
      for (int c = 0; c < kCols; ++c) acc[i][c] *= al;
    }
#pragma unroll
    for (int jk = 0; jk < 8; ++jk) {
      const int jj = warp * 8 + jk;
      const uint32_t* vrow = reinterpret_cast<const uint32_t*>(&sm.v[buf][jj][0]);
      float vf[kCols];
#pragma unroll
      for (int c = 0; c < kCols / 2; ++c) {
        const uint32_t w = vrow[lane * (kCols / 2) + c];
        vf[2 * c] = bf16lo(w);
        vf[2 * c + 1] = bf16hi(w);
      }
#pragma unroll
      for (int i = 0; i < kMaxDecodeQueries; ++i) {
        if (i >= Nq) break;
        const float pi = sm.p[i][jj];
#pragma unroll
        for (int c = 0; c < kCols; ++c) acc[i][c] = fmaf(pi, vf[c], acc[i][c]);
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();
  // ---- reduce the 8 warps' accumulators (the K/V buffers are free now)
  float* red = reinterpret_cast<float*>(&sm.k[0][0][0]);  // [8 warps][Nq][D]
#pragma unroll
  for (int i = 0; i < kMaxDecodeQueries; ++i) {
    if (i >= Nq) break;
#pragma unroll
    for (int c = 0; c < kCols; ++c) red[(warp * Nq + i) * D + lane * kCols + c] = acc[i][c];
  }
  __syncthreads();
  for (int e = t; e < Nq * D; e += kDecThreads) {
    const int i = e / D, c = e % D;
    float sum = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) sum += red[(w * Nq + i) * D + c];
    const float l = sm.l[i];
    part_o[((bh * S + s) * Nq + i) * D + c] = l > 0.0f ? sum / l : 0.0f;
    if (c == 0)
      part_lse[(bh * S + s) * Nq + i] = l > 0.0f ? (sm.m[i] + log2f(l)) * kDecLn2 : -INFINITY;
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
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(DecSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(decode_split<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long blocks = static_cast<long long>(a.BH) * a.S;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  decode_split<D><<<static_cast<unsigned>(blocks), kDecThreads, smem, st>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), a.part_o, a.part_lse, a.Nq, a.Nk, a.S, a.chunk,
      a.scale * kDecLog2e, a.causal);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long rows = static_cast<long long>(a.BH) * a.Nq;
  decode_combine<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
      a.part_o, a.part_lse, static_cast<__nv_bfloat16*>(a.o), a.lse, rows, a.Nq, a.S);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  return a.d == 64 ? launch_decode_t<64>(a, s) : launch_decode_t<128>(a, s);
}

}  // namespace fa
