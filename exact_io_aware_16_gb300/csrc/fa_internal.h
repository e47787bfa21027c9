// fa_internal.h — host-side declarations shared by the C-ABI layer and the
// kernel translation units of libfa (not part of the public ABI).
#pragma once

#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "philox.cuh"

namespace fa {

constexpr int kTileM = 128;   // query rows per tile
constexpr int kTileN = 128;   // key rows per tile
constexpr int kBoxCols = 64;  // bf16 columns per 128-byte swizzled TMA box
constexpr int kMaxSparseTiles = 1024;  // block-sparse calls: at most 1024 tiles along N
constexpr int kMaxDecodeQueries = 16;  // decode calls: at most 16 query rows

// A [BH][N][d] bf16 tensor seen by TMA as a 3-D tensor (d, N, BH) with
// 64-column boxes of 128 rows (resident tiles) or 64 rows (streamed tiles) and
// 128-byte swizzle.  Rows past N read as zero.
struct TensorMaps {
  CUtensorMap q, k, v, dO;          // 128-row boxes
  CUtensorMap q64, k64, v64, dO64;  // 64-row boxes
};

struct FwdArgs {
  const CUtensorMap* tq;
  const CUtensorMap* tk;
  const CUtensorMap* tv;
  void* o;
  float* lse;
  int BH, N, d;
  float scale_log2;  // scale * log2(e)
  int causal;
  const uint8_t* bmask = nullptr;  // block-sparse mask (nullptr: dense)
  long long mstride = 0;           // elements between (b,h) masks (0: one shared mask)
  bool dropout = false;            // dropout on P with the parameters in drop
  DropArgs drop;
  bool fp8 = false;                // e4m3 Q, K and V^T (tv maps V^T [BH][d][N])
  float o_scale = 1.0f;            // e4m3: V descale, applied to O
  int num_sms = 0;                 // SMs of the device: persistent grid size (0: one CTA per item)
};

struct BwdArgs {
  const CUtensorMap* tq;
  const CUtensorMap* tk;
  const CUtensorMap* tv;
  const CUtensorMap* tdo;
  const float* lse;
  float* D;  // D~ in; the dQ kernel overwrites it with the exact D
  void* dq;
  void* dk;
  void* dv;
  int BH, N, d;
  float scale;
  float scale_log2;
  int causal;
  const uint8_t* bmask = nullptr;  // block-sparse mask (nullptr: dense)
  long long mstride = 0;
  bool dropout = false;  // dropout on P with the parameters in drop
  DropArgs drop;
  int num_sms = 0;  // SMs of the device: persistent grid size (0: one CTA per tile)
};

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  float* part_o;    // workspace: [BH][S][Nq][d] partial outputs
  float* part_lse;  // workspace: [BH][S][Nq] partial lse
  int BH, Nq, Nk, d, S, chunk;
  float scale;
  int causal;
};

// Upper bound on the number of key ranges of a decode step (shape-only, so
// the workspace size needs no device): four waves of 152 SMs, ranges of at
// least 256 keys.
inline int decode_splits(long long BH, int Nk) {
  const long long by_len = (Nk + 255) / 256;
  long long by_sms = (608 + BH - 1) / BH;
  if (by_sms < 1) by_sms = 1;
  const long long s = by_len < by_sms ? by_len : by_sms;
  return static_cast<int>(s < 1 ? 1 : s);
}

// Key ranges a decode step actually uses: one wave of two CTAs per SM,
// ranges of at least 256 keys, never more than decode_splits().
inline int decode_splits_run(long long BH, int Nk, int num_sms) {
  const long long by_len = (Nk + 255) / 256;
  long long by_sms = (2ll * num_sms) / BH;
  if (by_sms < 1) by_sms = 1;
  long long s = by_len < by_sms ? by_len : by_sms;
  const long long cap = decode_splits(BH, Nk);
  if (s > cap) s = cap;
  return static_cast<int>(s < 1 ? 1 : s);
}

cudaError_t launch_forward(const FwdArgs& a, cudaStream_t s);
// Decode (split on the tensor core, then combine): tq maps q as (d, Nq, BH)
// with 128-row boxes, tk / tv map k / v as (d, Nk, BH) with 64-row boxes.
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap* tq, const CUtensorMap* tk,
                          const CUtensorMap* tv, cudaStream_t s);
cudaError_t launch_bwd_preprocess(const void* o, const void* dO, float* D, long long rows, int d,
                                  cudaStream_t s);
cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t s);

// Device error words of each kernel translation unit: read-and-clear.
cudaError_t fwd_read_clear_error(uint32_t* out, cudaStream_t s);
// Zero the work-item counters of the forward's persistent launches (after a
// device error, which may have left a slot dirty); synchronises s.
cudaError_t fwd_reset_sched(cudaStream_t s);
cudaError_t bwd_reset_sched(cudaStream_t s);
cudaError_t bwd_read_clear_error(uint32_t* out, cudaStream_t s);
cudaError_t dtc_read_clear_error(uint32_t* out, cudaStream_t s);

// Self-test of failure reporting: one CTA whose barrier wait runs out (its
// code, kSelftestWaitCode, lands in the self-test error word).
constexpr uint32_t kSelftestWaitCode = 0x7e0;
cudaError_t launch_selftest_wait(cudaStream_t s);
cudaError_t st_read_clear_error(uint32_t* out, cudaStream_t s);

// Work-item counter slots of a kernel file's persistent launches.  A
// persistent launch is given one slot ({claimed items, finished CTAs}); its
// CTAs claim items with atomicAdd on the first word and the launch's last CTA
// zeroes both words.  Eager launches take slots [0, kEagerSlots) in turn.  A
// launch made while its stream is being captured into a CUDA graph keeps its
// slot for every replay, so captured launches take slots from a separate ring
// [kEagerSlots, kSchedSlots): an eager launch never shares a slot with a graph.
// (Replays of one graph that run at the same time on different streams share
// its slots and must not overlap.)
constexpr int kSchedSlots = 1024;
constexpr int kEagerSlots = 768;

struct SchedRing {
  std::mutex mu;
  unsigned int* base[64] = {};  // the slot array's device address per device
  unsigned int next_eager = 0;
  unsigned int next_capture = 0;
};

// Claims the next slot of `ring` for a launch on stream s of the current
// device.  `symbol` is the host-side stand-in of the kernel file's
// __device__ unsigned int[kSchedSlots][2]; its device address is looked up
// once per device (the first persistent launch on a device should come
// before any stream capture).
inline cudaError_t claim_sched_slot(SchedRing& ring, const void* symbol, cudaStream_t s,
                                    unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((e = cudaStreamIsCapturing(s, &cap)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(ring.mu);
  if (!ring.base[dev]) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, symbol)) != cudaSuccess) return e;
    ring.base[dev] = static_cast<unsigned int*>(p);
  }
  const unsigned int slot =
      cap == cudaStreamCaptureStatusActive
          ? kEagerSlots + ring.next_capture++ % (kSchedSlots - kEagerSlots)
          : ring.next_eager++ % kEagerSlots;
  *out = ring.base[dev] + 2 * slot;
  return cudaSuccess;
}

// Tile counts (host-side mirror of the kernels' loop bounds).
inline int num_tiles(int N, int tile) { return (N + tile - 1) / tile; }

// Shape rules shared by every [B][H][N][d] entry point.  Device offsets are
// 64-bit throughout, so the element count is not limited to 32 bits; what is
// limited is B*H (the third coordinate of the TMA tensor maps, an int32) and
// the work items of one launch, B*H*ceil(N/128) (an int32 item index).  Those
// bound B*H*N*d*4 well below 2^63, so every byte size fits in size_t.
inline int check_bhnd(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffll) return FA_ERR_SHAPE;
  if (BH * num_tiles(N, kTileM) > 0x7fffffffll) return FA_ERR_SHAPE;
  return FA_OK;
}

}  // namespace fa
