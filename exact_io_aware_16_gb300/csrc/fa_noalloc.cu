// fa_noalloc.cu — fa_backward_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// fa_backward needs a small fp32 workspace (the D = rowsum(dO o O) vector)
// that the caller passes in.  Some callers have no way to provide it: a host
// runtime that hands all device memory to its own pool at start-up and forbids
// further allocations, a plugin-style interface that passes only the tensors
// and a stream, or a latency-critical loop where cudaMalloc's implicit device
// synchronisation is not acceptable.  For them this file keeps the workspace
// in a fixed-size device array that is part of the library image, so the call
// allocates nothing.
//
// Cost and limits:
//  * every GPU that loads the library holds kNoallocScratchBytes (8 MiB) for
//    it until the process exits;
//  * B*H*N must not exceed FA_NOALLOC_MAX_ROWS (2,097,152 rows);
//  * all calls share the one array, so calls whose kernels overlap on the GPU
//    (different streams, no ordering between them) race on it; calls on one
//    stream, or otherwise ordered, are safe.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kNoallocScratchFloats = FA_NOALLOC_MAX_ROWS;
constexpr size_t kNoallocScratchBytes = kNoallocScratchFloats * sizeof(float);
static_assert(kNoallocScratchBytes == 8u * 1024u * 1024u, "scratch is 8 MiB");

// The workspace.  In host code this name is only a host-side stand-in for the
// symbol, never a device address: the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};  // device address of the array, per device

// Device address of the array on the current device, looked up once per
// device (the first call on a device does this; it must have that device
// current, which cudaGetDevice guarantees here).
int scratch_address(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = static_cast<float*>(g_scratch_ptr[dev]);
  return FA_OK;
}

}  // namespace

extern "C" int fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                                   const void* dO, const float* lse, void* dq, void* dk,
                                   void* dv, int B, int H, int N, int d, float scale, int causal,
                                   void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows > static_cast<long long>(FA_NOALLOC_MAX_ROWS)) return FA_ERR_WORKSPACE;
  // Shape, scale, alignment and device checks are those of fa_backward,
  // which runs them before anything is launched.
  const size_t need = fa_backward_workspace_size(B, H, N, d);
  if (need == 0) return d == 64 || d == 128 ? FA_ERR_SHAPE : FA_ERR_HEADDIM;
  float* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  // D is written in full by the pre-pass before the recompute kernels read
  // it, so the array's stale contents from an earlier call never matter and
  // nothing needs clearing.
  return fa_backward(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, scratch,
                     kNoallocScratchBytes, stream);
}
