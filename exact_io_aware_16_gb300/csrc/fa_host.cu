// fa_host.cu — the host-buffer runtime of libfa: training steps whose inputs
// and outputs live in host memory.
//
// A plan owns the device buffers of two step slots and three streams (H2D
// copies, kernels, D2H copies).  fa_host_step enqueues one step — copy q, k,
// v, dO in; fa_forward; fa_backward; copy o, lse, dq, dk, dv out — into the
// next slot and returns; events order the three streams so that a slot's
// inputs are not overwritten before its kernels have read them and its
// outputs are not overwritten before they have been copied out.  With
// page-locked host memory the copies of step i+1 (in) and step i-1 (out) run
// on the copy engines while the kernels of step i run, so a sequence of steps
// is bound by the kernels, not by the host link.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "fa_internal.h"

struct fa_host_plan {
  int B, H, N, d, causal;
  float scale;
  int device;
  size_t t_bytes;    // one [B][H][N][d] bf16 tensor
  size_t lse_bytes;  // one [B][H][N] fp32 tensor
  size_t ws_bytes;
  cudaStream_t s_in, s_comp, s_out;
  struct Slot {
    void* buf;  // one allocation: q k v dO o dq dk dv | lse | workspace
    void *q, *k, *v, *dO, *o, *dq, *dk, *dv;
    float* lse;
    void* ws;
    cudaEvent_t in_ready, comp_done, out_done;
    bool used;
  } slot[2];
  long long steps;
};

namespace {

// Restores the caller's current device when it goes out of scope.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

void release(fa_host_plan* p) {
  for (auto& s : p->slot) {
    if (s.buf) cudaFree(s.buf);
    if (s.in_ready) cudaEventDestroy(s.in_ready);
    if (s.comp_done) cudaEventDestroy(s.comp_done);
    if (s.out_done) cudaEventDestroy(s.out_done);
  }
  if (p->s_in) cudaStreamDestroy(p->s_in);
  if (p->s_comp) cudaStreamDestroy(p->s_comp);
  if (p->s_out) cudaStreamDestroy(p->s_out);
}

}  // namespace

extern "C" {

int fa_host_plan_create(int B, int H, int N, int d, float scale, int causal,
                        fa_host_plan** plan) {
  if (!plan) return FA_ERR_NULL;
  *plan = nullptr;
  const int shape_st = fa::check_bhnd(B, H, N, d);
  if (shape_st != FA_OK) return shape_st;
  if (!(scale > 0.0f) || !std::isfinite(scale)) return FA_ERR_SHAPE;
  const size_t ws = fa_backward_workspace_size(B, H, N, d);
  if (ws == 0) return FA_ERR_SHAPE;
  fa_host_plan* p = new (std::nothrow) fa_host_plan;
  if (!p) return FA_ERR_CUDA;
  std::memset(p, 0, sizeof(*p));
  p->B = B;
  p->H = H;
  p->N = N;
  p->d = d;
  p->causal = causal ? 1 : 0;
  p->scale = scale;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return FA_ERR_CUDA;
  }
  p->t_bytes = static_cast<size_t>(B) * H * N * d * 2;
  p->lse_bytes = static_cast<size_t>(B) * H * N * sizeof(float);
  p->ws_bytes = ws;
  bool ok = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->s_comp, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking) == cudaSuccess;
  const size_t tb = align256(p->t_bytes), lb = align256(p->lse_bytes);
  for (int i = 0; ok && i < 2; ++i) {
    auto& s = p->slot[i];
    ok = cudaMalloc(&s.buf, 8 * tb + lb + ws) == cudaSuccess &&
         cudaEventCreateWithFlags(&s.in_ready, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&s.comp_done, cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&s.out_done, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) break;
    char* b = static_cast<char*>(s.buf);
    void** t[8] = {&s.q, &s.k, &s.v, &s.dO, &s.o, &s.dq, &s.dk, &s.dv};
    for (int j = 0; j < 8; ++j) *t[j] = b + j * tb;
    s.lse = reinterpret_cast<float*>(b + 8 * tb);
    s.ws = b + 8 * tb + lb;
  }
  if (!ok) {
    release(p);
    delete p;
    return FA_ERR_CUDA;
  }
  *plan = p;
  return FA_OK;
}

int fa_host_step(fa_host_plan* p, const void* q, const void* k, const void* v, const void* dO,
                 void* o, float* lse, void* dq, void* dk, void* dv) {
  if (!p) return FA_ERR_NULL;
  if (!q || !k || !v || !dO || !o || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  DeviceGuard guard(p->device);
  if (!guard.ok) return FA_ERR_CUDA;
  auto& s = p->slot[p->steps & 1];
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  // inputs: the slot's previous step must have finished reading them
  if (s.used && cudaStreamWaitEvent(p->s_in, s.comp_done, 0) != cudaSuccess) return FA_ERR_CUDA;
  const void* src[4] = {q, k, v, dO};
  void* dst[4] = {s.q, s.k, s.v, s.dO};
  for (int i = 0; i < 4; ++i)
    if (cudaMemcpyAsync(dst[i], src[i], p->t_bytes, h2d, p->s_in) != cudaSuccess)
      return FA_ERR_CUDA;
  if (cudaEventRecord(s.in_ready, p->s_in) != cudaSuccess) return FA_ERR_CUDA;
  // kernels: inputs here, and the slot's previous outputs already copied out
  if (cudaStreamWaitEvent(p->s_comp, s.in_ready, 0) != cudaSuccess) return FA_ERR_CUDA;
  if (s.used && cudaStreamWaitEvent(p->s_comp, s.out_done, 0) != cudaSuccess) return FA_ERR_CUDA;
  int st = fa_forward(s.q, s.k, s.v, s.o, s.lse, p->B, p->H, p->N, p->d, p->scale, p->causal,
                      p->s_comp);
  if (st != FA_OK) return st;
  st = fa_backward(s.q, s.k, s.v, s.o, s.dO, s.lse, s.dq, s.dk, s.dv, p->B, p->H, p->N, p->d,
                   p->scale, p->causal, s.ws, p->ws_bytes, p->s_comp);
  if (st != FA_OK) return st;
  if (cudaEventRecord(s.comp_done, p->s_comp) != cudaSuccess) return FA_ERR_CUDA;
  // outputs
  if (cudaStreamWaitEvent(p->s_out, s.comp_done, 0) != cudaSuccess) return FA_ERR_CUDA;
  void* hdst[4] = {o, dq, dk, dv};
  const void* dsrc[4] = {s.o, s.dq, s.dk, s.dv};
  for (int i = 0; i < 4; ++i)
    if (cudaMemcpyAsync(hdst[i], dsrc[i], p->t_bytes, d2h, p->s_out) != cudaSuccess)
      return FA_ERR_CUDA;
  if (cudaMemcpyAsync(lse, s.lse, p->lse_bytes, d2h, p->s_out) != cudaSuccess) return FA_ERR_CUDA;
  if (cudaEventRecord(s.out_done, p->s_out) != cudaSuccess) return FA_ERR_CUDA;
  s.used = true;
  ++p->steps;
  return FA_OK;
}

int fa_host_wait(fa_host_plan* p) {
  if (!p) return FA_ERR_NULL;
  DeviceGuard guard(p->device);
  if (!guard.ok) return FA_ERR_CUDA;
  if (cudaStreamSynchronize(p->s_in) != cudaSuccess ||
      cudaStreamSynchronize(p->s_comp) != cudaSuccess ||
      cudaStreamSynchronize(p->s_out) != cudaSuccess)
    return FA_ERR_CUDA;
  return fa_get_device_error(p->s_comp, nullptr);
}

int fa_host_plan_destroy(fa_host_plan* p) {
  if (!p) return FA_OK;
  int st = FA_OK;
  {
    DeviceGuard guard(p->device);
    if (!guard.ok) {
      st = FA_ERR_CUDA;
    } else {
      if (cudaStreamSynchronize(p->s_in) != cudaSuccess ||
          cudaStreamSynchronize(p->s_comp) != cudaSuccess ||
          cudaStreamSynchronize(p->s_out) != cudaSuccess)
        st = FA_ERR_CUDA;
      release(p);
    }
  }
  delete p;
  return st;
}

}  // extern "C"
