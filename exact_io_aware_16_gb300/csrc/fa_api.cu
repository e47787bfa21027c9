// fa_api.cu — the C ABI of libfa: argument validation, TMA tensor-map
// construction and kernel launches.  No device memory is allocated here.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int B, int H, int N, int d) { return fa::check_bhnd(B, H, N, d); }

int check_scale(float scale) {
  if (!(scale > 0.0f) || !std::isfinite(scale)) return FA_ERR_SHAPE;
  return FA_OK;
}

// Is the current device an sm_103 part?  Cached per device ordinal.
int check_arch() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return FA_ERR_CUDA;
  static std::atomic<int> cache[64];  // 0 unknown, 1 ok, 2 bad (any thread may fill it)
  if (dev < 64 && cache[dev].load(std::memory_order_relaxed) == 1) return FA_OK;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  const bool ok = (major == 10 && minor == 3);
  if (dev < 64) cache[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  return ok ? FA_OK : FA_ERR_ARCH;
}

// [BH][N][d] bf16 as a 3-D tensor (d, N, BH); box 64 x rows x 1, 128B swizzle.
int encode_bhnd(CUtensorMap* map, const void* base, int BH, int N, int d, int rows) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return FA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(fa::kBoxCols), static_cast<cuuint32_t>(rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// A [BH][rows][cols] uint8 (e4m3) tensor as a 3-D tensor (cols, rows, BH);
// box 128 x 128 x 1 (128-byte rows, 128-byte swizzle).  cols must be a
// multiple of 16 (row stride in bytes).
int encode_u8(CUtensorMap* map, const void* base, int BH, int rows, int cols) {
  EncodeTiledFn enc = get_encode_tiled();
  if (!enc) return FA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols),
                           static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(cols)};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// SM count of the current device (cached per device ordinal).
int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  static std::atomic<int> cache[64];
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 1;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

float log2e_times(float scale) { return static_cast<float>(static_cast<double>(scale) * 1.4426950408889634); }

}  // namespace

extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "null pointer";
    case FA_ERR_SHAPE: return "invalid shape, scale or dropout probability";
    case FA_ERR_HEADDIM: return "head dimension must be 64 or 128";
    case FA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FA_ERR_ARCH: return "device is not sm_103 (GB300)";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_CUDA: return "CUDA call failed";
    case FA_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    default: return "unknown status";
  }
}

long long fa_forward_tile_count(int N, int causal) {
  if (N < 1) return 0;
  const long long nq = fa::num_tiles(N, fa::kTileM);
  const long long nk = fa::num_tiles(N, fa::kTileN);
  if (!causal) return nq * nk;
  return nq * (nq + 1) / 2;  // tiles are square: query tile i visits key tiles 0..i
}

static int forward_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int N, int d, float scale, int causal, const uint8_t* bmask,
                        long long mstride, void* stream, const fa::DropArgs* drop = nullptr) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_ALIGN;
  if ((st = check_arch()) != FA_OK) return st;
  const int BH = B * H;
  fa::TensorMaps maps;
  if (encode_bhnd(&maps.q, q, BH, N, d, 128) != FA_OK ||
      encode_bhnd(&maps.k, k, BH, N, d, 128) != FA_OK ||
      encode_bhnd(&maps.v, v, BH, N, d, 128) != FA_OK)
    return FA_ERR_CUDA;
  fa::FwdArgs a;
  a.tq = &maps.q;
  a.tk = &maps.k;
  a.tv = &maps.v;
  a.o = o;
  a.lse = lse;
  a.BH = BH;
  a.N = N;
  a.d = d;
  a.scale_log2 = log2e_times(scale);
  a.causal = causal ? 1 : 0;
  a.bmask = bmask;
  a.mstride = mstride;
  a.num_sms = num_sms();
  if (drop) {
    a.dropout = true;
    a.drop = *drop;
  }
  cudaError_t e = fa::launch_forward(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// block-sparse calls: mask present, at most kMaxSparseTiles tiles, stride >= 0
static int check_sparse(const uint8_t* bmask, long long mstride, int N) {
  if (!bmask) return FA_ERR_NULL;
  if (N > 128 * fa::kMaxSparseTiles || mstride < 0) return FA_ERR_SHAPE;
  return FA_OK;
}

int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, float scale, int causal, void* stream) {
  return forward_impl(q, k, v, o, lse, B, H, N, d, scale, causal, nullptr, 0, stream);
}

int fa_forward_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, float scale, int causal,
                           const uint8_t* block_mask, long long mask_head_stride, void* stream) {
  const int st = check_sparse(block_mask, mask_head_stride, N);
  if (st != FA_OK) return st;
  return forward_impl(q, k, v, o, lse, B, H, N, d, scale, causal, block_mask, mask_head_stride,
                      stream);
}

size_t fa_backward_workspace_size(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d) != FA_OK) return 0;
  const size_t bytes = static_cast<size_t>(B) * H * N * sizeof(float);
  return (bytes + 255) & ~static_cast<size_t>(255);
}

int fa_backward_preprocess(const void* o, const void* dO, float* D, int B, int H, int N, int d,
                           void* stream) {
  if (!o || !dO || !D) return FA_ERR_NULL;
  int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(D)) return FA_ERR_ALIGN;
  if ((st = check_arch()) != FA_OK) return st;
  const long long rows = static_cast<long long>(B) * H * N;
  cudaError_t e = fa::launch_bwd_preprocess(o, dO, D, rows, d, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

static int bwd_step(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                    float* D, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                    float scale, int causal, void* stream, bool do_dkdv, bool do_dq,
                    const uint8_t* bmask = nullptr, long long mstride = 0,
                    const fa::DropArgs* drop = nullptr) {
  if (!q || !k || !v || !dO || !lse || !D) return FA_ERR_NULL;
  if ((do_dkdv && (!dk || !dv)) || (do_dq && !dq)) return FA_ERR_NULL;
  int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(D) || (do_dq && !aligned16(dq)) || (do_dkdv && (!aligned16(dk) || !aligned16(dv))))
    return FA_ERR_ALIGN;
  if ((st = check_arch()) != FA_OK) return st;
  const int BH = B * H;
  fa::TensorMaps maps;
  if (encode_bhnd(&maps.q, q, BH, N, d, 128) != FA_OK ||
      encode_bhnd(&maps.k, k, BH, N, d, 128) != FA_OK ||
      encode_bhnd(&maps.v, v, BH, N, d, 128) != FA_OK ||
      encode_bhnd(&maps.dO, dO, BH, N, d, 128) != FA_OK)
    return FA_ERR_CUDA;
  fa::BwdArgs a;
  a.tq = &maps.q;
  a.tk = &maps.k;
  a.tv = &maps.v;
  a.tdo = &maps.dO;
  a.lse = lse;
  a.D = D;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.BH = BH;
  a.N = N;
  a.d = d;
  a.scale = scale;
  a.scale_log2 = log2e_times(scale);
  a.causal = causal ? 1 : 0;
  a.bmask = bmask;
  a.mstride = mstride;
  a.num_sms = num_sms();
  if (drop) {
    a.dropout = true;
    a.drop = *drop;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // dQ first: it refines D in place (exact D = sum_j P_ij dP_ij), which the
  // dK / dV kernel then reads.
  if (do_dq && fa::launch_bwd_dq(a, s) != cudaSuccess) return FA_ERR_CUDA;
  if (do_dkdv && fa::launch_bwd_dkdv(a, s) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
}

int fa_backward_dkdv(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* D, void* dk, void* dv, int B, int H, int N,
                     int d, float scale, int causal, void* stream) {
  return bwd_step(q, k, v, dO, lse, const_cast<float*>(D), nullptr, dk, dv, B, H, N, d, scale,
                  causal, stream, true, false);
}

int fa_backward_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                   float* D, void* dq, int B, int H, int N, int d, float scale, int causal,
                   void* stream) {
  return bwd_step(q, k, v, dO, lse, D, dq, nullptr, nullptr, B, H, N, d, scale, causal, stream,
                  false, true);
}

static int backward_impl(const void* q, const void* k, const void* v, const void* o,
                         const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                         int H, int N, int d, float scale, int causal, const uint8_t* bmask,
                         long long mstride, void* workspace, size_t workspace_bytes,
                         void* stream, const fa::DropArgs* drop = nullptr) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!workspace || workspace_bytes < fa_backward_workspace_size(B, H, N, d) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FA_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_ALIGN;
  if ((st = check_arch()) != FA_OK) return st;
  float* D = static_cast<float*>(workspace);
  if ((st = fa_backward_preprocess(o, dO, D, B, H, N, d, stream)) != FA_OK) return st;
  return bwd_step(q, k, v, dO, lse, D, dq, dk, dv, B, H, N, d, scale, causal, stream, true, true,
                  bmask, mstride, drop);
}

int fa_backward(const void* q, const void* k, const void* v, const void* o, const void* dO,
                const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, nullptr, 0,
                       workspace, workspace_bytes, stream);
}

int fa_backward_blocksparse(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv,
                            int B, int H, int N, int d, float scale, int causal,
                            const uint8_t* block_mask, long long mask_head_stride,
                            void* workspace, size_t workspace_bytes, void* stream) {
  const int st = check_sparse(block_mask, mask_head_stride, N);
  if (st != FA_OK) return st;
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, block_mask,
                       mask_head_stride, workspace, workspace_bytes, stream);
}

// Dropout parameters of probability p: keep iff the element's 16 random bits
// are >= thr16 = floor(p * 2^16), kept values times the inverse keep
// probability 65536 / (65536 - thr16).  p must lie in [0, 1); thr16 = 0 keeps
// everything and runs the kernels without dropout (*active = false).
static int make_drop(float p, unsigned long long seed, unsigned int offset, fa::DropArgs* out,
                     bool* active) {
  if (!(p >= 0.0f && p < 1.0f)) return FA_ERR_SHAPE;  // also rejects NaN
  const uint32_t thr16 = static_cast<uint32_t>(static_cast<double>(p) * 65536.0);  // floor
  *active = thr16 > 0;
  out->set_seed(static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  out->offset = offset;
  out->thr_hi = thr16 << 16;
  out->rs = static_cast<float>(65536.0 / (65536.0 - thr16));
  return FA_OK;
}

int fa_forward_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N, int d, float scale, int causal, float p_drop,
                       unsigned long long seed, unsigned int offset, const uint8_t* block_mask,
                       long long mask_head_stride, void* stream) {
  fa::DropArgs dr;
  bool active = false;
  int st = make_drop(p_drop, seed, offset, &dr, &active);
  if (st != FA_OK) return st;
  if (block_mask && (st = check_sparse(block_mask, mask_head_stride, N)) != FA_OK) return st;
  return forward_impl(q, k, v, o, lse, B, H, N, d, scale, causal, block_mask,
                      block_mask ? mask_head_stride : 0, stream, active ? &dr : nullptr);
}

int fa_backward_dropout(const void* q, const void* k, const void* v, const void* o,
                        const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                        int H, int N, int d, float scale, int causal, float p_drop,
                        unsigned long long seed, unsigned int offset, const uint8_t* block_mask,
                        long long mask_head_stride, void* workspace, size_t workspace_bytes,
                        void* stream) {
  fa::DropArgs dr;
  bool active = false;
  int st = make_drop(p_drop, seed, offset, &dr, &active);
  if (st != FA_OK) return st;
  if (block_mask && (st = check_sparse(block_mask, mask_head_stride, N)) != FA_OK) return st;
  return backward_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, block_mask,
                       block_mask ? mask_head_stride : 0, workspace, workspace_bytes, stream,
                       active ? &dr : nullptr);
}

int fa_forward_fp8(const void* q8, const void* k8, const void* vt8, float q_descale,
                   float k_descale, float v_descale, void* o, float* lse, int B, int H, int N,
                   int d, float scale, int causal, void* stream) {
  if (!q8 || !k8 || !vt8 || !o || !lse) return FA_ERR_NULL;
  int st = check_shape(B, H, N, d);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_HEADDIM;
  if (N % 16 != 0) return FA_ERR_SHAPE;  // rows of V^T must be 16-byte aligned
  if ((st = check_scale(scale)) != FA_OK || (st = check_scale(q_descale)) != FA_OK ||
      (st = check_scale(k_descale)) != FA_OK || (st = check_scale(v_descale)) != FA_OK)
    return st;
  const double s2 = static_cast<double>(scale) * q_descale * k_descale;
  if (!std::isfinite(s2) || !(s2 > 0.0) || !std::isfinite(static_cast<float>(s2)))
    return FA_ERR_SHAPE;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_ALIGN;
  if ((st = check_arch()) != FA_OK) return st;
  const int BH = B * H;
  fa::TensorMaps maps;
  if (encode_u8(&maps.q, q8, BH, N, d) != FA_OK || encode_u8(&maps.k, k8, BH, N, d) != FA_OK ||
      encode_u8(&maps.v, vt8, BH, d, N) != FA_OK)
    return FA_ERR_CUDA;
  fa::FwdArgs a;
  a.tq = &maps.q;
  a.tk = &maps.k;
  a.tv = &maps.v;
  a.o = o;
  a.lse = lse;
  a.BH = BH;
  a.N = N;
  a.d = d;
  a.scale_log2 = static_cast<float>(s2 * 1.4426950408889634);
  a.causal = causal ? 1 : 0;
  a.fp8 = true;
  a.o_scale = v_descale;
  a.num_sms = num_sms();
  cudaError_t e = fa::launch_forward(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Decode shapes: the cache as for check_bhnd (B*H a TMA coordinate, its key
// tiles an int32 count), and the (head, key range) CTAs of the split kernel
// within an int32 grid.
static int check_decode_shape(int B, int H, int Nq, int Nk, int d) {
  if (Nq < 1 || Nq > fa::kMaxDecodeQueries) return FA_ERR_SHAPE;
  const int st = fa::check_bhnd(B, H, Nk, d);
  if (st != FA_OK) return st;
  const long long BH = static_cast<long long>(B) * H;
  if (BH * fa::decode_splits(BH, Nk) > 0x7fffffffll) return FA_ERR_SHAPE;
  return FA_OK;
}

size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d) {
  if (check_decode_shape(B, H, Nq, Nk, d) != FA_OK) return 0;
  const long long BH = static_cast<long long>(B) * H;
  const long long S = fa::decode_splits(BH, Nk);
  const size_t floats = static_cast<size_t>(BH * S * Nq) * (d + 1);
  return (floats * sizeof(float) + 512 + 255) & ~static_cast<size_t>(255);
}

int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, float scale, int causal, void* workspace,
              size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  int st = check_decode_shape(B, H, Nq, Nk, d);
  if (st != FA_OK) return st;
  if (causal && Nk < Nq) return FA_ERR_SHAPE;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!workspace || workspace_bytes < fa_decode_workspace_size(B, H, Nq, Nk, d) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FA_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_ALIGN;
  if ((st = check_arch()) != FA_OK) return st;
  fa::DecodeArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.BH = B * H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.S = fa::decode_splits_run(a.BH, Nk, num_sms());
  a.chunk = ((Nk + a.S - 1) / a.S + 63) / 64 * 64;
  a.S = (Nk + a.chunk - 1) / a.chunk;  // no empty ranges
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  const size_t n_o = static_cast<size_t>(a.BH) * a.S * Nq * d;
  a.part_o = static_cast<float*>(workspace);
  // partial lse after the partial outputs, 256-byte aligned
  a.part_lse = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(a.part_o + n_o) + 255) & ~static_cast<uintptr_t>(255));
  fa::TensorMaps maps;
  if (encode_bhnd(&maps.q, q, a.BH, Nq, d, 128) != FA_OK ||
      encode_bhnd(&maps.k64, k, a.BH, Nk, d, 64) != FA_OK ||
      encode_bhnd(&maps.v64, v, a.BH, Nk, d, 64) != FA_OK)
    return FA_ERR_CUDA;
  cudaError_t e =
      fa::launch_decode(a, &maps.q, &maps.k64, &maps.v64, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_selftest_wait_timeout(void* stream) {
  const int st = check_arch();
  if (st != FA_OK) return st;
  return fa::launch_selftest_wait(static_cast<cudaStream_t>(stream)) == cudaSuccess ? FA_OK
                                                                                    : FA_ERR_CUDA;
}

int fa_get_device_error(void* stream, uint32_t* detail) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t w_fwd = 0, w_bwd = 0, w_dtc = 0, w_st = 0;
  if (fa::fwd_read_clear_error(&w_fwd, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::bwd_read_clear_error(&w_bwd, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::dtc_read_clear_error(&w_dtc, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::st_read_clear_error(&w_st, s) != cudaSuccess) return FA_ERR_CUDA;
  // a launch that gave up may have left its work-item counters dirty
  if (w_fwd && fa::fwd_reset_sched(s) != cudaSuccess) return FA_ERR_CUDA;
  if (w_bwd && fa::bwd_reset_sched(s) != cudaSuccess) return FA_ERR_CUDA;
  const uint32_t w = w_fwd ? w_fwd : (w_bwd ? w_bwd : (w_dtc ? w_dtc : w_st));
  if (detail) *detail = w;
  return w ? FA_ERR_DEVICE_TIMEOUT : FA_OK;
}

}  // extern "C"
