/*
 * fa.h — C ABI of the exact IO-aware attention library (libfa.so, sm_103a).
 *
 * Exact scaled-dot-product attention O = softmax(scale * Q K^T) V computed
 * tile by tile with an online softmax, so the N x N score and probability
 * matrices never reach device memory, plus the recompute backward that
 * rebuilds probability tiles from Q, K and the stored per-row logsumexp.
 *
 * Sources:
 *  - "What is Flash Attention?" (Data Science in your pocket), transcript
 *    02:38-03:44 (one fused kernel, only O is written), 03:44-04:15 (tiling:
 *    a Q block stays on chip while K/V blocks stream through), 04:46-05:17
 *    (running max m and sum l with rescaling of the output accumulator),
 *    06:52-07:24 (keep O and two statistics per row; recompute P block by
 *    block in the backward pass).
 *  - "Atencao exata, acelerada por nunca escrever a grade gigante."
 *    (mentria.ai): block scores S_ij = Q_i K_j^T / sqrt(d); safe softmax;
 *    o_flash = o_exact.
 *  - "FlashAttention: fast and memory-efficient exact attention with
 *    IO-awareness" (talk): optional masking before the softmax.
 *
 * Conventions shared by every entry point:
 *  - Tensors q, k, v, o, dO, dq, dk, dv are bf16, contiguous, layout
 *    [B][H][N][d] (row-major; element (b,h,i,c) at ((b*H + h)*N + i)*d + c).
 *  - lse and the D pre-pass are fp32 [B][H][N].  lse_i = m_i + ln l_i is the
 *    natural-log logsumexp of row i of the SCALED scores scale*q_i.k_j.
 *  - causal != 0 masks key j for query i when j > i (square, top-left
 *    aligned); masked scores are -inf before the softmax.
 *  - d must be 64 or 128; B, H, N >= 1; scale > 0 and finite.  B*H must be
 *    below 2^31 (it is a coordinate of the TMA tensor maps) and so must
 *    B*H*ceil(N/128) (the work items of one launch); FA_ERR_SHAPE otherwise.
 *    There is no limit on B*H*N*d itself: every device offset is 64-bit.
 *  - Every pointer is a DEVICE pointer owned by the caller, 16-byte aligned.
 *    The library allocates no device memory in these calls.  In-place use
 *    (an output aliasing an input) is undefined.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; 0 = legacy default
 *    stream).  They return after the kernels are enqueued.  Argument errors
 *    are returned immediately and nothing is launched.  A launch failure
 *    returns FA_ERR_CUDA.  A device-side pipeline timeout is reported later
 *    by fa_get_device_error().
 *  - A recorded timeout is sticky: until fa_get_device_error() reads and
 *    clears it, every later launch of this library on the device exits at
 *    entry without computing anything, while the calls that made those
 *    launches still return FA_OK.  Outputs written after a timeout are
 *    therefore stale until the record is cleared: check fa_get_device_error()
 *    (or fa_host_wait(), which does the same) before trusting results.
 *  - Only sm_103 (GB300) devices are accepted (FA_ERR_ARCH otherwise).
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_NULL = -1,           /* a required pointer is NULL */
  FA_ERR_SHAPE = -2,          /* B, H or N < 1, sizes overflow, bad scale or p_drop */
  FA_ERR_HEADDIM = -3,        /* d not in {64, 128} */
  FA_ERR_ALIGN = -4,          /* a pointer is not 16-byte aligned */
  FA_ERR_ARCH = -5,           /* current device is not sm_103 */
  FA_ERR_WORKSPACE = -6,      /* workspace missing or too small */
  FA_ERR_CUDA = -7,           /* a CUDA runtime / driver call failed */
  FA_ERR_DEVICE_TIMEOUT = -8  /* a kernel pipeline wait timed out */
} fa_status;

/*
 * Forward pass.  q, k, v: [B][H][N][d] bf16 inputs.  o: [B][H][N][d] bf16
 * output.  lse: [B][H][N] fp32 output (logsumexp of the scaled scores).
 * Follows the fused tiled forward with the online softmax ("What is Flash
 * Attention?", 02:38-06:52).  The score matrix is never written to memory.
 */
int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, float scale, int causal, void* stream);

/*
 * Bytes of device workspace fa_backward needs: the D pre-pass,
 * 4 * B * H * N bytes (fp32 [B][H][N]), rounded up to 256.  Returns 0 when
 * the shape is invalid.
 */
size_t fa_backward_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass by recomputation ("What is Flash Attention?", 06:52-07:24:
 * P is rebuilt block by block from Q, K and the per-row statistics).
 * Inputs: q, k, v, o (the forward output), dO (gradient of o), all bf16
 * [B][H][N][d]; lse fp32 [B][H][N] from fa_forward.  Outputs dq, dk, dv
 * bf16 [B][H][N][d].  workspace: caller-owned device memory of at least
 * fa_backward_workspace_size() bytes, 256-byte aligned; its contents on entry
 * do not matter.  Gradients are those of the chain rule through the exact
 * definition: dV = P^T dO, dP = dO V^T, D_i = sum_j P_ij dP_ij (which equals
 * rowsum(dO o O)_i), dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q.
 * Kernels: the D pre-pass (from the bf16 O), the dQ kernel (which also
 * leaves the exact D in the workspace) and the dK/dV kernel.
 */
int fa_backward(const void* q, const void* k, const void* v, const void* o, const void* dO,
                const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                float scale, int causal, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Largest B*H*N that fa_backward_noalloc accepts (its built-in workspace
 * holds one fp32 per row: 8 MiB).
 */
#define FA_NOALLOC_MAX_ROWS 2097152

/*
 * fa_backward without a caller-provided workspace.  The paper has no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory -- a host runtime that hands all device memory to its own
 * pool at start-up, a plugin-style interface that passes only tensors and a
 * stream, or a latency-critical loop that cannot afford cudaMalloc's implicit
 * device synchronisation.  Arguments and results are those of fa_backward
 * minus the workspace; the call itself allocates nothing.
 *  - The workspace is a fixed 8 MiB array inside the library, held by every
 *    GPU that loads the library until the process exits.
 *  - B*H*N > FA_NOALLOC_MAX_ROWS returns FA_ERR_WORKSPACE; nothing runs.
 *  - The first call on each device looks up the array's device address (with
 *    that device current); make that first call before any stream capture.
 *  - All calls share the one array.  Calls on one stream (or otherwise
 *    ordered) are safe; calls whose kernels overlap on the GPU race on it.
 *    No state carries over between calls: the array is fully rewritten
 *    before it is read.
 */
int fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                        const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                        int H, int N, int d, float scale, int causal, void* stream);

/*
 * D pre-pass alone: D[b,h,i] = sum_c dO[b,h,i,c] * o[b,h,i,c] in fp32
 * (bf16 inputs, fp32 output [B][H][N]).  fa_backward runs it itself; it is
 * exported so that the step can be checked and timed on its own.
 */
int fa_backward_preprocess(const void* o, const void* dO, float* D, int B, int H, int N, int d,
                           void* stream);

/*
 * The two recompute kernels of fa_backward, callable one at a time (for
 * timing and checking each step).  fa_backward runs the D pre-pass, then
 * fa_backward_dq, then fa_backward_dkdv; separate callers must keep that
 * order on one stream.
 *  - fa_backward_dq: for each 128-row query tile, streams key tiles,
 *    rebuilds P and dS and writes dq = scale * dS K.  D (fp32 [B][H][N]) is
 *    read and written: it enters as the pre-pass estimate rowsum(dO o O),
 *    whose O is bf16-rounded, and leaves as the exact sum_j P_ij dP_ij
 *    accumulated in fp32 while the row is swept; dq is corrected for the
 *    difference (dq -= scale * (D - D~) * P K).
 *  - fa_backward_dkdv: for each 128-row key tile, streams query tiles,
 *    rebuilds P^T from lse, and writes dk = scale * dS^T Q and dv = P^T dO,
 *    using the D left by fa_backward_dq.
 * Arguments and errors as for fa_backward.
 */
int fa_backward_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                   float* D, void* dq, int B, int H, int N, int d, float scale, int causal,
                   void* stream);
int fa_backward_dkdv(const void* q, const void* k, const void* v, const void* dO,
                     const float* lse, const float* D, void* dk, void* dv, int B, int H, int N,
                     int d, float scale, int causal, void* stream);

/*
 * Block-sparse attention (the talk's block-sparse FlashAttention): exact
 * attention restricted to the (query tile, key tile) pairs a block mask keeps,
 * with whole tiles skipped, not computed and masked.
 *  - block_mask: DEVICE uint8 [nt][nt], nt = ceil(N / 128), row-major; entry
 *    (i, j) != 0 keeps query rows [128i, 128i+128) x key rows [128j, 128j+128).
 *  - mask_head_stride: elements between the masks of consecutive (b, h)
 *    pairs (b*H + h order); 0 = one mask shared by every head.
 *  - causal applies on top of the mask.  A query row that sees no key has
 *    o = 0, lse = -inf and dq = 0, and adds nothing to dk, dv.
 *  - N <= 131072 (at most 1024 tiles); larger N returns FA_ERR_SHAPE.
 * All other arguments, layouts and errors as for fa_forward / fa_backward.
 */
int fa_forward_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, float scale, int causal,
                           const uint8_t* block_mask, long long mask_head_stride, void* stream);
int fa_backward_blocksparse(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv,
                            int B, int H, int N, int d, float scale, int causal,
                            const uint8_t* block_mask, long long mask_head_stride,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * Attention with dropout on the probabilities (the talk's dropout applied to
 * P before the product with V, fused with the softmax so P never reaches
 * memory):  O = (P o Z / q) V, with P = softmax(scale Q K^T), q the keep
 * probability and lse that of P (before dropout).
 *  - Z is replayed, never stored.  One call of Philox4x32-10 (Salmon et al.,
 *    "Parallel random numbers: as easy as 1, 2, 3", SC 2011) at counter
 *    (j / 8, i, bh, offset), bh = b*H + h, with key (seed & 0xffffffff,
 *    seed >> 32) gives 4 words that decide keys 8(j/8) .. 8(j/8)+7 of row
 *    i: key j takes the low (even j) or high (odd j) 16 bits of word
 *    (j / 2) % 4 and is kept iff they are >= thr16 = floor(p_drop * 2^16).
 *    So q = 1 - thr16 / 65536 (p_drop taken to 16 bits), and kept values
 *    are scaled by 1 / q exactly.  The backward must get the same p_drop,
 *    seed and offset as the forward; callers advance offset (or the seed)
 *    between independent draws.
 *  - 0 <= p_drop < 1, else FA_ERR_SHAPE.  thr16 = 0 (p_drop < 2^-16) runs the
 *    kernels of fa_forward / fa_backward (identical results).
 *  - block_mask: NULL for dense attention, else a block mask as for
 *    fa_forward_blocksparse (with its limits); dropout applies on top.
 *  - The backward gives the gradients of that O: dv = (P o Z)^T dO / q,
 *    dP = (dO V^T) o Z / q, dS = P o (dP - D), dq, dk as usual.
 * All other arguments, layouts and errors as for fa_forward / fa_backward.
 */
int fa_forward_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N, int d, float scale, int causal, float p_drop,
                       unsigned long long seed, unsigned int offset, const uint8_t* block_mask,
                       long long mask_head_stride, void* stream);
int fa_backward_dropout(const void* q, const void* k, const void* v, const void* o,
                        const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                        int H, int N, int d, float scale, int causal, float p_drop,
                        unsigned long long seed, unsigned int offset, const uint8_t* block_mask,
                        long long mask_head_stride, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * FP8 forward (e4m3 inputs, FlashAttention-3's FP8 mode named on the pages):
 * O = softmax(scale * Qd Kd^T) Vd with Qd = q_descale * q8 (likewise K, V),
 * i.e. exact attention of the dequantised inputs, computed with e4m3 tensor
 * core products: S = q8 k8^T in fp32, P rounded to e4m3 for the P V
 * product, fp32 accumulation, O and lse as for fa_forward.
 *  - q8, k8: DEVICE e4m3 (one byte each, IEEE-style 1-4-3 with bias 7, no
 *    infinities) [B][H][N][d].  vt8: V TRANSPOSED per head, e4m3
 *    [B][H][d][N] (element (b,h,c,j) at ((b*H + h)*d + c)*N + j), so that
 *    both products read their operands K-major.
 *  - q_descale, k_descale, v_descale: per-tensor factors (> 0, finite) that
 *    map the stored e4m3 values back to the real inputs.
 *  - o: bf16 [B][H][N][d]; lse: fp32 [B][H][N], logsumexp of the scaled
 *    scores of the dequantised inputs.
 *  - d must be 128 (FA_ERR_HEADDIM otherwise); N must be a multiple of 16
 *    (rows of vt8 are 16-byte aligned), else FA_ERR_SHAPE.
 *  - Accuracy: besides bf16 output rounding, the one approximation is the
 *    e4m3 rounding of each probability (relative 2^-4, absolute 2^-10
 *    below the normal range) before the P V product.
 * Other conventions as for fa_forward.
 */
int fa_forward_fp8(const void* q8, const void* k8, const void* vt8, float q_descale,
                   float k_descale, float v_descale, void* o, float* lse, int B, int H, int N,
                   int d, float scale, int causal, void* stream);

/*
 * Decode step: Nq new query rows against an Nk-row key/value cache (the KV
 * cache the transcript of "What is Flash Attention?" names as the next stop,
 * 11:33).  q [B][H][Nq][d], k and v [B][H][Nk][d] bf16; o [B][H][Nq][d] bf16,
 * lse [B][H][Nq] fp32.  Query i sits at cache position Nk - Nq + i: with
 * causal != 0 it sees keys 0 .. Nk - Nq + i, else all Nk keys.  1 <= Nq <= 16,
 * Nk >= 1 (Nk >= Nq when causal), d in {64, 128}; B, H and Nk obey the shape
 * rules above (with Nk for N).  The key axis is split into
 * ranges processed in parallel, merged by the online-softmax update; the
 * workspace (device memory, 256-byte aligned, contents irrelevant) holds the
 * partial results: fa_decode_workspace_size() bytes.  Errors as fa_forward,
 * FA_ERR_WORKSPACE for a missing or small workspace.
 */
size_t fa_decode_workspace_size(int B, int H, int Nq, int Nk, int d);
int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, float scale, int causal, void* workspace,
              size_t workspace_bytes, void* stream);

/*
 * Host-buffer runtime: training steps (fa_forward + fa_backward) whose
 * inputs and outputs live in HOST memory.  The paper has no counterpart
 * (its kernels start from tensors in HBM); this is the call a host program
 * makes when its data arrive from and return to the CPU side.
 *  - fa_host_plan_create: fixes B, H, N, d, scale, causal; allocates, on the
 *    current device, the device buffers of two step slots (q, k, v, dO, o,
 *    lse, dq, dk, dv and the backward workspace each), and three streams.
 *    The only allocating call of this runtime; FA_ERR_CUDA if it fails.
 *  - fa_host_step: enqueues one step and returns without waiting: copy q, k,
 *    v, dO ([B][H][N][d] bf16, host) in, run the step, copy o (bf16), lse
 *    (fp32 [B][H][N]), dq, dk, dv out to the host buffers given.  Steps
 *    alternate between the two slots; the copies of the next and previous
 *    steps overlap the kernels of this one.  Host buffers must stay valid
 *    and untouched until fa_host_wait returns; page-locked (pinned) host
 *    memory is needed for the copies to overlap (other memory works, with
 *    copies that block the calling thread).
 *  - fa_host_wait: blocks until every enqueued step has finished and its
 *    outputs are in host memory; returns the first device error, as
 *    fa_get_device_error does (and clears it).  fa_host_step itself never
 *    reads the device error record: after a timeout, the steps enqueued
 *    before the next fa_host_wait produce stale outputs, and only that
 *    fa_host_wait's FA_ERR_DEVICE_TIMEOUT reports it.
 *  - fa_host_plan_destroy: waits, then frees the plan (NULL is a no-op).
 *  - A plan holds unguarded step state (the next slot, the slots' events):
 *    one thread at a time may call it.  Different plans are independent.
 * Argument errors as for fa_forward; NULL pointers give FA_ERR_NULL.
 */
typedef struct fa_host_plan fa_host_plan;
int fa_host_plan_create(int B, int H, int N, int d, float scale, int causal,
                        fa_host_plan** plan);
int fa_host_step(fa_host_plan* plan, const void* q, const void* k, const void* v,
                 const void* dO, void* o, float* lse, void* dq, void* dk, void* dv);
int fa_host_wait(fa_host_plan* plan);
int fa_host_plan_destroy(fa_host_plan* plan);

/*
 * Synchronises `stream`, then returns FA_ERR_DEVICE_TIMEOUT if any kernel of
 * this library timed out in a pipeline wait since the last call (and clears
 * the record), FA_ERR_CUDA if the synchronisation failed, else FA_OK.
 * *detail (may be NULL) receives the raw device record (0 when clean).
 */
int fa_get_device_error(void* stream, uint32_t* detail);

/*
 * Self-test of the failure reporting above, without any fault: launches on
 * `stream` one CTA of 32 threads that waits on a barrier nothing ever arrives
 * on.  The wait is the same bounded wait every kernel of the library uses; it
 * gives up after its limit (2 s), records the code 0x7e0 and the kernel
 * returns normally, so the next fa_get_device_error returns
 * FA_ERR_DEVICE_TIMEOUT with *detail = 0x800007e0 (timeout flag | code) and
 * clears it; the context stays usable.  FA_ERR_ARCH off sm_103; FA_ERR_CUDA if
 * the launch fails.
 */
int fa_selftest_wait_timeout(void* stream);

/* Static description of a status code. */
const char* fa_status_string(int status);

/*
 * Number of (query tile, key tile) pairs the forward pass visits for one
 * (batch, head): nq * nk without masking, sum over query tiles i of (i + 1)
 * with the causal mask (tiles of 128 x 128).  Host-only arithmetic.
 */
long long fa_forward_tile_count(int N, int causal);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
