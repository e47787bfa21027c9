/*
 * fa_oracle.c — plain, slow, fp64 CPU oracle for exact scaled-dot-product
 * attention and its gradients.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  Only the tests, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py use it.  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * Sources followed (web pages on FlashAttention):
 *  - "What is Flash Attention?" (Data Science in your pocket), transcript
 *    01:04: S = Q K^T / sqrt(d), softmax row by row to P, O = P V.
 *  - "Atencao exata, acelerada por nunca escrever a grade gigante."
 *    (mentria.ai), safe-softmax formula: softmax(x)_i = e^{x_i-m} / sum_j
 *    e^{x_j-m} with m = max_j x_j; and o_flash = o_exact (the tiled method
 *    reaches the plain definition exactly, so the oracle IS the definition).
 *  - "What is Flash Attention?", transcript 04:46-05:17: the online-softmax
 *    update (m' = max(m, m_blk), alpha = e^{m-m'}, beta = e^{m_blk-m'},
 *    l' = alpha l + beta sum e^{x-m_blk}, O_acc <- alpha O_acc + beta P_blk
 *    V_blk, divide by l at the end).  Used here ONLY by the pin helpers
 *    (online == two-pass), never by the definition functions.
 *  - "What is Flash Attention?", transcript 06:52-07:24: only O and two
 *    per-row statistics (m, l) are kept; P is rebuilt in the backward pass.
 *    The gradient formulas are not printed on the pages; they are the plain
 *    chain rule of L(O) through the definition above:
 *      dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,
 *      dS_ij = P_ij (dP_ij - D_i),  dQ = scale dS K,  dK = scale dS^T Q.
 *
 * Readings where the pages are silent:
 *  - causal: key j is visible to query i iff j <= i (square, top-left
 *    aligned); masked scores are -inf before the softmax.
 *  - the stored statistic is lse_i = m_i + ln l_i (natural log of the scaled
 *    scores), which is the pair (m, l) folded into one number.
 *  - block-sparse masks ("FlashAttention: fast and memory-efficient exact
 *    attention with IO-awareness" talk, block-sparse FlashAttention): an
 *    optional block mask marks whole (query block, key block) pairs as
 *    skipped; their scores are -inf, which is exact attention restricted to
 *    the kept blocks.  A row with no visible key has no softmax; it is defined
 *    here as o = 0, lse = -inf and zero gradients.
 *  - dropout (the talk: dropout applied to P before the product with V):
 *    O = (P o Z / q) V with Z_ij in {0, 1} drawn by the counter-based
 *    Philox4x32-10 generator (see philox4x32_10), so the same Z can be
 *    replayed exactly, and q the keep probability; lse is that of P (before
 *    dropout).  Each decision uses 16 random bits: p is taken as the
 *    multiple thr / 65536 of 2^-16 below it, q = 1 - thr / 65536.
 *
 * Layout: every [BH][N][d] array is row-major with index (bh*N + i)*d + c.
 * Row / column selections are flat indices r = bh*N + i.
 * All arithmetic is IEEE double; libm exp/log only.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Philox4x32-10 counter-based generator (Salmon, Moraes, Dror, Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC 2011): ten rounds of
 * two 32x32->64 multiplications mixed with the other counter words and the
 * key; the key is bumped by the two Weyl constants between rounds. */
static void philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * x0;
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * x2;
    const uint32_t y0 = (uint32_t)(p1 >> 32) ^ x1 ^ k0;
    const uint32_t y1 = (uint32_t)p1;
    const uint32_t y2 = (uint32_t)(p0 >> 32) ^ x3 ^ k1;
    const uint32_t y3 = (uint32_t)p0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The generator itself, exported for its known-answer pins. */
void fa_oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  philox4x32_10(ctr, key, out);
}

/* The 16-bit uniform that decides element (i, j) of head bh: one Philox
 * call (counter = (j / 8, i, bh, offset), key = seed) serves eight
 * consecutive keys; key j takes word (j / 2) % 4 of it, its low half for
 * even j and its high half for odd j. */
uint32_t fa_oracle_dropout_u16(uint64_t seed, uint32_t offset, int64_t bh, int i, int j) {
  const uint32_t ctr[4] = {(uint32_t)(j / 8), (uint32_t)i, (uint32_t)bh, offset};
  const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  const uint32_t word = out[(j / 2) % 4];
  return (j % 2 == 0) ? (word & 0xFFFFu) : (word >> 16);
}

/* ------------------------------------------------------------------ */
/* a minimal work-sharing loop over items (no arithmetic of the method) */

typedef void (*item_fn)(void* ctx, int64_t item, double* scratch);

typedef struct {
  item_fn fn;
  void* ctx;
  int64_t n_items;
  int64_t next; /* shared counter */
  size_t scratch_doubles;
  int failed;
} pool_t;

static void* pool_worker(void* arg) {
  pool_t* p = (pool_t*)arg;
  double* scratch = (double*)malloc(sizeof(double) * (p->scratch_doubles + 1));
  if (!scratch) {
    __atomic_store_n(&p->failed, 1, __ATOMIC_SEQ_CST);
    return NULL;
  }
  for (;;) {
    int64_t it = __atomic_fetch_add(&p->next, 1, __ATOMIC_SEQ_CST);
    if (it >= p->n_items) break;
    p->fn(p->ctx, it, scratch);
  }
  free(scratch);
  return NULL;
}

static int run_pool(item_fn fn, void* ctx, int64_t n_items, size_t scratch_doubles,
                    int nthreads) {
  pool_t p;
  p.fn = fn;
  p.ctx = ctx;
  p.n_items = n_items;
  p.next = 0;
  p.scratch_doubles = scratch_doubles;
  p.failed = 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  if ((int64_t)nthreads > n_items) nthreads = (int)(n_items > 0 ? n_items : 1);
  if (nthreads == 1) {
    pool_worker(&p);
    return p.failed ? -1 : 0;
  }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return -1;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, pool_worker, &p) != 0) break;
    ++started;
  }
  if (started == 0) pool_worker(&p);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  return p.failed ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* the definition                                                       */

typedef struct {
  const double *q, *k, *v, *dO;
  int BH, N, d, causal;
  double scale;
  const int64_t* sel; /* selected flat rows / columns, or NULL = all */
  /* optional block mask: visible iff bmask[bh*mstride + (i/bq)*nkb + j/bk] */
  const uint8_t* bmask;
  int bq, bk, nkb;
  int64_t mstride;
  /* optional dropout on P: keep (i, j) iff its 16-bit uniform >= thr, kept
   * values scaled by rs = 65536 / (65536 - thr), the inverse of the keep
   * probability */
  int dropout;
  uint64_t seed;
  uint32_t offset, thr;
  double rs;
  /* forward outputs */
  double *o, *lse;
  /* backward-row outputs */
  double *dq, *m_out, *l_out, *D_out, *D_alt_out;
  /* backward-column inputs/outputs */
  const double *m_all, *l_all, *D_all;
  double *dk, *dv;
} job_t;

/* s_ij = scale * sum_c q_ic k_jc, or -inf when causal and j > i, or when the
 * block mask drops the (i, j) block. */
static double score(const job_t* J, int64_t bh, int i, int j) {
  if (J->causal && j > i) return -INFINITY;
  if (J->bmask && !J->bmask[bh * J->mstride + (int64_t)(i / J->bq) * J->nkb + j / J->bk])
    return -INFINITY;
  const double* qi = J->q + ((size_t)bh * J->N + i) * J->d;
  const double* kj = J->k + ((size_t)bh * J->N + j) * J->d;
  double acc = 0.0;
  for (int c = 0; c < J->d; ++c) acc += qi[c] * kj[c];
  return J->scale * acc;
}

/* z_ij * rs: the dropout factor of element (i, j), 1 without dropout. */
static double drop_factor(const job_t* J, int64_t bh, int i, int j) {
  if (!J->dropout) return 1.0;
  return fa_oracle_dropout_u16(J->seed, J->offset, bh, i, j) >= J->thr ? J->rs : 0.0;
}

/* Row i of S and P written out in full (scratch holds 2N doubles):
 * s_j, m = max_j s_j, l = sum_j e^{s_j - m}, p_j = e^{s_j - m} / l. */
static void softmax_row(const job_t* J, int64_t bh, int i, double* s, double* p,
                        double* m_ret, double* l_ret) {
  const int N = J->N;
  double m = -INFINITY;
  for (int j = 0; j < N; ++j) {
    s[j] = score(J, bh, i, j);
    if (s[j] > m) m = s[j];
  }
  if (m == -INFINITY) { /* no visible key: p = 0, l = 0 */
    for (int j = 0; j < N; ++j) p[j] = 0.0;
    *m_ret = m;
    *l_ret = 0.0;
    return;
  }
  double l = 0.0;
  for (int j = 0; j < N; ++j) l += exp(s[j] - m); /* e^{-inf} = 0 */
  for (int j = 0; j < N; ++j) p[j] = exp(s[j] - m) / l;
  *m_ret = m;
  *l_ret = l;
}

static void fwd_item(void* ctx, int64_t it, double* scratch) {
  const job_t* J = (const job_t*)ctx;
  const int64_t r = J->sel ? J->sel[it] : it;
  const int64_t bh = r / J->N;
  const int i = (int)(r % J->N);
  double* s = scratch;
  double* p = scratch + J->N;
  double m, l;
  softmax_row(J, bh, i, s, p, &m, &l);
  double* oi = J->o + (size_t)it * J->d;
  if (J->dropout) /* dropout acts on P before P V (lse is unchanged) */
    for (int j = 0; j < J->N; ++j) p[j] *= drop_factor(J, bh, i, j);
  for (int c = 0; c < J->d; ++c) {
    double acc = 0.0;
    for (int j = 0; j < J->N; ++j)
      acc += p[j] * J->v[((size_t)bh * J->N + j) * J->d + c];
    oi[c] = acc;
  }
  J->lse[it] = (l > 0.0) ? m + log(l) : -INFINITY;
}

static void set_mask(job_t* J, const uint8_t* bmask, int bq, int bk, int nkb, int64_t mstride);

/* the masked entry points below take the block mask as set by the caller
 * through this thread-local pointer, so the unmasked signatures stay as they
 * are */
static __thread const uint8_t* t_bmask = 0;
static __thread int t_bq = 1, t_bk = 1, t_nkb = 0;
static __thread int64_t t_mstride = 0;
static __thread int t_dropout = 0;
static __thread uint64_t t_seed = 0;
static __thread uint32_t t_offset = 0, t_thr = 0;
static __thread double t_rs = 1.0;

/* Set (enable = 1) or clear dropout for the next calls made by this thread:
 * element (i, j) of head bh is kept iff fa_oracle_dropout_u16(seed, offset,
 * bh, i, j) >= thr, and kept probabilities are multiplied by rs. */
void fa_oracle_set_dropout(int enable, uint64_t seed, uint32_t offset, uint32_t thr, double rs) {
  t_dropout = enable;
  t_seed = seed;
  t_offset = offset;
  t_thr = thr;
  t_rs = rs;
}


/* Set (or clear with bmask = NULL) the block mask for the next calls made by
 * this thread: bmask[bh * mstride + qb * nkb + kb] != 0 keeps the block of
 * query rows [qb*bq, qb*bq+bq) and key rows [kb*bk, kb*bk+bk). */
void fa_oracle_set_block_mask(const uint8_t* bmask, int bq, int bk, int nkb, int64_t mstride) {
  t_bmask = bmask;
  t_bq = bq;
  t_bk = bk;
  t_nkb = nkb;
  t_mstride = mstride;
}

static void set_mask(job_t* J, const uint8_t* bmask, int bq, int bk, int nkb, int64_t mstride) {
  J->bmask = bmask;
  J->bq = bq > 0 ? bq : 1;
  J->bk = bk > 0 ? bk : 1;
  J->nkb = nkb;
  J->mstride = mstride;
  J->dropout = t_dropout;
  J->seed = t_seed;
  J->offset = t_offset;
  J->thr = t_thr;
  J->rs = t_rs;
}

/* O = P V and lse = m + ln l for the selected rows (all rows when sel is
 * NULL).  o is [n_rows][d], lse is [n_rows]. */
int fa_oracle_forward(const double* q, const double* k, const double* v, int BH, int N, int d,
                      double scale, int causal, const int64_t* sel, int64_t n_rows, double* o,
                      double* lse, int nthreads) {
  if (!q || !k || !v || !o || !lse || BH < 1 || N < 1 || d < 1) return -1;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.q = q; J.k = k; J.v = v;
  J.BH = BH; J.N = N; J.d = d; J.causal = causal; J.scale = scale;
  J.sel = sel; J.o = o; J.lse = lse;
  set_mask(&J, t_bmask, t_bq, t_bk, t_nkb, t_mstride);
  if (!sel) n_rows = (int64_t)BH * N;
  return run_pool(fwd_item, &J, n_rows, (size_t)2 * N, nthreads);
}

static void bwd_row_item(void* ctx, int64_t it, double* scratch) {
  const job_t* J = (const job_t*)ctx;
  const int64_t r = J->sel ? J->sel[it] : it;
  const int64_t bh = r / J->N;
  const int i = (int)(r % J->N);
  const int N = J->N, d = J->d;
  double* s = scratch;
  double* p = scratch + N;
  double* dP = scratch + 2 * (size_t)N;
  double m, l;
  softmax_row(J, bh, i, s, p, &m, &l);
  const double* dOi = J->dO + ((size_t)bh * N + i) * d;
  /* dP_ij = sum_c dO_ic v_jc, times the dropout factor z_ij rs (the
   * gradient with respect to P of O = (P o Z rs) V) */
  for (int j = 0; j < N; ++j) {
    const double* vj = J->v + ((size_t)bh * N + j) * d;
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += dOi[c] * vj[c];
    dP[j] = acc * drop_factor(J, bh, i, j);
  }
  /* D_i from its definition sum_j P_ij dP_ij ... */
  double D = 0.0;
  for (int j = 0; j < N; ++j) D += p[j] * dP[j];
  /* ... and from sum_c dO_ic o_ic with o_i = sum_j p_ij v_j */
  double D_alt = 0.0;
  for (int c = 0; c < d; ++c) {
    double oc = 0.0;
    for (int j = 0; j < N; ++j)
      oc += p[j] * drop_factor(J, bh, i, j) * J->v[((size_t)bh * N + j) * d + c];
    D_alt += dOi[c] * oc;
  }
  /* dQ_i = scale * sum_j dS_ij k_j with dS_ij = p_ij (dP_ij - D_i) */
  double* dqi = J->dq + (size_t)it * d;
  for (int c = 0; c < d; ++c) dqi[c] = 0.0;
  for (int j = 0; j < N; ++j) {
    const double dS = p[j] * (dP[j] - D);
    const double* kj = J->k + ((size_t)bh * N + j) * d;
    for (int c = 0; c < d; ++c) dqi[c] += dS * kj[c];
  }
  for (int c = 0; c < d; ++c) dqi[c] *= J->scale;
  if (J->m_out) J->m_out[it] = m;
  if (J->l_out) J->l_out[it] = l;
  if (J->D_out) J->D_out[it] = D;
  if (J->D_alt_out) J->D_alt_out[it] = D_alt;
}

/* Row pass of the backward for the selected rows: dq [n][d], and the
 * per-row m, l, D (both forms of D, which must agree).  Any of m_out,
 * l_out, D_out, D_alt_out may be NULL. */
int fa_oracle_backward_rows(const double* q, const double* k, const double* v, const double* dO,
                            int BH, int N, int d, double scale, int causal, const int64_t* sel,
                            int64_t n_rows, double* dq, double* m_out, double* l_out,
                            double* D_out, double* D_alt_out, int nthreads) {
  if (!q || !k || !v || !dO || !dq || BH < 1 || N < 1 || d < 1) return -1;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.q = q; J.k = k; J.v = v; J.dO = dO;
  J.BH = BH; J.N = N; J.d = d; J.causal = causal; J.scale = scale;
  J.sel = sel; J.dq = dq; J.m_out = m_out; J.l_out = l_out;
  J.D_out = D_out; J.D_alt_out = D_alt_out;
  set_mask(&J, t_bmask, t_bq, t_bk, t_nkb, t_mstride);
  if (!sel) n_rows = (int64_t)BH * N;
  return run_pool(bwd_row_item, &J, n_rows, (size_t)3 * N, nthreads);
}

static void bwd_col_item(void* ctx, int64_t it, double* scratch) {
  (void)scratch;
  const job_t* J = (const job_t*)ctx;
  const int64_t r = J->sel ? J->sel[it] : it;
  const int64_t bh = r / J->N;
  const int j = (int)(r % J->N);
  const int N = J->N, d = J->d;
  const double* vj = J->v + ((size_t)bh * N + j) * d;
  double* dkj = J->dk + (size_t)it * d;
  double* dvj = J->dv + (size_t)it * d;
  for (int c = 0; c < d; ++c) { dkj[c] = 0.0; dvj[c] = 0.0; }
  for (int i = 0; i < N; ++i) {
    const double s = score(J, bh, i, j);
    if (s == -INFINITY) continue; /* p_ij = 0 exactly */
    const int64_t ri = bh * N + i;
    const double p = exp(s - J->m_all[ri]) / J->l_all[ri];
    const double* dOi = J->dO + (size_t)ri * d;
    const double* qi = J->q + (size_t)ri * d;
    const double z = drop_factor(J, bh, i, j);
    double dP = 0.0;
    for (int c = 0; c < d; ++c) dP += dOi[c] * vj[c];
    dP *= z;
    const double dS = p * (dP - J->D_all[ri]);
    for (int c = 0; c < d; ++c) {
      dvj[c] += p * z * dOi[c]; /* dV = (P o Z rs)^T dO */
      dkj[c] += dS * qi[c];     /* dK = scale dS^T Q */
    }
  }
  for (int c = 0; c < d; ++c) dkj[c] *= J->scale;
}

/* Column pass of the backward for the selected key rows j: dk, dv [n][d].
 * Needs m, l, D of EVERY row ([BH*N] each, from fa_oracle_backward_rows with
 * sel = NULL), since column j of P touches all rows. */
int fa_oracle_backward_cols(const double* q, const double* k, const double* v, const double* dO,
                            const double* m_all, const double* l_all, const double* D_all,
                            int BH, int N, int d, double scale, int causal, const int64_t* sel,
                            int64_t n_cols, double* dk, double* dv, int nthreads) {
  if (!q || !k || !v || !dO || !m_all || !l_all || !D_all || !dk || !dv || BH < 1 || N < 1 ||
      d < 1)
    return -1;
  job_t J;
  memset(&J, 0, sizeof(J));
  J.q = q; J.k = k; J.v = v; J.dO = dO;
  J.BH = BH; J.N = N; J.d = d; J.causal = causal; J.scale = scale;
  J.sel = sel; J.m_all = m_all; J.l_all = l_all; J.D_all = D_all;
  J.dk = dk; J.dv = dv;
  set_mask(&J, t_bmask, t_bq, t_bk, t_nkb, t_mstride);
  if (!sel) n_cols = (int64_t)BH * N;
  return run_pool(bwd_col_item, &J, n_cols, 1, nthreads);
}

/* ------------------------------------------------------------------ */
/* decode: a few queries against a long key/value cache                 */

typedef struct {
  const double *q, *k, *v;
  int Nq, Nk, d, causal;
  double scale;
  double *o, *lse;
} dec_t;

/* Query i of a decode step sits at cache position Nk - Nq + i (the new tokens
 * are the last Nq positions); with the causal mask it sees keys 0 .. that
 * position.  The row is the plain definition: scores, safe softmax, P V. */
static void dec_item(void* ctx, int64_t it, double* s) {
  const dec_t* J = (const dec_t*)ctx;
  const int64_t bh = it / J->Nq;
  const int i = (int)(it % J->Nq);
  const int Nk = J->Nk, d = J->d;
  const int last = J->causal ? Nk - J->Nq + i : Nk - 1;
  const double* qi = J->q + ((size_t)bh * J->Nq + i) * d;
  double m = -INFINITY;
  for (int j = 0; j < Nk; ++j) {
    if (j > last) {
      s[j] = -INFINITY;
      continue;
    }
    const double* kj = J->k + ((size_t)bh * Nk + j) * d;
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += qi[c] * kj[c];
    s[j] = J->scale * acc;
    if (s[j] > m) m = s[j];
  }
  double* oi = J->o + (size_t)it * d;
  for (int c = 0; c < d; ++c) oi[c] = 0.0;
  if (m == -INFINITY) { /* no visible key */
    J->lse[it] = -INFINITY;
    return;
  }
  double l = 0.0;
  for (int j = 0; j < Nk; ++j) l += exp(s[j] - m);
  for (int j = 0; j < Nk; ++j) {
    const double p = exp(s[j] - m) / l;
    if (p == 0.0) continue;
    const double* vj = J->v + ((size_t)bh * Nk + j) * d;
    for (int c = 0; c < d; ++c) oi[c] += p * vj[c];
  }
  J->lse[it] = m + log(l);
}

/* q [BH][Nq][d], k and v [BH][Nk][d]; o [BH][Nq][d], lse [BH][Nq]. */
int fa_oracle_decode(const double* q, const double* k, const double* v, int BH, int Nq, int Nk,
                     int d, double scale, int causal, double* o, double* lse, int nthreads) {
  if (!q || !k || !v || !o || !lse || BH < 1 || Nq < 1 || Nk < 1 || d < 1) return -1;
  dec_t J;
  J.q = q; J.k = k; J.v = v;
  J.Nq = Nq; J.Nk = Nk; J.d = d; J.causal = causal; J.scale = scale;
  J.o = o; J.lse = lse;
  return run_pool(dec_item, &J, (int64_t)BH * Nq, (size_t)Nk, nthreads);
}

/* ------------------------------------------------------------------ */
/* online-softmax helpers, used only to pin the online update against
 * the two-pass definition ("What is Flash Attention?", 04:46-05:17).    */

/* Row x[0..n) processed in blocks of `block` entries.  After block b the
 * running (m, l) are written to m_trace[b], l_trace[b].  Returns the number
 * of blocks.  The block sum is taken relative to the block max m_blk and
 * put on the running scale with beta = e^{m_blk - m'}. */
int fa_oracle_online_softmax(const double* x, int n, int block, double* m_trace,
                             double* l_trace) {
  if (!x || n < 1 || block < 1) return -1;
  double m = -INFINITY, l = 0.0;
  int nb = 0;
  for (int start = 0; start < n; start += block, ++nb) {
    const int end = start + block < n ? start + block : n;
    double m_blk = -INFINITY;
    for (int t = start; t < end; ++t)
      if (x[t] > m_blk) m_blk = x[t];
    double m_new = m > m_blk ? m : m_blk;
    double alpha, beta, blk_sum = 0.0;
    if (m_new == -INFINITY) { /* every entry so far is -inf */
      alpha = 0.0; beta = 0.0;
    } else {
      alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
      beta = (m_blk == -INFINITY) ? 0.0 : exp(m_blk - m_new);
      if (m_blk != -INFINITY)
        for (int t = start; t < end; ++t) blk_sum += exp(x[t] - m_blk);
    }
    l = alpha * l + beta * blk_sum;
    m = m_new;
    if (m_trace) m_trace[nb] = m;
    if (l_trace) l_trace[nb] = l;
  }
  return nb;
}

/* One attention row done the online way: scores s[0..n), values v [n][d],
 * blocks of `block` keys.  O_acc <- alpha O_acc + beta P_blk V_blk with
 * P_blk = e^{s - m_blk}; at the end o = O_acc / l and lse = m + ln l. */
int fa_oracle_online_attention_row(const double* s, const double* v, int n, int d, int block,
                                   double* o, double* lse) {
  if (!s || !v || !o || !lse || n < 1 || d < 1 || block < 1) return -1;
  double m = -INFINITY, l = 0.0;
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  for (int start = 0; start < n; start += block) {
    const int end = start + block < n ? start + block : n;
    double m_blk = -INFINITY;
    for (int t = start; t < end; ++t)
      if (s[t] > m_blk) m_blk = s[t];
    if (m_blk == -INFINITY) continue; /* a fully masked block adds nothing */
    const double m_new = m > m_blk ? m : m_blk;
    const double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
    const double beta = exp(m_blk - m_new);
    double blk_sum = 0.0;
    for (int c = 0; c < d; ++c) o[c] *= alpha;
    for (int t = start; t < end; ++t) {
      const double pt = exp(s[t] - m_blk);
      blk_sum += pt;
      for (int c = 0; c < d; ++c) o[c] += beta * pt * v[(size_t)t * d + c];
    }
    l = alpha * l + beta * blk_sum;
    m = m_new;
  }
  if (!(l > 0.0)) return -2; /* every score was -inf: undefined row */
  for (int c = 0; c < d; ++c) o[c] /= l;
  *lse = m + log(l);
  return 0;
}
